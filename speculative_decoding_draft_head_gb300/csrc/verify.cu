// Rejection-sampling verification of one drafted block per request.
//
// Method: "Les mathematiques derriere l'acceleration" (seventnews.com),
// section "La garantie de l'echantillonnage par rejet": accept x with
// probability min(1, p(x)/q(x)), stop at the first rejection and draw that
// position again from the residual distribution; "DeepSeek发布DSpark"
// (learnblockchain.cn), section "DSpark 是什么？": a bonus token from the target
// follows a fully accepted block.  The residual is normalise(max(0, p - q)).
//
// Four launches:
//  1. verify_rows     grid (segments, B*(G+1)): streams the target rows j < L
//                     of every sampled request once with 16-byte loads
//                     (online softmax of t/T), and rows j <= L of greedy
//                     requests (argmax);
//  2. verify_decide   one warp per request: merges the row partials and tests
//                     every row at once (a lane per row; the first rejection is
//                     a ballot), writes the emitted tokens and
//                     marks the final draw: a residual at the rejected row or a
//                     bonus from row L (sampled requests only);
//  3. final draw      residual rows rebuild the draft logits of the rejected
//                     row (base + Markov bias on the tensor cores for bf16
//                     weights, CUDA cores for fp32, or the stored draft logits)
//                     and draw from max(0, p - q); bonus rows draw from p_L;
//  4. verify_final_merge: merges the final-draw partials into the token.
#include <climits>

#include "device_common.cuh"
#include "internal.h"

namespace dspark {
namespace {

constexpr int kRowThreads = 256;
constexpr int kResThreads = 256;

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long w) {
#pragma unroll
    for (int mask = 16; mask > 0; mask >>= 1) w = max(w, __shfl_xor_sync(0xffffffffu, w, mask));
    return w;
}

__device__ __forceinline__ int read_verify_len(const int32_t *verify_len, int b, int G) {
    const int L = verify_len ? verify_len[b] : G;
    return (L < 0 || L > G) ? -1 : L;
}

__device__ __forceinline__ bool temperature_ok(float T) { return T >= 0.f && !isinf(T); }

// Eight consecutive elements (16 bytes of bf16, 32 bytes of fp32).
__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&x)[8]) {
    const uint4 r = __ldg(reinterpret_cast<const uint4 *>(p));
    x[0] = bf16_lo(r.x); x[1] = bf16_hi(r.x); x[2] = bf16_lo(r.y); x[3] = bf16_hi(r.y);
    x[4] = bf16_lo(r.z); x[5] = bf16_hi(r.z); x[6] = bf16_lo(r.w); x[7] = bf16_hi(r.w);
}
__device__ __forceinline__ void load8(const float *p, float (&x)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// Online softmax of 8 logits x scaled by c2 (log2 units) against an integer
// reference m that may lag the running maximum, as in the draft: a term
// 2^(x c2 - m) above 1 is fine, and only a group whose sum leaves [0, 2^64]
// (far above the reference, or overflowed) is redone against its own maximum
// (an exact power-of-two rescaling of the sum).  The result m + log2 S is the
// same log-sum-exp; the common case costs one fused multiply-add, one exp2
// and one add per logit.
__device__ __forceinline__ void softmax_push8_lagging(RowState &st, const float (&x)[8], float c2, float c2l) {
    if (st.m == -INFINITY) {  // this thread's first group: its maximum, rounded up, is the reference
        float xm = x[0];
#pragma unroll
        for (int i = 1; i < 8; ++i) xm = fmaxf(xm, x[i]);
        st.m = ceilf(xm * c2);
        if (st.m == -INFINITY) return;  // every logit so far is -inf: nothing to add
    }
    float e[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) e[i] = term_exp2(x[i], c2, c2l, st.m);
    float acc = ((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]));
    if (!(acc <= 0x1p64f)) {
        float xm = x[0];
#pragma unroll
        for (int i = 1; i < 8; ++i) xm = fmaxf(xm, x[i]);
        const float cm = ceilf(fmaxf(st.m, xm * c2));
        st.S = scale_pow2(st.S, st.m - cm);
        st.m = cm;
        acc = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc += term_exp2(x[i], c2, c2l, st.m);
    }
    st.S += acc;
}

// ---------------------------------------------------------------- pass 1 ----
template <typename TIn>
__global__ void __launch_bounds__(kRowThreads)
verify_rows_kernel(const TIn *__restrict__ target, const int64_t *__restrict__ row0, int64_t n_rows,
                   const int32_t *__restrict__ verify_len,
                   const float *__restrict__ temperature, int B, int G, int V, int chunk, int nsplit,
                   RowState *__restrict__ part, uint32_t *__restrict__ flags) {
    __shared__ RowState scratch[kRowThreads / 32];
    griddep_wait();  // a programmatic dependent: the previous launch's writes are visible after this
    // the call's flag words start clear: this pass, the call's first launch,
    // raises none, and every later launch of the call reads or raises them
    // only after waiting for the launch before it
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x < kFlagBytes / sizeof(uint32_t)) flags[threadIdx.x] = 0u;
    // Unit u = seg * rows + row; launched as (rows, segments), every block takes
    // one unit (rows along x: their count B (G + 1) can pass the 65535 limit of
    // y).
    const long rows = (long)B * (G + 1);
    const long units = rows * nsplit;
    const long stride = (long)gridDim.x * gridDim.y;
    for (long u = (long)blockIdx.y * gridDim.x + blockIdx.x; u < units; u += stride) {
        const int row = (int)(u % rows);
        const int seg = (int)(u / rows);
        const int b = row / (G + 1);
        const int j = row - b * (G + 1);
        const int L = read_verify_len(verify_len, b, G);
        const float T = temperature[b];
        // sampled requests read rows j < L here (row L only for a bonus draw, in
        // the final pass); greedy requests read rows j <= L (uniform per unit)
        if (L < 0 || !temperature_ok(T) || j > L || (T > 0.f && j == L)) continue;
        const TIn *t_row = target_row(target, row0, n_rows, b, G, j, V);
        if (!t_row) continue;  // flagged by the decide kernel
        const float2 c2s = T > 0.f ? c2_split(T) : make_float2(0.f, 0.f);
        const float c2 = c2s.x, c2l = c2s.y;
        const int vb = seg * chunk;
        const int ve = min(V, vb + chunk);

        RowState st = row_state_init();
        if (T > 0.f) {
            int v = vb + 8 * threadIdx.x;
            for (; v + 8 * kRowThreads < ve; v += 16 * kRowThreads) {  // two loads in flight
                float x[8], y[8];
                load8(t_row + v, x);
                load8(t_row + v + 8 * kRowThreads, y);
                softmax_push8_lagging(st, x, c2, c2l);
                softmax_push8_lagging(st, y, c2, c2l);
            }
            if (v < ve) {
                float x[8];
                load8(t_row + v, x);
                softmax_push8_lagging(st, x, c2, c2l);
            }
        } else {  // greedy request
            for (int v = vb + 8 * threadIdx.x; v < ve; v += 8 * kRowThreads) {
                float x[8];
                load8(t_row + v, x);
#pragma unroll
                for (int e = 0; e < 8; ++e) argmax_push(st, x[e], v + e);
            }
        }
        st = block_merge(st, scratch);
        if (threadIdx.x == 0) part[(size_t)row * nsplit + seg] = st;
    }
}

// ---------------------------------------------------------------- pass 2 ----
// The greedy argmax of one row from its partials: the largest key word.
__device__ __forceinline__ unsigned long long best_of_partials(const RowState *part, int n, float *z_at) {
    unsigned long long w = 0ull;
    float z = 0.f;
    for (int i = 0; i < n; ++i)
        if (part[i].best > w) {
            w = part[i].best;
            z = part[i].z_at;
        }
    *z_at = z;
    return w;
}

template <typename TIn>
__global__ void verify_decide_kernel(const TIn *__restrict__ target, const int64_t *__restrict__ row0,
                                     int64_t n_rows, const RowState *__restrict__ part,
                                     int nsplit, const int32_t *__restrict__ anchor,
                                     const int32_t *__restrict__ draft_tokens,
                                     const float *__restrict__ draft_logq,
                                     const int32_t *__restrict__ verify_len,
                                     const float *__restrict__ temperature,
                                     const uint32_t *__restrict__ request_id, int B, int G, int V,
                                     uint32_t k0, uint32_t k1, int32_t *__restrict__ accept_len,
                                     int32_t *__restrict__ out_tokens, int32_t *__restrict__ num_out,
                                     float *__restrict__ target_lse, float *__restrict__ logp_sel,
                                     int32_t *__restrict__ final_code, float2 *__restrict__ lse_t_row,
                                     uint32_t *__restrict__ res_best, uint32_t *__restrict__ flags) {
    griddep_wait();  // a programmatic dependent: the previous launch's writes are visible after this
    const int b = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (b >= B) return;
    const float nan = __int_as_float(0x7fc00000);
    const int L = read_verify_len(verify_len, b, G);
    const float T = temperature[b];
    bool bad = false;
    if (L < 0) {
        if (lane == 0) atomicOr(flags, kFlagBadVerifyLen);
        bad = true;
    }
    if (!temperature_ok(T)) {
        if (lane == 0) atomicOr(flags, kFlagBadTemperature);
        bad = true;
    }
    if (!bad) {
        const int an = anchor[b];
        if (an < 0 || an >= V) bad = true;
        for (int j = 0; j < L; ++j) {
            const int x = draft_tokens[(size_t)b * G + j];
            if (x < 0 || x >= V) bad = true;
        }
        if (bad && lane == 0) atomicOr(flags, kFlagBadToken);
    }
    if (!bad && row0 && !target_row(target, row0, n_rows, b, G, L, V)) {
        // rows 0 .. L of a packed target must all be inside the array
        if (lane == 0) atomicOr(flags, kFlagBadTargetRow);
        bad = true;
    }
    // clear the per-row outputs of this request
    for (int j = lane; j <= G; j += 32) {
        out_tokens[(size_t)b * (G + 1) + j] = -1;
        if (target_lse) target_lse[(size_t)b * (G + 1) + j] = nan;
        if (logp_sel && j < G) logp_sel[(size_t)b * G + j] = nan;
    }
    __syncwarp();
    if (bad) {
        if (lane == 0) {
            accept_len[b] = -1;
            num_out[b] = 0;
            final_code[b] = -1;
            res_best[b] = 0u;
        }
        return;
    }
    const uint32_t id = request_id ? request_id[b] : (uint32_t)b;
    // Every tested row at once: lane j merges row j's partials (in segment
    // order), reads the target logit of x_j and decides its acceptance in
    // float-float: log p = t_x / T - lse_t, accept iff log p >= log q or
    // ln u < log p - log q (u < min(1, p / q) without an exponential); the
    // first rejection (or greedy mismatch) is the lowest set bit of a ballot.
    // Rows after it were never tested: their outputs stay NaN.
    int k = L, y = -1, d = -1;
    for (int j0 = 0; j0 < L; j0 += 32) {
        const int j = j0 + lane;
        const bool tested = j < L;
        bool pass = true;
        float lse_out = 0.f, logp_out = 0.f;
        FF lse{0.f, 0.f};
        int amax = -1;
        if (tested) {
            const RowState *pr = part + ((size_t)b * (G + 1) + j) * nsplit;
            const int x = draft_tokens[(size_t)b * G + j];
            if (T > 0.f) {
                lse = lse_of_partials(pr, nsplit);
                const float tx = to_f32(target_row(target, row0, n_rows, b, G, j, V)[x]);
                const FF logp = ff_add(div_ff(tx, T, __frcp_rn(T)), ff_neg(lse));
                const FF diff = ff_add(logp, FF{-draft_logq[(size_t)b * G + j], 0.f});  // log p - log q
                const uint4 w4 = philox4x32_10(make_uint4(0u, (uint32_t)j, id, kStreamAccept), k0, k1);
                // (a normalised float-float has the sign of its high part)
                pass = diff.hi >= 0.f || ff_add(diff, ff_neg(ln_ff(word_to_uniform(w4.x)))).hi > 0.f;
                lse_out = lse.hi;
                logp_out = logp.hi;
            } else {
                float zmax;
                const unsigned long long bw = best_of_partials(pr, nsplit, &zmax);
                amax = word_token(bw);
                lse_out = zmax;
                logp_out = (amax == x) ? 0.f : -INFINITY;
                pass = (amax == x);
            }
        }
        const unsigned int fail = __ballot_sync(0xffffffffu, tested && !pass);
        const int first = fail ? j0 + __ffs(fail) - 1 : INT_MAX;  // the first failing row
        if (tested && j <= first) {
            if (target_lse) target_lse[(size_t)b * (G + 1) + j] = lse_out;
            if (logp_sel) logp_sel[(size_t)b * G + j] = logp_out;
        }
        if (fail) {
            k = first;
            if (T > 0.f) {
                d = first;
                if (j == first) lse_t_row[b] = make_float2(lse.hi, lse.lo);
            } else {
                y = __shfl_sync(0xffffffffu, amax, first - j0);
            }
            break;
        }
    }
    int code = -1;
    if (d >= 0) {
        code = (1 << 16) | d;              // residual draw at the rejected row
    } else if (y < 0 && T > 0.f) {
        code = (2 << 16) | L;              // bonus draw from row L
    } else if (y < 0) {                    // greedy bonus: argmax of row L
        const RowState *pr = part + ((size_t)b * (G + 1) + L) * nsplit;
        unsigned long long bw = 0ull;
        float zb = 0.f;
        for (int i = lane; i < nsplit; i += 32)
            if (pr[i].best > bw) {
                bw = pr[i].best;
                zb = pr[i].z_at;
            }
        const unsigned long long mw = warp_max_u64(bw);
        y = word_token(mw);
        const unsigned int own = __ballot_sync(0xffffffffu, bw == mw);
        const float zmax = __shfl_sync(0xffffffffu, zb, __ffs(own) - 1);
        if (lane == 0 && target_lse) target_lse[(size_t)b * (G + 1) + L] = zmax;
    }
    for (int j = lane; j < k; j += 32) out_tokens[(size_t)b * (G + 1) + j] = draft_tokens[(size_t)b * G + j];
    if (lane == 0) {
        out_tokens[(size_t)b * (G + 1) + k] = (code >= 0) ? -1 : y;
        accept_len[b] = k;
        num_out[b] = k + 1;
        final_code[b] = code;
        res_best[b] = 0u;  // "none" for the final draw's row-wide best key
    }
}

// ------------------------------------------------- pass 3 (SIMT / stored) ----
// The screened per-token Gumbel-max step of the final draw for one token with
// word w, against the best key kbest this thread has seen (natural-log units).
// Residual rows (lse_q < +inf): weight r = p - q with p = exp(t/T - lse_t),
// q = exp(z/T - lse_q), key ln r + g(u) where r > 0; bonus and fallback rows
// (lse_q = +inf): key t/T + g(u).  The screen (1 - u) < (weight bound) 2^-K
// loses no winner; survivors within rounding of the threshold get the
// float-float key, and the key words decide.
__device__ __forceinline__ void final_token_step(unsigned long long &best, float &kbest, float t, float z, float T,
                                                 float rT, float c2, FF lse_t, float lse_q, uint32_t w, int v) {
    const bool residual = lse_q != INFINITY;
    const float K2 = kbest * kLog2e;
    float k2;
    if (residual) {
        const float pv = exp2f(fmaf(t, c2, -lse_t.hi * kLog2e));
        const float qv = exp2f(fmaf(z, c2, -lse_q * kLog2e));
        const float ub = (pv - qv) + 4e-7f * (pv + qv);
        if (!(ub > 0.f)) return;
        if (!(one_minus_uniform_plus_one(w) < fmaf(ub, screen_q(0.f, kbest), 1.f))) return;
        k2 = log2f(ub) - log2f(neg_log_uniform(w));
    } else {
        const float s2 = t * c2;
        if (!(one_minus_uniform_plus_one(w) < screen_q(s2, kbest) + 1.f)) return;
        k2 = s2 - log2f(neg_log_uniform(w));
    }
    if (!(k2 > K2 - key_tol2(k2, K2))) return;
    float key_hi;
    const unsigned long long word = final_key_word(t, z, w, v, !residual, T, rT, lse_t, lse_q, &key_hi);
    if (word > best) {
        best = word;
        kbest = fmaxf(kbest, key_hi);
    }
}

// Final draw with CUDA cores: residual rows take the draft logits of the
// rejected row from the stored draft logits (any dtype) or rebuild them with
// FMAs (fp32 weights); bonus rows draw from the target row L.  Each thread
// takes four tokens at a time (one Philox block).
template <typename TIn>
__global__ void __launch_bounds__(kResThreads)
verify_final_simt_kernel(const TIn *__restrict__ target, const int64_t *__restrict__ row0, int64_t n_rows,
                         const TIn *__restrict__ base,
                         const TIn *__restrict__ e_in, const TIn *__restrict__ w_out,
                         const float *__restrict__ z_in, const int32_t *__restrict__ anchor,
                         const int32_t *__restrict__ draft_tokens, const float *__restrict__ draft_lse,
                         const float *__restrict__ temperature, const uint32_t *__restrict__ request_id,
                         const int32_t *__restrict__ final_code, const float2 *__restrict__ lse_t_row,
                         int B, int G, int V, int r, uint32_t k0, uint32_t k1, int chunk, int nsplit,
                         ResidualState *__restrict__ part) {
    extern __shared__ float a_row[];  // [r]
    __shared__ unsigned long long scratch[kResThreads / 32];
    const int b = blockIdx.x;  // requests along x, segments along y
    const int code = final_code[b];
    if (code < 0) return;
    const int kind = code >> 16, d = code & 0xFFFF;
    const int seg = blockIdx.y;
    const float T = temperature[b];
    const float c2 = kLog2e / T, rT = __frcp_rn(T);
    const uint32_t id = request_id ? request_id[b] : (uint32_t)b;
    const bool residual = (kind == 1);
    const float lse_q = residual ? draft_lse[(size_t)b * G + d] : INFINITY;
    FF lse_t{0.f, 0.f};
    if (residual) {
        const float2 lt = lse_t_row[b];
        lse_t = FF{lt.x, lt.y};
    }
    if (residual && !z_in) {
        const int prev = (d == 0) ? anchor[b] : draft_tokens[(size_t)b * G + d - 1];
        for (int k = threadIdx.x; k < r; k += blockDim.x) a_row[k] = to_f32(e_in[(size_t)prev * r + k]);
    }
    __syncthreads();
    const size_t drow = (size_t)b * G + d;
    const TIn *t_row = target_row(target, row0, n_rows, b, G, d, V);  // checked by the decide kernel
    const uint32_t stream = residual ? kStreamResidual : kStreamBonus;
    const int vb = seg * chunk;  // a multiple of 16
    const int ve = min(V, vb + chunk);
    unsigned long long best = 0ull;
    float kbest = -INFINITY;
    for (int v = vb + 4 * threadIdx.x; v < ve; v += 4 * kResThreads) {  // V % 8 == 0: four tokens at once
        float t[4], z[4] = {0.f, 0.f, 0.f, 0.f};
        const float4 t4 = load4(t_row + v);
#pragma unroll
        for (int e = 0; e < 4; ++e) t[e] = elem(t4, e);
        if (residual) {
            if (z_in) {
                const float4 z4 = *reinterpret_cast<const float4 *>(z_in + drow * V + v);
                z[0] = z4.x; z[1] = z4.y; z[2] = z4.z; z[3] = z4.w;
            } else {
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                for (int k = 0; k < r; k += 4) {
                    const float4 a = *reinterpret_cast<const float4 *>(a_row + k);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float4 w = load4(w_out + (size_t)(v + e) * r + k);
                        float x = acc[e];
                        x = fmaf(a.x, w.x, x);
                        x = fmaf(a.y, w.y, x);
                        x = fmaf(a.z, w.z, x);
                        x = fmaf(a.w, w.w, x);
                        acc[e] = x;
                    }
                }
                const float4 u4 = load4(base + drow * V + v);
#pragma unroll
                for (int e = 0; e < 4; ++e) z[e] = elem(u4, e) + acc[e];
            }
        }
        const uint4 wd = philox4x32_10(make_uint4((uint32_t)v >> 2, (uint32_t)d, id, stream), k0, k1);
        final_token_step(best, kbest, t[0], z[0], T, rT, c2, lse_t, lse_q, wd.x, v);
        final_token_step(best, kbest, t[1], z[1], T, rT, c2, lse_t, lse_q, wd.y, v + 1);
        final_token_step(best, kbest, t[2], z[2], T, rT, c2, lse_t, lse_q, wd.z, v + 2);
        final_token_step(best, kbest, t[3], z[3], T, rT, c2, lse_t, lse_q, wd.w, v + 3);
    }
    best = warp_max_u64(best);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) scratch[warp] = best;
    __syncthreads();
    if (warp == 0) {
        best = (lane < kResThreads / 32) ? scratch[lane] : 0ull;
        best = warp_max_u64(best);
        if (lane == 0) part[(size_t)b * nsplit + seg].best = best;
    }
}

// One warp per request with a final draw: merge the partials, emit the token.
// If a residual row had no entry with p > q at all (impossible in exact
// arithmetic after a rejection), the token is drawn from p with the residual
// stream instead (a per-token Gumbel-max over the target row, here).
template <typename TIn>
__global__ void verify_final_merge_kernel(const ResidualState *__restrict__ part, int nsplit,
                                          const int32_t *__restrict__ final_code,
                                          const int32_t *__restrict__ accept_len,
                                          const TIn *__restrict__ target, const int64_t *__restrict__ row0,
                                          int64_t n_rows, const float *__restrict__ temperature,
                                          const uint32_t *__restrict__ request_id, int B, int G, int V,
                                          uint32_t k0, uint32_t k1, int32_t *__restrict__ out_tokens) {
    griddep_wait();  // a programmatic dependent: the previous launch's writes are visible after this
    const int b = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (b >= B) return;
    const int code = final_code[b];
    if (code < 0) return;
    unsigned long long w = 0ull;
    for (int i = lane; i < nsplit; i += 32) w = max(w, part[(size_t)b * nsplit + i].best);
    w = warp_max_u64(w);
    if (w == 0ull) {  // degenerate residual: a draw from p (stream 2)
        const int d = code & 0xFFFF;
        const float T = temperature[b];
        const float c2 = kLog2e / T, rT = __frcp_rn(T);
        const uint32_t id = request_id ? request_id[b] : (uint32_t)b;
        const TIn *t_row = target_row(target, row0, n_rows, b, G, d, V);
        float kbest = -INFINITY;
        for (int v = 4 * lane; v < V; v += 4 * 32) {
            const float4 t4 = load4(t_row + v);
            const uint4 wd = philox4x32_10(make_uint4((uint32_t)v >> 2, (uint32_t)d, id, kStreamResidual), k0, k1);
            final_token_step(w, kbest, t4.x, 0.f, T, rT, c2, FF{0.f, 0.f}, INFINITY, wd.x, v);
            final_token_step(w, kbest, t4.y, 0.f, T, rT, c2, FF{0.f, 0.f}, INFINITY, wd.y, v + 1);
            final_token_step(w, kbest, t4.z, 0.f, T, rT, c2, FF{0.f, 0.f}, INFINITY, wd.z, v + 2);
            final_token_step(w, kbest, t4.w, 0.f, T, rT, c2, FF{0.f, 0.f}, INFINITY, wd.w, v + 3);
        }
        w = warp_max_u64(w);
    }
    if (lane == 0) out_tokens[(size_t)b * (G + 1) + accept_len[b]] = word_token(w);
}

template <typename TIn>
cudaError_t launch_verify_rows_t(const VerifyArgs &a, const VerifyPlan &p, cudaStream_t s) {
    RowState *row_part = reinterpret_cast<RowState *>(a.ws + p.row_part_offset);
    const TIn *target = static_cast<const TIn *>(a.target);
    const dim3 grid((unsigned int)(a.B * (a.G + 1)), (unsigned int)p.row_split);
    return launch_dependent(verify_rows_kernel<TIn>, grid, dim3(kRowThreads), 0, s, target, a.target_row0,
                            a.n_target_rows, a.verify_len, a.temperature, a.B, a.G, a.V, p.row_chunk, p.row_split,
                            row_part, reinterpret_cast<uint32_t *>(a.ws));
}

template <typename TIn>
cudaError_t launch_verify_finish_t(const VerifyArgs &a, const VerifyPlan &p, cudaStream_t s) {
    uint32_t *flags = reinterpret_cast<uint32_t *>(a.ws);
    RowState *row_part = reinterpret_cast<RowState *>(a.ws + p.row_part_offset);
    int32_t *final_code = reinterpret_cast<int32_t *>(a.ws + p.res_row_offset);
    float2 *lse_t_row = reinterpret_cast<float2 *>(a.ws + p.lse_t_offset);
    ResidualState *res_part = reinterpret_cast<ResidualState *>(a.ws + p.res_part_offset);
    uint32_t *res_best = reinterpret_cast<uint32_t *>(a.ws + p.res_best_offset);
    const uint32_t k0 = (uint32_t)(a.seed & 0xFFFFFFFFu), k1 = (uint32_t)(a.seed >> 32);
    const TIn *target = static_cast<const TIn *>(a.target);

    cudaError_t e;
    const int warps = 4;
    e = launch_dependent(verify_decide_kernel<TIn>, dim3((a.B + warps - 1) / warps), dim3(32 * warps), 0, s,
                         target, a.target_row0, a.n_target_rows, (const RowState *)row_part, p.row_split, a.anchor,
                         a.draft_tokens, a.draft_logq, a.verify_len, a.temperature, a.request_id, a.B, a.G, a.V, k0,
                         k1, a.accept_len, a.out_tokens, a.num_out, a.target_lse, a.logp_sel, final_code, lse_t_row,
                         res_best, flags);
    if (e != cudaSuccess) return e;
    const bool tensor = p.tensor_residual && !a.z_in;
    const int res_nsplit = tensor ? p.res_split_tc : p.res_split;
    if (tensor) {
        // the last draft launch (position G-1) walked in direction G-1: continue from its end
        FinalArgs fa{a.target, a.target_row0, a.n_target_rows, a.base, a.e_in, a.w_out, a.anchor, a.draft_tokens, a.temperature,
                     a.request_id, final_code, lse_t_row, a.draft_lse, a.B, a.G, a.V, a.r, res_nsplit,
                     a.G, a.seed, res_part, res_best, flags};
        e = launch_final_tensor(fa, s);
    } else {
        const size_t smem = sizeof(float) * (size_t)a.r;
        verify_final_simt_kernel<TIn><<<dim3(a.B, p.res_split), kResThreads, smem, s>>>(
            target, a.target_row0, a.n_target_rows, static_cast<const TIn *>(a.base), static_cast<const TIn *>(a.e_in),
            static_cast<const TIn *>(a.w_out), a.z_in, a.anchor, a.draft_tokens, a.draft_lse,
            a.temperature, a.request_id, final_code, lse_t_row, a.B, a.G, a.V, a.r, k0, k1, p.res_chunk,
            p.res_split, res_part);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    return launch_dependent(verify_final_merge_kernel<TIn>, dim3((a.B + warps - 1) / warps), dim3(32 * warps), 0, s,
                            (const ResidualState *)res_part, res_nsplit, (const int32_t *)final_code,
                            (const int32_t *)a.accept_len, target, a.target_row0, a.n_target_rows, a.temperature,
                            a.request_id, a.B, a.G, a.V, k0, k1, a.out_tokens);
}

}  // namespace

cudaError_t launch_verify(const VerifyArgs &a, const VerifyPlan &p, cudaStream_t s) {
    cudaError_t e = (a.dt == DSPARK_BF16) ? launch_verify_rows_t<__nv_bfloat16>(a, p, s) : launch_verify_rows_t<float>(a, p, s);
    if (e != cudaSuccess) return e;
    return (a.dt == DSPARK_BF16) ? launch_verify_finish_t<__nv_bfloat16>(a, p, s) : launch_verify_finish_t<float>(a, p, s);
}

VerifyPlan plan_verify(int B, int G, int V, int r, dspark_dtype dt) {
    (void)r;
    VerifyPlan p{};
    const long rows = (long)B * (G + 1);
    // target rows: aim for ~8 blocks per SM among the rows that are read
    // (about half of them with scheduled lengths), segments >= 4096 entries;
    // twice as many segments measured slower (dspark5, qwen3, largev)
    long want = (16L * kNumSMs + rows - 1) / rows;
    int max_split = (V + 4095) / 4096;
    int split = (int)(want < 1 ? 1 : (want > max_split ? max_split : want));
    int chunk = ((V + split - 1) / split + 7) / 8 * 8;
    p.row_split = (V + chunk - 1) / chunk;
    p.row_chunk = chunk;
    // residual rows: the tensor-core kernel's segments (bf16), else SIMT segments
    p.tensor_residual = (dt == DSPARK_BF16);
    long want_r = (2L * kNumSMs + B - 1) / B;
    int max_r = (V + 1023) / 1024;
    int rs = (int)(want_r < 1 ? 1 : (want_r > max_r ? max_r : want_r));
    int rchunk = ((V + rs - 1) / rs + 15) / 16 * 16;
    p.res_chunk = rchunk;
    p.res_split = (V + rchunk - 1) / rchunk;
    p.res_split_tc = p.tensor_residual ? tc_segments(B, V) : 0;
    const int res_slots = p.res_split > p.res_split_tc ? p.res_split : p.res_split_tc;
    size_t off = kFlagBytes;
    p.row_part_offset = off;
    off = align_up(off + sizeof(RowState) * (size_t)rows * p.row_split, 256);
    p.res_row_offset = off;
    off = align_up(off + sizeof(int32_t) * (size_t)B, 256);
    p.lse_t_offset = off;
    off = align_up(off + sizeof(float2) * (size_t)B, 256);
    p.res_part_offset = off;
    off = align_up(off + sizeof(ResidualState) * (size_t)B * res_slots, 256);
    p.res_best_offset = off;
    off = align_up(off + sizeof(uint32_t) * (size_t)B, 256);
    p.ws_bytes = off;
    return p;
}

}  // namespace dspark

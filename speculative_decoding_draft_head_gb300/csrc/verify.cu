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

__device__ __forceinline__ ResidualState residual_warp_merge(ResidualState s) {
#pragma unroll
    for (int mask = 16; mask > 0; mask >>= 1) {
        ResidualState o;
        o.key_res = __shfl_xor_sync(0xffffffffu, s.key_res, mask);
        o.idx_res = __shfl_xor_sync(0xffffffffu, s.idx_res, mask);
        residual_merge(s, o);
    }
    return s;
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

// Online softmax of 8 logits x scaled by c2 (log2 units) against a reference
// m that may lag the running maximum, as in the draft: a term 2^(x c2 - m)
// above 1 is fine, and only a group whose sum leaves [0, 2^64] (far above the
// reference, or overflowed) is redone against its own maximum.  The result
// m + log2 S is the same log-sum-exp; the common case costs one fused
// multiply-add, one exp2 and one add per logit.
__device__ __forceinline__ void softmax_push8_lagging(RowState &st, const float (&x)[8], float c2) {
    if (st.m == -INFINITY) {  // this thread's first group: its maximum is the reference
        float xm = x[0];
#pragma unroll
        for (int i = 1; i < 8; ++i) xm = fmaxf(xm, x[i]);
        st.m = xm * c2;
        if (st.m == -INFINITY) return;  // every logit so far is -inf: nothing to add
    }
    float e[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) e[i] = fast_exp2(fmaf(x[i], c2, -st.m));
    float acc = ((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]));
    if (!(acc <= 0x1p64f)) {
        float xm = x[0];
#pragma unroll
        for (int i = 1; i < 8; ++i) xm = fmaxf(xm, x[i]);
        const float cm = fmaxf(st.m, xm * c2);
        st.S *= fast_exp2(st.m - cm);
        st.m = cm;
        acc = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc += fast_exp2(fmaf(x[i], c2, -st.m));
    }
    st.S += acc;
}

// ---------------------------------------------------------------- pass 1 ----
template <typename TIn>
__global__ void __launch_bounds__(kRowThreads)
verify_rows_kernel(const TIn *__restrict__ target, const int64_t *__restrict__ row0, int64_t n_rows,
                   const int32_t *__restrict__ verify_len,
                   const float *__restrict__ temperature, int B, int G, int V, int chunk, int nsplit,
                   RowState *__restrict__ part) {
    __shared__ RowState scratch[kRowThreads / 32];
    // Unit u = seg * rows + row.  Launched as (rows, segments) every block takes
    // one unit (rows along x: their count B (G + 1) can pass the 65535 limit of
    // y); launched with fewer blocks (beside the draft kernel, one block per SM)
    // the blocks walk the units.
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
        const float c2 = T > 0.f ? kLog2e / T : 0.f;
        const int vb = seg * chunk;
        const int ve = min(V, vb + chunk);

        RowState st = row_state_init();
        if (T > 0.f) {
            int v = vb + 8 * threadIdx.x;
            for (; v + 8 * kRowThreads < ve; v += 16 * kRowThreads) {  // two loads in flight
                float x[8], y[8];
                load8(t_row + v, x);
                load8(t_row + v + 8 * kRowThreads, y);
                softmax_push8_lagging(st, x, c2);
                softmax_push8_lagging(st, y, c2);
            }
            if (v < ve) {
                float x[8];
                load8(t_row + v, x);
                softmax_push8_lagging(st, x, c2);
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
                                     int32_t *__restrict__ final_code, float *__restrict__ lse_t_row,
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
    const float c2 = T > 0.f ? kLog2e / T : 0.f;
    const uint32_t id = request_id ? request_id[b] : (uint32_t)b;
    // Every tested row at once: lane j merges row j's partials (in segment
    // order), reads the target logit of x_j and decides its acceptance; the
    // first rejection (or greedy mismatch) is the lowest set bit of a ballot.
    // Rows after it were never tested: their outputs stay NaN.
    int k = L, y = -1, d = -1;
    for (int j0 = 0; j0 < L; j0 += 32) {
        const int j = j0 + lane;
        const bool tested = j < L;
        bool pass = true;
        float lse_out = 0.f, logp = 0.f, lse2 = 0.f;
        int amax = -1;
        if (tested) {
            RowState s = row_state_init();
            const RowState *pr = part + ((size_t)b * (G + 1) + j) * nsplit;
            for (int i = 0; i < nsplit; ++i) row_state_merge(s, pr[i]);
            const int x = draft_tokens[(size_t)b * G + j];
            if (T > 0.f) {
                lse2 = s.m + log2f(s.S);
                const float tx = to_f32(target_row(target, row0, n_rows, b, G, j, V)[x]);
                logp = kLn2 * (fmaf(tx, c2, -s.m) - log2f(s.S));
                const float logq = draft_logq[(size_t)b * G + j];
                const uint4 w4 = philox4x32_10(make_uint4(0u, (uint32_t)j, id, kStreamAccept), k0, k1);
                pass = word_to_uniform(w4.x) < expf(logp - logq);
                lse_out = kLn2 * lse2;
            } else {
                lse_out = s.key;
                logp = (s.idx == x) ? 0.f : -INFINITY;
                pass = (s.idx == x);
                amax = s.idx;
            }
        }
        const unsigned int fail = __ballot_sync(0xffffffffu, tested && !pass);
        const int first = fail ? j0 + __ffs(fail) - 1 : INT_MAX;  // the first failing row
        if (tested && j <= first) {
            if (target_lse) target_lse[(size_t)b * (G + 1) + j] = lse_out;
            if (logp_sel) logp_sel[(size_t)b * G + j] = logp;
        }
        if (fail) {
            k = first;
            if (T > 0.f) {
                d = first;
                if (j == first) lse_t_row[b] = lse2;
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
        RowState s = row_state_init();
        const RowState *pr = part + ((size_t)b * (G + 1) + L) * nsplit;
        for (int i = lane; i < nsplit; i += 32) row_state_merge(s, pr[i]);
        s = warp_merge(s);
        y = s.idx;
        if (lane == 0 && target_lse) target_lse[(size_t)b * (G + 1) + L] = s.key;
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
// Final draw with CUDA cores: residual rows take the draft logits of the
// rejected row from the stored draft logits (any dtype) or rebuild them with
// FMAs (fp32 weights); bonus rows draw from the target row L.
template <typename TIn>
__global__ void __launch_bounds__(kResThreads)
verify_final_simt_kernel(const TIn *__restrict__ target, const int64_t *__restrict__ row0, int64_t n_rows,
                         const TIn *__restrict__ base,
                         const TIn *__restrict__ e_in, const TIn *__restrict__ w_out,
                         const float *__restrict__ z_in, const int32_t *__restrict__ anchor,
                         const int32_t *__restrict__ draft_tokens, const float *__restrict__ draft_lse,
                         const float *__restrict__ temperature, const uint32_t *__restrict__ request_id,
                         const int32_t *__restrict__ final_code, const float *__restrict__ lse_t_row,
                         int B, int G, int V, int r, uint32_t k0, uint32_t k1, int chunk, int nsplit,
                         ResidualState *__restrict__ part) {
    extern __shared__ float a_row[];  // [r]
    __shared__ ResidualState scratch[kResThreads / 32];
    const int b = blockIdx.x;  // requests along x, segments along y
    const int code = final_code[b];
    if (code < 0) return;
    const int kind = code >> 16, d = code & 0xFFFF;
    const int seg = blockIdx.y;
    const float c2 = kLog2e / temperature[b];
    const uint32_t id = request_id ? request_id[b] : (uint32_t)b;
    const bool residual = (kind == 1);
    const float lse_q2 = residual ? draft_lse[(size_t)b * G + d] * kLog2e : INFINITY;
    const float lse_t2 = residual ? lse_t_row[b] : 0.f;
    if (residual && !z_in) {
        const int prev = (d == 0) ? anchor[b] : draft_tokens[(size_t)b * G + d - 1];
        for (int k = threadIdx.x; k < r; k += blockDim.x) a_row[k] = to_f32(e_in[(size_t)prev * r + k]);
    }
    __syncthreads();
    const size_t drow = (size_t)b * G + d;
    const TIn *t_row = target_row(target, row0, n_rows, b, G, d, V);  // checked by the decide kernel
    const uint32_t stream = residual ? kStreamResidual : kStreamBonus;
    const int vb = seg * chunk;  // a multiple of 16: whole draw groups
    const int ve = min(V, vb + chunk);
    const int lane = threadIdx.x & 31;
    ResidualState st = residual_init();
    // One 16-token draw group (R2b) per quad of lanes, four tokens each.  A
    // residual row weighs token v by r_v = p_v - q_v where positive (p and q
    // normalised); a bonus row by 2^(t_v c2 - tref) with the group's maximum
    // as tref.  Every thread runs the same iterations (the quads shuffle).
    for (int vbase = vb; vbase < ve; vbase += 4 * kResThreads) {
        const int v = vbase + 4 * threadIdx.x;
        const bool valid = v < ve;  // V % 8 == 0: all four tokens or none
        float t[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        float z[4] = {0.f, 0.f, 0.f, 0.f};
        if (valid) {
            const float4 t4 = load4(t_row + v);
#pragma unroll
            for (int e = 0; e < 4; ++e) t[e] = elem(t4, e);
        }
        if (valid && residual) {
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
        float tref = lse_t2, off = 0.f;
        if (!residual) {
            float tm = fmaxf(fmaxf(t[0], t[1]), fmaxf(t[2], t[3]));
            tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 1));
            tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 2));
            tref = off = tm * c2;
        }
        float w4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float we = 0.f;
            if (valid) {
                if (residual) {
                    // p (1 - 2^-delta), delta = log2 p - log2 q from the logits first
                    const float delta2 = fmaf(t[e] - z[e], c2, lse_q2 - lse_t2);
                    if (delta2 > 0.f)
                        we = exp2f(fmaf(t[e], c2, -lse_t2)) * (delta2 > 24.f ? 1.f : -expm1f(-delta2 * kLn2));
                } else {
                    we = exp2f(fmaf(t[e], c2, -tref));
                }
            }
            w4[e] = we;
        }
        float gs = ((w4[0] + w4[1]) + w4[2]) + w4[3];
        gs += __shfl_xor_sync(0xffffffffu, gs, 1);
        gs += __shfl_xor_sync(0xffffffffu, gs, 2);
        const bool leader = (lane & 3) == 0;
        bool take = false;
        float key = -INFINITY;
        uint4 wd = make_uint4(0u, 0u, 0u, 0u);
        if (leader && valid && gs > 0.f) {
            wd = philox4x32_10(make_uint4((uint32_t)v >> 4, (uint32_t)d, id, stream), k0, k1);
            key = off + log2f(gs) - log2f(neg_log_uniform(wd.x));
            take = key > st.key_res;  // an exact tie keeps the earlier, lower-numbered group
        }
        if (!__any_sync(0xffffffffu, take)) continue;
        float wq[16];
#pragma unroll
        for (int qd = 0; qd < 4; ++qd)
#pragma unroll
            for (int e = 0; e < 4; ++e) wq[4 * qd + e] = __shfl_sync(0xffffffffu, w4[e], (lane & ~3) + qd);
        if (!take) continue;
        float run = 0.f;
#pragma unroll
        for (int i2 = 0; i2 < 16; ++i2) run += wq[i2];
        const float target = word_to_uniform(wd.y) * run;
        int x = -1, last = 0;
        run = 0.f;
#pragma unroll
        for (int i2 = 0; i2 < 16; ++i2) {
            run += wq[i2];
            if (wq[i2] > 0.f) last = i2;
            if (x < 0 && run > target) x = i2;
        }
        if (x < 0) x = last;  // target rounded up to the group's sum
        st.key_res = key;
        st.idx_res = v + x;
    }
    st = residual_warp_merge(st);
    const int warp = threadIdx.x >> 5;
    if (lane == 0) scratch[warp] = st;
    __syncthreads();
    if (warp == 0) {
        st = (lane < kResThreads / 32) ? scratch[lane] : residual_init();
        st = residual_warp_merge(st);
        if (lane == 0) part[(size_t)b * nsplit + seg] = st;
    }
}

// One warp per request with a final draw: merge the partials, emit the token.
// If a residual row had no entry with p > q at all (impossible in exact
// arithmetic after a rejection), the token is drawn from p with the residual
// stream instead (a group draw over the target row, here).
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
    ResidualState s = residual_init();
    for (int i = lane; i < nsplit; i += 32) residual_merge(s, part[(size_t)b * nsplit + i]);
    s = residual_warp_merge(s);
    int y = s.idx_res;
    if (y == INT32_MAX) {  // degenerate residual: a group draw from p (stream 2)
        const int d = code & 0xFFFF;
        const float c2 = kLog2e / temperature[b];
        const uint32_t id = request_id ? request_id[b] : (uint32_t)b;
        const TIn *t_row = target_row(target, row0, n_rows, b, G, d, V);
        // each lane keys its own groups, then the warp keeps the best (lowest
        // group on ties) and resolves its token
        float kb = -INFINITY;
        int gb = INT32_MAX;
        for (int g0 = 16 * lane; g0 < V; g0 += 16 * 32) {
            const int g1 = min(g0 + 16, V);
            float m = -INFINITY;
            for (int v = g0; v < g1; ++v) m = fmaxf(m, to_f32(t_row[v]) * c2);
            float S = 0.f;
            for (int v = g0; v < g1; ++v) S += exp2f(fmaf(to_f32(t_row[v]), c2, -m));
            const uint4 wd = philox4x32_10(make_uint4((uint32_t)g0 >> 4, (uint32_t)d, id, kStreamResidual), k0, k1);
            const float key = m + log2f(S) - log2f(neg_log_uniform(wd.x));
            if (key > kb) {
                kb = key;
                gb = g0;
            }
        }
#pragma unroll
        for (int mask = 16; mask > 0; mask >>= 1) {
            const float ko = __shfl_xor_sync(0xffffffffu, kb, mask);
            const int go = __shfl_xor_sync(0xffffffffu, gb, mask);
            if (key_better(ko, go, kb, gb)) {
                kb = ko;
                gb = go;
            }
        }
        const int g1 = min(gb + 16, V);
        float m = -INFINITY;
        for (int v = gb; v < g1; ++v) m = fmaxf(m, to_f32(t_row[v]) * c2);
        float S = 0.f;
        for (int v = gb; v < g1; ++v) S += exp2f(fmaf(to_f32(t_row[v]), c2, -m));
        const uint4 wd = philox4x32_10(make_uint4((uint32_t)gb >> 4, (uint32_t)d, id, kStreamResidual), k0, k1);
        const float tgt = word_to_uniform(wd.y) * S;
        float run = 0.f;
        y = g1 - 1;
        for (int v = gb; v < g1; ++v) {
            run += exp2f(fmaf(to_f32(t_row[v]), c2, -m));
            if (run > tgt) {
                y = v;
                break;
            }
        }
    }
    if (lane == 0) out_tokens[(size_t)b * (G + 1) + accept_len[b]] = y;
}

// Beside the draft kernel the blocks must share an SM with a draft CTA, which
// runs with the largest shared-memory carveout; a block that reached an SM
// first under a smaller carveout would keep the draft CTA off it.
template <typename TIn>
cudaError_t set_rows_carveout() {
    static PerDeviceOnce once;
    return once.run([] {
        return cudaFuncSetAttribute(verify_rows_kernel<TIn>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                    (int)cudaSharedmemCarveoutMaxShared);
    });
}

template <typename TIn>
cudaError_t launch_verify_rows_t(const VerifyArgs &a, const VerifyPlan &p, bool beside, cudaStream_t s) {
    if (beside) {
        const cudaError_t e = set_rows_carveout<TIn>();
        if (e != cudaSuccess) return e;
    }
    RowState *row_part = reinterpret_cast<RowState *>(a.ws + p.row_part_offset);
    const TIn *target = static_cast<const TIn *>(a.target);
    const long units = (long)a.B * (a.G + 1) * p.row_split;
    // beside the draft kernel: one block per SM, which fits next to a draft CTA
    const dim3 grid = beside ? dim3((unsigned int)(units < kNumSMs ? units : kNumSMs))
                             : dim3((unsigned int)(a.B * (a.G + 1)), (unsigned int)p.row_split);
    verify_rows_kernel<TIn><<<grid, kRowThreads, 0, s>>>(target, a.target_row0, a.n_target_rows, a.verify_len,
                                                         a.temperature, a.B, a.G, a.V, p.row_chunk, p.row_split,
                                                         row_part);
    return cudaGetLastError();
}

template <typename TIn>
cudaError_t launch_verify_finish_t(const VerifyArgs &a, const VerifyPlan &p, cudaStream_t s) {
    uint32_t *flags = reinterpret_cast<uint32_t *>(a.ws);
    RowState *row_part = reinterpret_cast<RowState *>(a.ws + p.row_part_offset);
    int32_t *final_code = reinterpret_cast<int32_t *>(a.ws + p.res_row_offset);
    float *lse_t_row = reinterpret_cast<float *>(a.ws + p.lse_t_offset);
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

cudaError_t launch_verify_rows(const VerifyArgs &a, const VerifyPlan &p, bool beside, cudaStream_t s) {
    if (a.dt == DSPARK_BF16) return launch_verify_rows_t<__nv_bfloat16>(a, p, beside, s);
    return launch_verify_rows_t<float>(a, p, beside, s);
}

cudaError_t launch_verify_finish(const VerifyArgs &a, const VerifyPlan &p, cudaStream_t s) {
    if (a.dt == DSPARK_BF16) return launch_verify_finish_t<__nv_bfloat16>(a, p, s);
    return launch_verify_finish_t<float>(a, p, s);
}

cudaError_t launch_verify(const VerifyArgs &a, const VerifyPlan &p, cudaStream_t s) {
    cudaError_t e = launch_verify_rows(a, p, false, s);
    if (e != cudaSuccess) return e;
    return launch_verify_finish(a, p, s);
}

VerifyPlan plan_verify(int B, int G, int V, int r, dspark_dtype dt) {
    (void)r;
    VerifyPlan p{};
    const long rows = (long)B * (G + 1);
    // target rows: aim for ~8 blocks per SM among the rows that are read
    // (about half of them with scheduled lengths), segments >= 4096 entries
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
    int rchunk = ((V + rs - 1) / rs + 15) / 16 * 16;  // whole draw groups per segment
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
    off = align_up(off + sizeof(float) * (size_t)B, 256);
    p.res_part_offset = off;
    off = align_up(off + sizeof(ResidualState) * (size_t)B * res_slots, 256);
    p.res_best_offset = off;
    off = align_up(off + sizeof(uint32_t) * (size_t)B, 256);
    p.ws_bytes = off;
    return p;
}

}  // namespace dspark

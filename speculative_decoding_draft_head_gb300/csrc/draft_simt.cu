// Draft sampling, SIMT form (fp32 weights), plus the split-vocabulary merge
// shared with the tensor-core form.
//
// Method: "DSpark, la bozza che sa quando fermarsi" (paithon.it), section
// "Un po' di autoregressione basta", equation for p_k: position j draws from
// softmax((U_j + E_in[x_{j-1}] W_out^T) / T); the drawn token feeds position j+1.
//
// One launch per block position.  A block owns `rows_per_block` requests and
// one vocabulary segment: it gathers the E_in rows of the previous tokens into
// shared memory, forms the rank-r bias with register-tiled FMAs (4 vocabulary
// entries x rows_per_block requests per thread, W_out rows read along r), adds
// the base logits and streams every logit once through the online softmax and
// the per-token Gumbel-max draw (one Philox block gives the words of a
// thread's four tokens).  The per-(request, segment) partial states are
// merged by draft_finalize, which writes the token the next position reads.
// bf16 weights take the tensor-core kernel (markov_tc.cu) instead.
#include <climits>

#include "device_common.cuh"
#include "internal.h"

namespace dspark {
namespace {

constexpr int kSimtThreads = 256;
constexpr int kSimtRows = 8;

// The exact key word of draft token v with logit z and word w: z / T + g(u)
// in float-float.  Out of line: it runs for few tokens, and inlined at each of
// the kernel's unrolled call sites it would bloat the code (a launch fetches
// its instructions cold).
static __device__ __noinline__ unsigned long long draft_key_word(float z, float T, float rT, uint32_t w, int v,
                                                                 float *key_hi) {
    const FF key = ff_add(div_ff(z, T, rT), gumbel_ff(w));
    *key_hi = key.hi;
    return key_word(key, v);
}

// Online softmax and per-token Gumbel-max for four consecutive tokens
// v .. v + 3 of one row (T > 0, c2 = log2(e) / T, rT = fl(1 / T)); w holds
// their draft-stream words; lanes with valid = false hold no tokens.  Every
// lane of the warp calls it together (it reduces across the warp).  A token is
// screened without a logarithm against the best key K this thread knows for
// the row, (1 - u) < e Q with e = 2^(s2 - m) and Q = 2^(m - K log2 e)
// (E = -ln u >= 1 - u, so no winner is lost).  A survivor gets an fp32 key;
// the warp's largest fp32 key, less its error bound, is a lower bound of an
// exact key that its own lane forms below, so only tokens that can reach it
// form a float-float key, and the key words decide.
__device__ __forceinline__ void simt_draw4(RowState &st, float &kbest, const float (&z)[4], float2 c2, float T,
                                           float rT, int v, const uint4 &w, bool valid) {
    float e[4];
    if (valid) softmax_push_group<4>(st, z, c2.x, c2.y, e);
    const float Q = screen_q(st.m, kbest);
    float k2[4];
    float wm = -INFINITY;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t wi = i == 0 ? w.x : (i == 1 ? w.y : (i == 2 ? w.z : w.w));
        k2[i] = -INFINITY;
        if (valid && one_minus_uniform_plus_one(wi) < fmaf(e[i], Q, 1.f)) {
            k2[i] = fmaf(z[i], c2.x, -fast_log2(neg_log_uniform(wi)));
            wm = fmaxf(wm, k2[i]);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
    const float wlow = wm - key_tol2(wm, wm);  // log2 units; -inf when no lane has a survivor
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float K2 = fmaxf(kbest * kLog2e, wlow);
        if (!(k2[i] > K2 - key_tol2(k2[i], K2))) continue;
        const uint32_t wi = i == 0 ? w.x : (i == 1 ? w.y : (i == 2 ? w.z : w.w));
        float key_hi;
        const unsigned long long word = draft_key_word(z[i], T, rT, wi, v + i, &key_hi);
        if (word > st.best) {
            st.best = word;
            st.z_at = z[i];
            kbest = fmaxf(kbest, key_hi);
        }
    }
    // the warp's bound, in natural-log units, screens this thread's next tokens
    if (wlow > -INFINITY) kbest = fmaxf(kbest, wlow * kLn2 - 1e-6f * fabsf(wlow));
}

static_assert(kSimtThreads / 32 == kSimtRows, "one warp draws each row of the block");

// x_j, lse_j and log q_j of one request from its merged draw: bw the largest
// key word (0: the request was flagged invalid), zat its token's logit, lse_ff
// the row's log-sum-exp of z/T (T > 0).
__device__ __forceinline__ void write_draft_row(unsigned long long bw, float zat, FF lse_ff, float T, size_t o,
                                                int32_t *tokens, float *lse, float *logq) {
    if (bw == 0ull) {
        tokens[o] = -1;
        lse[o] = __int_as_float(0x7fc00000);
        logq[o] = __int_as_float(0x7fc00000);
        return;
    }
    tokens[o] = word_token(bw);
    if (T > 0.f) {
        lse[o] = lse_ff.hi;
        logq[o] = ff_add(div_ff(zat, T, __frcp_rn(T)), ff_neg(lse_ff)).hi;
    } else {
        lse[o] = zat;
        logq[o] = 0.f;
    }
}

// Two phases per 4 kSimtThreads tokens of the segment: every thread forms the
// logits of four tokens for all rows of the block (the rank-r bias
// register-tiled over the rows, so each W_out row is read once per block) into
// shared memory; then warp w draws row w over those tokens (softmax and
// per-token Gumbel-max), its lanes taking groups of four tokens in turn.  One
// copy of the draw code serves every row: the kernel is small enough that a
// launch does not wait on instruction fetch, and each row's state stays in its
// warp's registers.
template <typename TIn>
__global__ void __launch_bounds__(kSimtThreads)
draft_simt_kernel(const TIn *__restrict__ base, const TIn *__restrict__ e_in,
                  const TIn *__restrict__ w_out, const int32_t *__restrict__ anchor,
                  const int32_t *__restrict__ tokens, const float *__restrict__ temperature,
                  const uint32_t *__restrict__ request_id, int B, int G, int V, int r, int j,
                  uint32_t k0, uint32_t k1, int chunk, int nsplit, RowState *__restrict__ part,
                  uint32_t *__restrict__ flags, float *__restrict__ z_out, int32_t *__restrict__ tokens_out,
                  float *__restrict__ lse_out, float *__restrict__ logq_out, int j_end) {
    extern __shared__ float smem_f[];
    float *a_rows = smem_f;                       // [kSimtRows][r]
    float *zs = smem_f + (size_t)kSimtRows * r;   // [kSimtRows][4 kSimtThreads] logits of the current tokens
    __shared__ int prev_s[kSimtRows];
    __shared__ int next_s[kSimtRows];             // each row's token of the position just drawn
    __shared__ float2 c2_s[kSimtRows];
    __shared__ float T_s[kSimtRows];
    __shared__ uint32_t rid_s[kSimtRows];

    const int b0 = blockIdx.y * kSimtRows;
    const int seg = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Positions j0 .. j_end - 1: more than one only when this block's segment
    // covers the whole row (tokens_out set), so the block draws each next token
    // itself; it passes it on through shared memory (tokens is read-only here).
    const int j0 = j;
    for (j = j0; j < j_end; ++j) {
    if (threadIdx.x < kSimtRows) {
        const int b = b0 + threadIdx.x;
        int prev = -1;
        float2 c2 = make_float2(0.f, 0.f);
        uint32_t id = 0;
        if (b < B) {
            prev = (j == 0) ? anchor[b] : (j > j0 ? next_s[threadIdx.x] : tokens[(size_t)b * G + j - 1]);
            const float T = temperature[b];
            id = request_id ? request_id[b] : (uint32_t)b;
            const bool bad_prev = prev < 0 || prev >= V;
            // an earlier position already flagged this request and wrote -1
            if (bad_prev && (j == 0 || prev != -1) && seg == 0) atomicOr(flags, kFlagBadToken);
            const bool t_ok = T >= 0.f && !isinf(T);
            if (!t_ok && seg == 0 && j == 0) atomicOr(flags, kFlagBadTemperature);
            if (bad_prev || !t_ok) prev = -1;
            if (T > 0.f && t_ok) c2 = c2_split(T);
        }
        prev_s[threadIdx.x] = prev;
        c2_s[threadIdx.x] = c2;
        T_s[threadIdx.x] = (b < B) ? temperature[b] : 1.f;
        rid_s[threadIdx.x] = id;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kSimtRows * r; i += blockDim.x) {
        const int rb = i / r, k = i - rb * r;
        const int prev = prev_s[rb];
        a_rows[i] = prev >= 0 ? to_f32(e_in[(size_t)prev * r + k]) : 0.f;
    }
    __syncthreads();

    // this warp's row
    const int b_w = b0 + warp;
    const bool row_on = b_w < B && prev_s[warp] >= 0;  // uniform over the warp
    const float2 c2w = c2_s[warp];
    const float T_w = T_s[warp];
    const float rT_w = __frcp_rn(T_w);
    const uint32_t rid_w = rid_s[warp];
    RowState st = row_state_init();
    float kbest = -INFINITY;

    const int vb = seg * chunk;  // a multiple of 16
    const int ve = min(V, vb + chunk);
    for (int vbase = vb; vbase < ve; vbase += 4 * kSimtThreads) {
        // phase 1: the logits of tokens v .. v + 3 for every row of the block
        {
            const int v = vbase + 4 * threadIdx.x;
            if (v < ve) {  // V % 8 == 0: all four tokens or none
                float acc[kSimtRows][4];
#pragma unroll
                for (int rb = 0; rb < kSimtRows; ++rb)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[rb][e] = 0.f;
                for (int k = 0; k < r; k += 4) {
                    float4 w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) w[e] = load4(w_out + (size_t)(v + e) * r + k);
#pragma unroll
                    for (int rb = 0; rb < kSimtRows; ++rb) {
                        const float4 a = *reinterpret_cast<const float4 *>(a_rows + rb * r + k);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            float t = acc[rb][e];
                            t = fmaf(a.x, w[e].x, t);
                            t = fmaf(a.y, w[e].y, t);
                            t = fmaf(a.z, w[e].z, t);
                            t = fmaf(a.w, w[e].w, t);
                            acc[rb][e] = t;
                        }
                    }
                }
#pragma unroll
                for (int rb = 0; rb < kSimtRows; ++rb) {
                    const int b = b0 + rb;
                    if (b >= B || prev_s[rb] < 0) continue;  // uniform over the block
                    const size_t row = (size_t)b * G + j;
                    const float4 u4 = load4(base + row * V + v);
                    const float4 z4 = make_float4(u4.x + acc[rb][0], u4.y + acc[rb][1], u4.z + acc[rb][2],
                                                  u4.w + acc[rb][3]);
                    *reinterpret_cast<float4 *>(zs + rb * (4 * kSimtThreads) + 4 * threadIdx.x) = z4;
                    if (z_out) *reinterpret_cast<float4 *>(z_out + row * V + v) = z4;
                }
            }
        }
        __syncthreads();
        // phase 2: warp w draws row w over these tokens
        if (row_on) {
#pragma unroll 1
            for (int g = lane; g < kSimtThreads; g += 32) {
                const int v = vbase + 4 * g;
                const bool valid = v < ve;
                float z[4] = {0.f, 0.f, 0.f, 0.f};
                if (valid) {
                    const float4 z4 = *reinterpret_cast<const float4 *>(zs + warp * (4 * kSimtThreads) + 4 * g);
                    z[0] = z4.x;
                    z[1] = z4.y;
                    z[2] = z4.z;
                    z[3] = z4.w;
                }
                if (c2w.x > 0.f) {  // uniform over the warp: every lane draws
                    uint4 w = make_uint4(0u, 0u, 0u, 0u);
                    if (valid)
                        w = philox4x32_10(make_uint4((uint32_t)v >> 2, (uint32_t)j, rid_w, kStreamDraft), k0, k1);
                    simt_draw4(st, kbest, z, c2w, T_w, rT_w, v, w, valid);
                } else if (valid) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) argmax_push(st, z[e], v + e);
                }
            }
        }
        __syncthreads();  // the next tokens' logits overwrite zs
    }
    const RowState m = row_on ? warp_merge(st) : row_state_init();
    if (b_w < B && lane == 0) {
        if (!tokens_out) {
            part[(size_t)b_w * nsplit + seg] = m;
        } else {
            // one segment covers the row: this warp holds the row's whole draw
            const FF lse_ff = (row_on && T_w > 0.f) ? lse_of_partials(&m, 1) : FF{0.f, 0.f};
            write_draft_row(m.best, m.z_at, lse_ff, T_w, (size_t)b_w * G + j, tokens_out, lse_out, logq_out);
            next_s[warp] = word_token(m.best);  // -1 for a flagged request
        }
    }
    __syncthreads();  // next_s is complete; prev_s, a_rows and zs may be overwritten
    }
}

// One warp per (request, position): merge the segment partials, write token,
// lse, logq.  Position j0 + k reads its partials at part + k * pos_stride.
// The token is the largest key word; lse is the partial sums rescaled
// exactly and added in float-float (about 44 bits), and log q = z_x / T - lse
// in float-float, each rounded once to fp32.
__global__ void draft_finalize_kernel(const RowState *__restrict__ part, int nsplit, size_t pos_stride,
                                      const float *__restrict__ temperature, int B, int G, int j0, int npos,
                                      int32_t *__restrict__ tokens, float *__restrict__ lse,
                                      float *__restrict__ logq) {
    griddep_wait();  // a programmatic dependent: the previous launch's writes are visible after this
    const int gw = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (gw >= B * npos) return;  // warp-uniform
    const int k = gw / B, b = gw - k * B, j = j0 + k;
    const RowState *pr = part + (size_t)k * pos_stride + (size_t)b * nsplit;
    const float T = temperature[b];
    const FF lse_ff = (T > 0.f) ? warp_lse_of_partials(pr, nsplit) : FF{0.f, 0.f};
    unsigned long long bw = 0ull;
    float zat = 0.f;
    for (int i = lane; i < nsplit; i += 32)
        if (pr[i].best > bw) {
            bw = pr[i].best;
            zat = pr[i].z_at;
        }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
        const unsigned long long ob = __shfl_xor_sync(0xffffffffu, bw, m);
        const float oz = __shfl_xor_sync(0xffffffffu, zat, m);
        if (ob > bw) {
            bw = ob;
            zat = oz;
        }
    }
    if (lane != 0) return;
    write_draft_row(bw, zat, lse_ff, T, (size_t)b * G + j, tokens, lse, logq);
}

}  // namespace

bool simt_writes_rows(const DraftPlan &p) { return !p.tensor_path && p.nsplit == 1; }

cudaError_t launch_draft_simt(const DraftArgs &a, const DraftPlan &p, int j, cudaStream_t s) {
    const dim3 grid(p.nsplit, p.row_blocks);
    const size_t smem = sizeof(float) * kSimtRows * ((size_t)a.r + 4 * kSimtThreads);
    // one segment per row: the kernel writes x_j, lse_j and log q_j itself,
    // and walks every position from j in one launch
    const bool direct = simt_writes_rows(p);
    const int j_end = direct ? a.G : j + 1;
    uint32_t *flags = reinterpret_cast<uint32_t *>(a.ws);
    RowState *part = reinterpret_cast<RowState *>(a.ws + p.partial_offset);
    const uint32_t k0 = (uint32_t)(a.seed & 0xFFFFFFFFu), k1 = (uint32_t)(a.seed >> 32);
    if (a.dt == DSPARK_BF16) {
        draft_simt_kernel<__nv_bfloat16><<<grid, kSimtThreads, smem, s>>>(
            (const __nv_bfloat16 *)a.base, (const __nv_bfloat16 *)a.e_in, (const __nv_bfloat16 *)a.w_out,
            a.anchor, a.tokens, a.temperature, a.request_id, a.B, a.G, a.V, a.r, j, k0, k1, p.chunk,
            p.nsplit, part, flags, a.z_out, direct ? a.tokens : nullptr, a.lse, a.logq, j_end);
    } else {
        draft_simt_kernel<float><<<grid, kSimtThreads, smem, s>>>(
            (const float *)a.base, (const float *)a.e_in, (const float *)a.w_out, a.anchor, a.tokens,
            a.temperature, a.request_id, a.B, a.G, a.V, a.r, j, k0, k1, p.chunk, p.nsplit, part, flags,
            a.z_out, direct ? a.tokens : nullptr, a.lse, a.logq, j_end);
    }
    return cudaGetLastError();
}

cudaError_t launch_draft_finalize(const DraftArgs &a, const DraftPlan &p, int j, int npos, cudaStream_t s) {
    // the tensor path keeps every position's partials ([G][B][nsplit]); the
    // SIMT path reuses one [B][nsplit] array per position
    const RowState *part = reinterpret_cast<const RowState *>(a.ws + p.partial_offset);
    const size_t pos_stride = p.tensor_path ? (size_t)a.B * p.nsplit : 0;
    if (p.tensor_path) part += (size_t)j * pos_stride;
    const int warps = 4;
    const int rows = a.B * npos;
    return launch_dependent(draft_finalize_kernel, dim3((rows + warps - 1) / warps), dim3(32 * warps), 0, s, part,
                            p.nsplit, pos_stride, a.temperature, a.B, a.G, j, npos, a.tokens, a.lse, a.logq);
}

DraftPlan plan_draft(int B, int G, int V, int r, dspark_dtype dt) {
    (void)r;
    DraftPlan p{};
    if (dt == DSPARK_BF16) {
        p.tensor_path = true;
        p.rows_per_block = 128;
        p.row_blocks = tc_row_blocks(B);
        p.nsplit = tc_segments(B, V);
        p.chunk = 0;
    } else {
        p.tensor_path = false;
        p.rows_per_block = kSimtRows;
        p.row_blocks = (B + kSimtRows - 1) / kSimtRows;
        const int want_blocks = 2 * kNumSMs;
        int nsplit = (want_blocks + p.row_blocks - 1) / p.row_blocks;
        const int max_split = (V + 1023) / 1024;
        if (nsplit > max_split) nsplit = max_split;
        if (nsplit < 1) nsplit = 1;
        int chunk = (V + nsplit - 1) / nsplit;
        chunk = (chunk + 15) / 16 * 16;
        p.nsplit = (V + chunk - 1) / chunk;
        p.chunk = chunk;
    }
    // flag words, then (tensor path) the best words and barrier counters, so
    // that one clear of clear_bytes from offset 0 covers all three, then the
    // partials
    const size_t npart = (size_t)B * p.nsplit * (p.tensor_path ? (size_t)G : 1);
    p.best_offset = kFlagBytes;
    const size_t words = p.tensor_path ? sizeof(unsigned long long) * (size_t)B * (size_t)G : 0;
    p.bar_offset = p.best_offset + words;  // 8-byte aligned
    const size_t bars = p.tensor_path ? sizeof(unsigned int) * (size_t)p.row_blocks : 0;
    p.clear_bytes = p.bar_offset + bars;
    p.partial_offset = align_up(p.clear_bytes, 256);
    p.ws_bytes = align_up(p.partial_offset + sizeof(RowState) * npart, 256);
    return p;
}

}  // namespace dspark

// Recurrent draft head: the state update between block positions.
//
// Method: "DSpark, la bozza che sa quando fermarsi" (paithon.it), section
// "Un po' di autoregressione basta" (with the aitalk overview "Un drafter..."):
// beside the Markov head, whose bias at position j depends on x_{j-1} alone,
// the pages name a recurrent head that carries a state along the block.  They
// do not give its cell; the one computed here is an Elman cell whose input
// term is the previous token's embedding, kept in bf16 like the head's weights:
//     h_{-1} = 0,   h_j = bf16(tanh(E_in[x_{j-1}] + W_h h_{j-1})),
// W_h [r][r] with row n the weights of state unit n.  The draft kernel then
// forms bias_j = h_j W_out^T on the tensor cores with h_j as its A operand
// (launch_draft_tensor_rows), so everything after the state is the Markov
// head's path unchanged.
//
// Precision.  The products of two bf16 values are exact in fp32; they are
// summed with compensated two-sum chains (error about 2^-48 of the sum of
// magnitudes).  tanh is taken in fp32 unless the result lies within a few
// fp32 units of a bf16 rounding midpoint, where it is taken in fp64 and
// rounded once to bf16 from fp64 (about 1 value in 4000; GB300's fp64 rate
// makes an fp64 tanh for every value cost more than the whole dot product).
// A state therefore differs from the exactly rounded one only when its
// pre-rounding value lies within about 1e-13 (relative) of a rounding
// boundary.  (A faster-issuing variant, FMA chains with a running error bound
// and a two-sum recompute of the undecided values, measured no faster: the
// kernel is bound by latency at one block per SM, not by issue.)
//
// Work per position is B r^2 multiply-adds (16.8 M at B = r = 256): a small
// SIMT kernel, one thread per state unit and R requests per block, with W_h
// staged once per block in shared memory.
#include "device_common.cuh"
#include "internal.h"

namespace dspark {
namespace {

constexpr int kRnnThreads = 256;  // >= r: one thread per state unit

// Adds p to the compensated pair (s, c) with Knuth's two-sum: the new s plus
// the rounding error e of s + p is exactly the old s plus p, and e goes into c
// (round-to-nearest; the _rn intrinsics keep the compiler from fusing steps).
__device__ __forceinline__ void two_sum_acc(float &s, float &c, float p) {
    const float t = __fadd_rn(s, p);
    const float bp = __fsub_rn(t, s);
    const float e = __fadd_rn(__fsub_rn(s, __fsub_rn(t, bp)), __fsub_rn(p, bp));
    c = __fadd_rn(c, e);
    s = t;
}

// Round a double to bf16 (8 significant bits), ties to even, for normal
// values; the result is exact in fp32 and hence in bf16.
__device__ __forceinline__ __nv_bfloat16 double_to_bf16_rne(double x) {
    unsigned long long u = (unsigned long long)__double_as_longlong(x);
    const unsigned long long lsb = (u >> 45) & 1ull;  // 52 - 7 fraction bits dropped
    u += (1ull << 44) - 1ull + lsb;
    u &= ~((1ull << 45) - 1ull);
    return __float2bfloat16_rn((float)__longlong_as_double((long long)u));
}

// fp32 units (within a binade) between a tanhf result and the nearest bf16
// rounding midpoint below which the fp64 path decides the rounding: tanhf is
// within 2 ulp (CUDA's documented bound) and the fp32 argument adds at most
// 1 ulp of the result (|d tanh / da| * |a| <= |tanh a|), so 8 leaves a factor
// of two over the worst case
constexpr int kTanhGuard = 8;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// W_h rows in shared memory: 2 r bytes + 16 of padding, so that the 16-byte
// loads of eight consecutive threads (eight rows) fall on distinct banks
__host__ __device__ constexpr int w_row_bytes(int r) { return 2 * r + 16; }
size_t state_smem_bytes(int R, int r) { return (size_t)r * w_row_bytes(r) + sizeof(float) * (size_t)R * r; }

// One block: R requests, thread n = state unit n.  W_h (all r rows) is
// staged in shared memory with coalesced asynchronous copies; each thread
// then reads its own row from there.
template <int R>
__global__ void __launch_bounds__(kRnnThreads)
rnn_state_kernel(const __nv_bfloat16 *__restrict__ e_in, const __nv_bfloat16 *__restrict__ w_h,
                 const int32_t *__restrict__ anchor, const unsigned long long *__restrict__ best,
                 const __nv_bfloat16 *__restrict__ h_prev, __nv_bfloat16 *__restrict__ h_next,
                 __nv_bfloat16 *__restrict__ h_out, int B, int G, int V, int r, int j) {
    extern __shared__ __align__(16) unsigned char smem[];
    unsigned char *wsm = smem;                                            // [r][w_row_bytes]
    float *hs = reinterpret_cast<float *>(smem + (size_t)r * w_row_bytes(r));  // [R][r]: h_{j-1}
    __shared__ int prev_s[R];
    // the draw of this position (the next launch) may start its prologue
    if (threadIdx.x == 0) griddep_launch_dependents();
    const int n = threadIdx.x;
    if (j > 0) {
        // W_h is an input: its copy may start before the previous kernel ends
        const int parts = r / 8;  // 16-byte pieces per row
        const uint32_t wbase = (uint32_t)__cvta_generic_to_shared(wsm);
        for (int idx = threadIdx.x; idx < r * parts; idx += blockDim.x) {
            const int row = idx / parts, part = idx - row * parts;
            cp_async16(wbase + (uint32_t)(row * w_row_bytes(r) + part * 16), w_h + (size_t)row * r + part * 8);
        }
    }
    griddep_wait();
    const int b0 = blockIdx.x * R;
    if (threadIdx.x < R) {
        const int b = b0 + threadIdx.x;
        int prev = -1;
        if (b < B) {
            // x_{j-1}: the anchor, else the token drawn at position j - 1 (the
            // row-wide best word of the previous draft launch)
            prev = (j == 0) ? anchor[b] : word_token(best[(size_t)(j - 1) * B + b]);
            if (prev < 0 || prev >= V) prev = -1;
        }
        prev_s[threadIdx.x] = prev;
    }
    for (int i = threadIdx.x; i < R * r; i += blockDim.x) {
        const int rr = i / r, k = i - rr * r;
        const int b = b0 + rr;
        hs[i] = (j > 0 && b < B) ? __bfloat162float(h_prev[(size_t)b * r + k]) : 0.f;
    }
    cp_async_wait_all();
    __syncthreads();
    if (n >= r) return;

    // four interleaved compensated sums per request (k mod 4) keep four
    // independent dependency chains in flight; merged exactly at the end
    float s[R][4], c[R][4];
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) s[i][q] = c[i][q] = 0.f;
    if (j > 0) {
        const uint4 *wrow = reinterpret_cast<const uint4 *>(wsm + (size_t)n * w_row_bytes(r));
#pragma unroll 2
        for (int k8 = 0; k8 < r / 8; ++k8) {
            const uint4 w4 = wrow[k8];
            const uint32_t ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
            for (int i = 0; i < R; ++i) {
                const float4 h0 = *reinterpret_cast<const float4 *>(hs + i * r + 8 * k8);
                const float4 h1 = *reinterpret_cast<const float4 *>(hs + i * r + 8 * k8 + 4);
                const float hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float w = (e & 1) ? bf16_hi(ww[e >> 1]) : bf16_lo(ww[e >> 1]);
                    two_sum_acc(s[i][e & 3], c[i][e & 3], __fmul_rn(w, hv[e]));
                }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const int b = b0 + i;
        if (b >= B) break;
        const int prev = prev_s[i];
        __nv_bfloat16 h = __float2bfloat16_rn(0.f);
        if (prev >= 0) {
            float sm = s[i][0], cm = c[i][0] + c[i][1] + c[i][2] + c[i][3];
            two_sum_acc(sm, cm, s[i][1]);
            two_sum_acc(sm, cm, s[i][2]);
            two_sum_acc(sm, cm, s[i][3]);
            const double a = (double)__bfloat162float(e_in[(size_t)prev * r + n]) + (double)sm + (double)cm;
            const float t = tanhf((float)a);
            const int mid = abs((int)(__float_as_uint(t) & 0xFFFFu) - 0x8000);
            h = (mid > kTanhGuard) ? __float2bfloat16_rn(t) : double_to_bf16_rne(tanh(a));
        }
        h_next[(size_t)b * r + n] = h;
        if (h_out) h_out[((size_t)b * G + j) * r + n] = h;
    }
}

template <int R>
cudaError_t launch_rnn_r(const RnnStateArgs &a, int j, cudaStream_t s) {
    const size_t smem = state_smem_bytes(R, a.r);
    static PerDeviceOnce once;  // the limit for the largest r
    cudaError_t e = once.run([] {
        return cudaFuncSetAttribute(rnn_state_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)state_smem_bytes(R, 256));
    });
    if (e != cudaSuccess) return e;
    const int blocks = (a.B + R - 1) / R;
    const __nv_bfloat16 *h_prev = a.h_ws + (size_t)(j > 0 ? j - 1 : 0) * a.B * a.r;
    rnn_state_kernel<R><<<blocks, kRnnThreads, smem, s>>>(a.e_in, a.w_h, a.anchor, a.best, h_prev,
                                                          a.h_ws + (size_t)j * a.B * a.r, a.h_out, a.B, a.G,
                                                          a.V, a.r, j);
    return cudaGetLastError();
}

}  // namespace

RnnPlan plan_draft_rnn(int B, int G, int V, int r) {
    RnnPlan p{};
    p.draft = plan_draft(B, G, V, r, DSPARK_BF16);
    p.h_offset = align_up(p.draft.ws_bytes, 256);
    p.ws_bytes = align_up(p.h_offset + sizeof(__nv_bfloat16) * (size_t)G * (size_t)B * (size_t)r, 256);
    return p;
}

int rnn_rows_per_block(int B) {
    // a block fills an SM's shared memory with W_h: one wave of at most one
    // block per SM, and as few W_h copies as that allows
    int R = 1;
    while (R < 8 && (B + R - 1) / R > kNumSMs) R <<= 1;
    return R;
}

cudaError_t launch_rnn_state(const RnnStateArgs &a, int j, cudaStream_t s) {
    switch (rnn_rows_per_block(a.B)) {
        case 8: return launch_rnn_r<8>(a, j, s);
        case 4: return launch_rnn_r<4>(a, j, s);
        case 2: return launch_rnn_r<2>(a, j, s);
        default: return launch_rnn_r<1>(a, j, s);
    }
}

}  // namespace dspark

// Device helpers shared by the draft, verify and schedule kernels.
//
// Random stream: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random
// Numbers: As Easy as 1, 2, 3", SC'11) keyed by the 64-bit seed, counter =
// (v >> 2, position, request id, stream), word v & 3; the uniform keeps the
// top 23 bits of the word and centres it in its cell: u = (k + 1/2) 2^-23.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace dspark {

constexpr uint32_t kPhiloxM0 = 0xD2511F53u;
constexpr uint32_t kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u;   // golden ratio
constexpr uint32_t kPhiloxW1 = 0xBB67AE85u;   // sqrt(3) - 1

constexpr uint32_t kStreamDraft = 0;
constexpr uint32_t kStreamAccept = 1;
constexpr uint32_t kStreamResidual = 2;
constexpr uint32_t kStreamBonus = 3;

constexpr uint32_t kFlagBadToken = 1u;
constexpr uint32_t kFlagBadTemperature = 2u;
constexpr uint32_t kFlagBadVerifyLen = 4u;
constexpr uint32_t kFlagBadPosTemp = 8u;

// Ten rounds of the Philox4x32 bijection.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t lo0 = kPhiloxM0 * c.x;
        const uint32_t hi0 = __umulhi(kPhiloxM0, c.x);
        const uint32_t lo1 = kPhiloxM1 * c.z;
        const uint32_t hi1 = __umulhi(kPhiloxM1, c.z);
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
        k0 += kPhiloxW0;
        k1 += kPhiloxW1;
    }
    return c;
}

__device__ __forceinline__ uint32_t word_of(const uint4 &w, int e) {
    return e == 0 ? w.x : (e == 1 ? w.y : (e == 2 ? w.z : w.w));
}

// u = ((w >> 9) + 1/2) * 2^-23, exact: 1 + k 2^-23 minus (1 - 2^-24).
__device__ __forceinline__ float word_to_uniform(uint32_t w) {
    return __uint_as_float(0x3F800000u | (w >> 9)) - 0x1.fffffep-1f;
}

// Exponential variate E = -ln u (relative accuracy matters: small E wins).
__device__ __forceinline__ float neg_log_uniform(uint32_t w) {
    return -logf(word_to_uniform(w));
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// Four consecutive elements starting at a 4-aligned index.
__device__ __forceinline__ float4 load4(const float *p) {
    return __ldg(reinterpret_cast<const float4 *>(p));
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16 *p) {
    const uint2 raw = __ldg(reinterpret_cast<const uint2 *>(p));
    float4 f;
    f.x = __uint_as_float(raw.x << 16);
    f.y = __uint_as_float(raw.x & 0xFFFF0000u);
    f.z = __uint_as_float(raw.y << 16);
    f.w = __uint_as_float(raw.y & 0xFFFF0000u);
    return f;
}
__device__ __forceinline__ float elem(const float4 &f, int e) {
    return e == 0 ? f.x : (e == 1 ? f.y : (e == 2 ? f.z : f.w));
}

// Running state of one row segment: online softmax (m, S) and the best key.
struct RowState {
    float m;      // max of s seen
    float S;      // sum of exp(s - m)
    float key;    // best key (Gumbel-perturbed s, or z when greedy)
    float s_at;   // s at the best index
    int idx;      // best index, INT32_MAX if none
    int pad0, pad1, pad2;
};
static_assert(sizeof(RowState) == 32, "RowState is stored as two 16-byte words");

__device__ __forceinline__ RowState row_state_init() {
    RowState st;
    st.m = -INFINITY;
    st.S = 0.f;
    st.key = -INFINITY;
    st.s_at = 0.f;
    st.idx = INT32_MAX;
    st.pad0 = st.pad1 = st.pad2 = 0;
    return st;
}

__device__ __forceinline__ bool key_better(float ka, int ia, float kb, int ib) {
    return ka > kb || (ka == kb && ia < ib);
}

// Merge b into a (associative; ties on the key go to the lower index).
__device__ __forceinline__ void row_state_merge(RowState &a, const RowState &b) {
    const float m = fmaxf(a.m, b.m);
    if (m != -INFINITY) {
        const float sa = (a.m == -INFINITY) ? 0.f : a.S * expf(a.m - m);
        const float sb = (b.m == -INFINITY) ? 0.f : b.S * expf(b.m - m);
        a.S = sa + sb;
        a.m = m;
    }
    if (key_better(b.key, b.idx, a.key, a.idx)) {
        a.key = b.key;
        a.s_at = b.s_at;
        a.idx = b.idx;
    }
}

__device__ __forceinline__ RowState shfl_xor_state(const RowState &s, int mask) {
    RowState o;
    o.m = __shfl_xor_sync(0xffffffffu, s.m, mask);
    o.S = __shfl_xor_sync(0xffffffffu, s.S, mask);
    o.key = __shfl_xor_sync(0xffffffffu, s.key, mask);
    o.s_at = __shfl_xor_sync(0xffffffffu, s.s_at, mask);
    o.idx = __shfl_xor_sync(0xffffffffu, s.idx, mask);
    o.pad0 = o.pad1 = o.pad2 = 0;
    return o;
}

__device__ __forceinline__ RowState warp_merge(RowState s) {
#pragma unroll
    for (int mask = 16; mask > 0; mask >>= 1) {
        RowState o = shfl_xor_state(s, mask);
        row_state_merge(s, o);
    }
    return s;
}

// Online-softmax step with one value s (T > 0).
__device__ __forceinline__ void softmax_push(RowState &st, float s) {
    if (s > st.m) {
        st.S = st.S * expf(st.m - s) + 1.f;
        st.m = s;
    } else {
        st.S += expf(s - st.m);
    }
}

// Gumbel-max step: key = s + g(u) = s - ln(E), E = -ln u.
__device__ __forceinline__ void gumbel_push(RowState &st, float s, uint32_t word, int v) {
    const float key = s - logf(neg_log_uniform(word));
    if (key > st.key || (key == st.key && v < st.idx)) {
        st.key = key;
        st.s_at = s;
        st.idx = v;
    }
}

// Greedy step: key = value itself.
__device__ __forceinline__ void argmax_push(RowState &st, float z, int v) {
    if (z > st.key || (z == st.key && v < st.idx)) {
        st.key = z;
        st.s_at = z;
        st.idx = v;
    }
    st.m = fmaxf(st.m, z);
}

// Block-wide merge of one RowState per thread; the result is valid in thread 0.
// `scratch` holds blockDim.x / 32 states.
__device__ __forceinline__ RowState block_merge(RowState s, RowState *scratch) {
    s = warp_merge(s);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    __syncthreads();
    if (lane == 0) scratch[warp] = s;
    __syncthreads();
    if (warp == 0) {
        s = (lane < nwarps) ? scratch[lane] : row_state_init();
        s = warp_merge(s);
    }
    return s;
}

}  // namespace dspark

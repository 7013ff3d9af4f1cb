// Device helpers shared by the draft, verify and schedule kernels.
//
// Random stream: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random
// Numbers: As Easy as 1, 2, 3", SC'11) keyed by the 64-bit seed, counter =
// (v >> 2, position, request id, stream), word v & 3; the uniform keeps the
// top 23 bits of the word and centres it in its cell: u = (k + 1/2) 2^-23.
//
// Scores are kept in log2 units: s2 = z * log2(e) / T.  The online softmax
// holds (m, S) with S = sum 2^(s2 - m), so lse = ln 2 * (m + log2 S); the
// Gumbel-max key of token v is s2_v - log2(E_v) with E_v = -ln u_v, which
// orders tokens exactly as the natural-log key s_v - ln(E_v) = s_v + g_v.
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
constexpr uint32_t kFlagTimeout = 16u;
constexpr uint32_t kFlagBadTargetRow = 32u;

// Row j of request b's target logits: the dense layout [B][G+1][V], or the
// packed one (request b's rows 0, 1, .. from row row0[b] of n_rows rows).
// nullptr when a packed row falls outside the array.
template <typename T>
__device__ __forceinline__ const T *target_row(const T *target, const int64_t *row0, int64_t n_rows, int b, int G,
                                               int j, int V) {
    if (!row0) return target + ((size_t)b * (G + 1) + j) * (size_t)V;
    const int64_t r = row0[b] + j;
    return (row0[b] >= 0 && r < n_rows) ? target + (size_t)r * (size_t)V : nullptr;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

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

// Philox4x32-10 round keys: k0 + r W0, k1 + r W1 for r = 0..9.
struct PhiloxRoundKeys {
    uint32_t k0[10];
    uint32_t k1[10];
};

// Philox4x32-10 for counter (x0, pos, rid, stream) with the parts that do not
// depend on x0 precomputed per request and position (PhiloxRow).  After round 1
// the words are (y0c, y1c, hi(M0 x0) ^ sk, lo(M0 x0)) with
//   y0c = hi(M1 rid) ^ pos ^ k0[0],  y1c = lo(M1 rid),  sk = stream ^ k1[0];
// round 2 multiplies the constant y0c, so hi(M0 y0c) ^ k1[1] and lo(M0 y0c)
// are precomputed as well.  Same words as
// philox4x32_10(make_uint4(x0, pos, rid, stream), k0, k1).
struct PhiloxRow {
    uint32_t sk;   // stream ^ k1[0]
    uint32_t y1k;  // y1c ^ k0[1]
    uint32_t y2h;  // hi(M0 y0c) ^ k1[1]
    uint32_t y2l;  // lo(M0 y0c)
};
__device__ __forceinline__ PhiloxRow philox_row(uint32_t rid, uint32_t pos, uint32_t stream, const PhiloxRoundKeys &K) {
    const uint32_t y0c = __umulhi(kPhiloxM1, rid) ^ pos ^ K.k0[0];
    const uint32_t y1c = kPhiloxM1 * rid;
    const uint64_t p2 = (uint64_t)kPhiloxM0 * y0c;
    PhiloxRow R;
    R.sk = stream ^ K.k1[0];
    R.y1k = y1c ^ K.k0[1];
    R.y2h = (uint32_t)(p2 >> 32) ^ K.k1[1];
    R.y2l = (uint32_t)p2;
    return R;
}
__device__ __forceinline__ uint4 philox_folded(uint32_t x0, const PhiloxRow &R, const PhiloxRoundKeys &K) {
    // round 1
    const uint64_t p1 = (uint64_t)kPhiloxM0 * x0;
    const uint32_t c2r1 = (uint32_t)(p1 >> 32) ^ R.sk, c3r1 = (uint32_t)p1;
    // round 2: only the M1 product depends on x0
    const uint64_t pb2 = (uint64_t)kPhiloxM1 * c2r1;
    uint32_t c0 = (uint32_t)(pb2 >> 32) ^ R.y1k, c1 = (uint32_t)pb2, c2 = R.y2h ^ c3r1, c3 = R.y2l;
#pragma unroll
    for (int r = 2; r < 10; ++r) {
        const uint64_t pa = (uint64_t)kPhiloxM0 * c0;
        const uint64_t pb = (uint64_t)kPhiloxM1 * c2;
        const uint32_t n0 = (uint32_t)(pb >> 32) ^ c1 ^ K.k0[r];
        const uint32_t n2 = (uint32_t)(pa >> 32) ^ c3 ^ K.k1[r];
        c1 = (uint32_t)pb;
        c3 = (uint32_t)pa;
        c0 = n0;
        c2 = n2;
    }
    return make_uint4(c0, c1, c2, c3);
}

// u = ((w >> 9) + 1/2) * 2^-23, exact: 1 + k 2^-23 minus (1 - 2^-24).
__device__ __forceinline__ float word_to_uniform(uint32_t w) {
    return __uint_as_float(0x3F800000u | (w >> 9)) - 0x1.fffffep-1f;
}

// f1 = 1 + k' 2^-23 with k' = 0x7FFFFF - (w >> 9), which equals
// (1 - u) + 1 - 2^-24 exactly.  The test f1 < fl(t + 1) is a conservative form
// of (1 - u) < t: fl(t + 1) >= t + 1 - 2^-24 whenever t < 1 (round to
// nearest), and for t >= 1 both sides pass, so no true "yes" is lost.
__device__ __forceinline__ float one_minus_uniform_plus_one(uint32_t w) {
    return __uint_as_float(0x3F800000u | ((~w) >> 9));
}

// Exponential variate E = -ln u (relative accuracy matters: small E wins).
__device__ __forceinline__ float neg_log_uniform(uint32_t w) {
    return -logf(word_to_uniform(w));
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float fast_log2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

// Four consecutive elements starting at a 4-aligned index.
__device__ __forceinline__ float4 load4(const float *p) {
    return __ldg(reinterpret_cast<const float4 *>(p));
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16 *p) {
    const uint2 raw = __ldg(reinterpret_cast<const uint2 *>(p));
    return make_float4(bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y));
}
__device__ __forceinline__ float elem(const float4 &f, int e) {
    return e == 0 ? f.x : (e == 1 ? f.y : (e == 2 ? f.z : f.w));
}

// Running state of one row segment: online softmax (m, S) and the best key.
// T > 0: m = max s2, S = sum 2^(s2 - m), key = best s2 - log2(E), s_at = s2
// at the best token.  T = 0: key = m = max z, s_at = z at the best token.
struct RowState {
    float m;
    float S;
    float key;
    float s_at;
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
        const float sa = (a.m == -INFINITY) ? 0.f : a.S * exp2f(a.m - m);
        const float sb = (b.m == -INFINITY) ? 0.f : b.S * exp2f(b.m - m);
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

// Online-softmax step with a group of n scores (log2 units), n <= 16.
template <int N>
__device__ __forceinline__ void softmax_push_group(RowState &st, const float (&s2)[N], int n) {
    float cm = -INFINITY;
#pragma unroll
    for (int i = 0; i < N; ++i)
        if (i < n) cm = fmaxf(cm, s2[i]);
    if (cm > st.m) {
        st.S = (st.m == -INFINITY) ? 0.f : st.S * fast_exp2(st.m - cm);
        st.m = cm;
    }
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < N; ++i)
        if (i < n) acc += fast_exp2(s2[i] - st.m);
    st.S += acc;
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

// Float keys as unsigned integers whose order is the float order, so that a
// row-wide running best can be kept with atomicMax.  0 encodes "none" (-inf).
__device__ __forceinline__ uint32_t key_to_ordered(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float ordered_to_key(uint32_t o) {
    if (o == 0u) return -INFINITY;
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}
__device__ __forceinline__ uint32_t load_relaxed(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// Programmatic dependent launch: let the next kernel of the stream start its
// independent prologue (launch_dependents), and wait until every earlier
// kernel of the stream has completed with its writes visible (wait).  Both
// are no-ops when the launch carries no programmatic serialization attribute.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Row-wide best draw of a block position as one 64-bit word: the key's
// order-preserving encoding above the complemented token id, so that
// atomicMax keeps the largest key and, on an exact tie, the lowest id (the
// merge rule of the partial states).  0 means "none".
__device__ __forceinline__ unsigned long long best_encode(float key, int idx) {
    return ((unsigned long long)key_to_ordered(key) << 32) | (unsigned long long)(~(uint32_t)idx);
}
__device__ __forceinline__ int best_token(unsigned long long w) { return w ? (int)~(uint32_t)w : -1; }
__device__ __forceinline__ unsigned int load_acquire_u32(const unsigned int *p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Bounded wait until a global counter reaches `target` (the waiting half of a
// grid barrier): gives up after about `limit` clock cycles or when *abort is
// raised.  Returns whether the counter got there.
__device__ __forceinline__ bool counter_wait(const unsigned int *ctr, unsigned int target, volatile int *abort,
                                             long long limit) {
    const long long t0 = clock64();
    while (load_acquire_u32(ctr) < target) {
        if (*abort) return false;
        if (clock64() - t0 > limit) return false;
        __nanosleep(64);
    }
    return true;
}

// Fire-and-forget maxima (no value returned, so the issuing warp does not
// wait for the memory system).
__device__ __forceinline__ void red_max_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void red_max_shared_u32(uint32_t *p, uint32_t v) {
    asm volatile("red.shared.max.u32 [%0], %1;" ::"r"((uint32_t)__cvta_generic_to_shared(p)), "r"(v) : "memory");
}
__device__ __forceinline__ void red_max_u32(uint32_t *p, uint32_t v) {
    asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned long long load_relaxed_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Final draw state (residual or bonus): the best group key and its token.
// A residual row whose entries all have p <= q (impossible in exact
// arithmetic after a rejection) keeps key -inf here and is redrawn from p by
// the merge step.
struct ResidualState {
    float key_res;
    int idx_res;
};

__device__ __forceinline__ ResidualState residual_init() { return ResidualState{-INFINITY, INT32_MAX}; }

__device__ __forceinline__ void residual_merge(ResidualState &a, const ResidualState &b) {
    if (key_better(b.key_res, b.idx_res, a.key_res, a.idx_res)) {
        a.key_res = b.key_res;
        a.idx_res = b.idx_res;
    }
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

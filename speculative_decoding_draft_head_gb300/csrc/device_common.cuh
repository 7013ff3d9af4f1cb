// Device helpers shared by the draft, verify and schedule kernels.
//
// Random stream: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random
// Numbers: As Easy as 1, 2, 3", SC'11) keyed by the 64-bit seed, counter =
// (v >> 2, position, request id, stream), word v & 3; the uniform keeps the
// top 23 bits of the word and centres it in its cell: u = (k + 1/2) 2^-23.
//
// Scores are kept in log2 units: s2 = z * log2(e) / T.  The online softmax
// holds (m, S) with S = sum 2^(s2 - m) and an integer reference m, so that
// rescaling a partial sum is an exact power-of-two scaling and lse =
// ln 2 * (m + log2 S).  The Gumbel-max key of token v is s_v + g(u_v) with
// s_v = z_v / T and g(u) = -ln(-ln u).  Tokens are screened in fp32 (log2
// units, no logarithm for almost all of them); the few that can still win get
// their key in float-float arithmetic (about 44 significant bits), so the
// winner agrees with an fp64 evaluation of the same keys except on ties far
// below fp32 rounding.
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

// c2 = log2(e) / T as float-float (hi, lo).  A logit's exponent z c2 - m is
// formed as fmaf(z, lo, fmaf(z, hi, -m)): rounding c2 to fp32 alone would
// shift every exponent by about 6e-8 |z c2| (3e-6 nats at |z / T| = 50).
__device__ __forceinline__ float2 c2_split(float T) {
    constexpr float kLog2eHi = 1.44269502162933349609375f;  // fp32(log2 e)
    constexpr float kLog2eLo = 1.925963e-08f;               // log2 e - kLog2eHi
    const float hi = __fdiv_rn(kLog2eHi, T);
    const float rem = fmaf(-hi, T, kLog2eHi);               // exact
    return make_float2(hi, __fdiv_rn(rem + kLog2eLo, T));
}
// 2^(z c2 - m) with c2 = (c2h, c2l) from c2_split.
__device__ __forceinline__ float term_exp2(float z, float c2h, float c2l, float m);

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
// The high and low words of a 32 x 32 -> 64-bit product as two separate
// multiplies (measured on GB300: Philox runs about 8 % faster this way than
// with one widening multiply).
__device__ __forceinline__ void mul_hilo(uint32_t a, uint32_t M, uint32_t &hi, uint32_t &lo) {
    asm("mul.hi.u32 %0, %1, %2;" : "=r"(hi) : "r"(a), "r"(M));
    asm("mul.lo.u32 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(M));
}
// Rounds 2-10 of the folded form from the round-1 product p1 = M0 x0.
__device__ __forceinline__ uint4 philox_folded_p(uint64_t p1, const PhiloxRow &R, const PhiloxRoundKeys &K) {
    // round 1
    const uint32_t c2r1 = (uint32_t)(p1 >> 32) ^ R.sk, c3r1 = (uint32_t)p1;
    // round 2: only the M1 product depends on x0
    uint32_t h2, l2;
    mul_hilo(c2r1, kPhiloxM1, h2, l2);
    uint32_t c0 = h2 ^ R.y1k, c1 = l2, c2 = R.y2h ^ c3r1, c3 = R.y2l;
#pragma unroll
    for (int r = 2; r < 10; ++r) {
        uint32_t ha, la, hb, lb;
        mul_hilo(c0, kPhiloxM0, ha, la);
        mul_hilo(c2, kPhiloxM1, hb, lb);
        const uint32_t n0 = hb ^ c1 ^ K.k0[r];
        const uint32_t n2 = ha ^ c3 ^ K.k1[r];
        c1 = lb;
        c3 = la;
        c0 = n0;
        c2 = n2;
    }
    return make_uint4(c0, c1, c2, c3);
}
__device__ __forceinline__ uint4 philox_folded(uint32_t x0, const PhiloxRow &R, const PhiloxRoundKeys &K) {
    return philox_folded_p((uint64_t)kPhiloxM0 * x0, R, K);
}
// Four consecutive blocks x0 .. x0 + 3: their round-1 products differ by M0,
// so one multiply and three 64-bit additions give all four.
__device__ __forceinline__ void philox_folded4(uint32_t x0, const PhiloxRow &R, const PhiloxRoundKeys &K,
                                               uint4 (&w)[4]) {
    const uint64_t p = (uint64_t)kPhiloxM0 * x0;
#pragma unroll
    for (int g = 0; g < 4; ++g) w[g] = philox_folded_p(p + (uint64_t)g * kPhiloxM0, R, K);
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

// log2(E), E = -ln u, for screening (relative error of E below 7e-6, so
// log2 E within 1e-5 plus the lg2 approximation's 2^-22.6): with
// e1 = 1 - u (exact), E = e1 (1 + e1 / 2 + e1^2 / 3) for e1 < 2^-6 (the series
// of -ln(1 - e1), truncation below 1e-6 relative), else -lg2(u) ln 2.
__device__ __forceinline__ float log2_neg_log_uniform_fast(uint32_t w) {
    const float f1 = __uint_as_float(0x3F800000u | ((~w) >> 9));  // (1 - u) + 1 - 2^-24
    const float e1 = (f1 - 1.f) + 0x1p-24f;                        // 1 - u, exact
    float E;
    if (e1 < 0x1p-6f) {
        E = e1 * fmaf(e1, fmaf(e1, 0.33333334f, 0.5f), 1.f);
    } else {
        float l;
        asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(l) : "f"(1.f - e1));
        E = -l * 0.6931471805599453f;
    }
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(E));
    return y;
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

// ------------------------------------------------------------ keys ----
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

// A float-float number hi + lo with |lo| <= ulp(hi) / 2.
struct FF {
    float hi, lo;
};

// a + b exactly (Knuth's two-sum).
__device__ __forceinline__ FF two_sum(float a, float b) {
    const float s = a + b;
    const float bv = s - a;
    const float av = s - bv;
    return FF{s, (a - av) + (b - bv)};
}
// a + b exactly when |a| >= |b| (or a == 0): the normalising step.
__device__ __forceinline__ FF quick_two_sum(float a, float b) {
    const float s = a + b;
    return FF{s, b - (s - a)};
}
__device__ __forceinline__ FF ff_add(FF a, FF b) {
    const FF s = two_sum(a.hi, b.hi);
    return quick_two_sum(s.hi, s.lo + (a.lo + b.lo));
}
__device__ __forceinline__ FF ff_neg(FF a) { return FF{-a.hi, -a.lo}; }

// Natural logarithm of a positive normal float as float-float, from
// ln x = e ln 2 + ln m with m in [sqrt(1/2), sqrt(2)) and
// ln m = 2 atanh(t), t = (m - 1) / (m + 1), |t| <= 0.1716:
// 2 atanh(t) = 2t + t^3 (2/3 + 2/5 t^2 + 2/7 t^4 + ...) (the Taylor series of
// atanh).  t is formed in float-float; the series tail (below 0.0034) in fp32.
// Absolute error about 1e-10 for the arguments used here.
__device__ __forceinline__ FF ln_ff(float x) {
    const uint32_t ix = __float_as_uint(x);
    int e = (int)((ix >> 23) & 0xFFu) - 127;
    uint32_t mb = (ix & 0x7FFFFFu) | 0x3F800000u;  // m in [1, 2)
    if (mb > 0x3FB504F3u) {                         // m > sqrt(2): halve it
        mb -= 0x00800000u;
        e += 1;
    }
    const float m = __uint_as_float(mb);
    const float f = m - 1.f;             // exact (Sterbenz)
    const FF d = two_sum(m, 1.f);        // m + 1
    const float rd = __frcp_rn(d.hi);
    const float t_hi = f * rd;
    float rem = fmaf(-t_hi, d.hi, f);    // f - t_hi (d.hi + d.lo)
    rem = fmaf(-t_hi, d.lo, rem);
    const float t_lo = rem * rd;
    const float t2 = t_hi * t_hi;
    float P = 2.f / 13.f;
    P = fmaf(P, t2, 2.f / 11.f);
    P = fmaf(P, t2, 2.f / 9.f);
    P = fmaf(P, t2, 2.f / 7.f);
    P = fmaf(P, t2, 2.f / 5.f);
    P = fmaf(P, t2, 2.f / 3.f);
    const float tail = t_hi * t2 * P;
    // ln 2 split so that e * kLn2Hi is exact for |e| < 256
    constexpr float kLn2Hi = 0.693145751953125f;        // 0x3F317200
    constexpr float kLn2Lo = 1.4286068203094172e-06f;   // ln 2 - kLn2Hi
    const float fe = (float)e;
    const FF a = two_sum(fe * kLn2Hi, 2.f * t_hi);
    return quick_two_sum(a.hi, a.lo + fmaf(fe, kLn2Lo, fmaf(2.f, t_lo, tail)));
}

// s = z / T as float-float (rT = fl(1 / T); the residual z - s_hi T is exact).
__device__ __forceinline__ FF div_ff(float z, float T, float rT) {
    const float hi = z * rT;
    const float lo = fmaf(-hi, T, z) * rT;
    return quick_two_sum(hi, lo);
}

// g(u) = -ln(-ln u) for the uniform of word w, as float-float.
__device__ __forceinline__ FF gumbel_ff(uint32_t w) {
    const FF l = ln_ff(word_to_uniform(w));         // ln u < 0, u exact in fp32
    const FF L = ln_ff(-l.hi);                       // ln E, E = -ln u = -(l.hi + l.lo)
    // ln(E_hi + E_lo) = ln E_hi + E_lo / E_hi (|E_lo / E_hi| <= 2^-24)
    const float corr = -l.lo * __frcp_rn(-l.hi);
    return quick_two_sum(-L.hi, -(L.lo + corr));
}

// The row-wide best draw as one 64-bit word whose unsigned order is the order
// of the keys, the lowest token id winning an exact tie: the key's high part
// in the order-preserving encoding (32 bits), its low part as a signed
// fraction of ulp(hi) in 12 bits, and the complemented token id in 20 bits
// (vocabularies up to 2^20).  0 means "none".
constexpr int kTokenBits = 20;
constexpr uint32_t kTokenMask = (1u << kTokenBits) - 1u;
__device__ __forceinline__ unsigned long long key_word(FF k, int idx) {
    const uint32_t oh = key_to_ordered(k.hi);
    uint32_t q = 2048u;
    const uint32_t e = (__float_as_uint(k.hi) >> 23) & 0xFFu;
    if (e >= 35u && e < 255u) {
        // lo / ulp(hi) * 4096 = lo * 2^(162 - e), in [-2048, 2048]
        const int qi = __float2int_rn(k.lo * __uint_as_float((289u - e) << 23));
        q = (uint32_t)(min(2047, max(-2047, qi)) + 2048);
    }
    return ((unsigned long long)oh << 32) | ((unsigned long long)q << kTokenBits) |
           (unsigned long long)(~(uint32_t)idx & kTokenMask);
}

// The exact key word of a final-draw contender: token tok with target logit
// tb, draft logit zb and word wb; 0 when a residual row gives it no mass
// (p <= q).  key_hi receives the float-float key's high part.  Out of line:
// it runs for a few tokens per row; inlined at every call site it would
// spill registers (tensor-core kernel) or bloat the code (SIMT kernel).
static __device__ __noinline__ unsigned long long final_key_word(float tb, float zb, uint32_t wb, int tok, bool bonus,
                                                          float T, float rT, FF lse_t, float lse_q,
                                                          float *key_hi) {
    FF key;
    if (bonus) {
        key = div_ff(tb, T, rT);  // t / T: the bonus key before its noise
    } else {
        // ln r = ln p + ln(1 - q / p), ln q - ln p formed in float-float from
        // the logits and the two lse
        const FF lp = ff_add(div_ff(tb, T, rT), ff_neg(lse_t));
        const FF dl = ff_add(ff_add(div_ff(zb, T, rT), FF{-lse_q, 0.f}), ff_neg(lp));
        const float d = dl.hi + dl.lo;
        if (!(d < 0.f)) return 0ull;  // p <= q: no residual mass
        const float l1m = (d > -0.6931472f) ? logf(-expm1f(d)) : log1pf(-expf(d));
        key = ff_add(lp, FF{l1m, 0.f});
    }
    key = ff_add(key, gumbel_ff(wb));
    *key_hi = key.hi;
    return key_word(key, tok);
}

__device__ __forceinline__ int word_token(unsigned long long w) {
    return w ? (int)(~(uint32_t)w & kTokenMask) : -1;
}
// The key's high part (natural-log units) of a word, -inf for "none".
__device__ __forceinline__ float word_key_hi(unsigned long long w) { return ordered_to_key((uint32_t)(w >> 32)); }

// The screening factor Q = 2^(m - K log2 e) (capped at 2^126) times a margin
// that covers the fp32 rounding of the exponents (relative 4e-7 of their
// size); K = -inf (no key yet) lets every token with mass through.
__device__ __forceinline__ float screen_q(float m, float kbest) {
    if (kbest == -INFINITY) return INFINITY;
    const float K2 = kbest * kLog2e;
    return fminf(fast_exp2(m - K2), 0x1p126f) * (1.f + 4e-7f * (fabsf(K2) + fabsf(m) + 64.f));
}

// Tolerance of an fp32 key (log2 units) against the threshold K2: the
// rounding of z c2, of c2 itself, of -ln u and lg2, and of K2.
__device__ __forceinline__ float key_tol2(float k2, float K2) {
    return 4e-7f * (fabsf(k2) + fabsf(K2)) + 2e-6f;
}

// 2^k for an integer-valued float k (exact power of two; 0 below 2^-149).
__device__ __forceinline__ float scale_pow2(float S, float k) {
    return (k < -300.f) ? 0.f : ldexpf(S, (int)k);
}

// Running state of one row segment: online softmax (m, S) and the best draw.
// T > 0: m an integer reference (log2 units), S = sum 2^(s2 - m), best the
// best key word, z_at the logit z of that token.  T = 0: m = max z, best the
// word of (max z, lowest id), z_at = max z.
struct RowState {
    float m;
    float S;
    unsigned long long best;
    float z_at;
    int pad0, pad1, pad2;
};
static_assert(sizeof(RowState) == 32, "RowState is stored as two 16-byte words");

__device__ __forceinline__ RowState row_state_init() {
    RowState st;
    st.m = -INFINITY;
    st.S = 0.f;
    st.best = 0ull;
    st.z_at = 0.f;
    st.pad0 = st.pad1 = st.pad2 = 0;
    return st;
}

// Merge b into a (associative; the larger word wins).
__device__ __forceinline__ void row_state_merge(RowState &a, const RowState &b) {
    const float m = fmaxf(a.m, b.m);
    if (m != -INFINITY) {
        const float sa = (a.m == -INFINITY) ? 0.f : scale_pow2(a.S, a.m - m);
        const float sb = (b.m == -INFINITY) ? 0.f : scale_pow2(b.S, b.m - m);
        a.S = sa + sb;
        a.m = m;
    }
    if (b.best > a.best) {
        a.best = b.best;
        a.z_at = b.z_at;
    }
}

__device__ __forceinline__ RowState shfl_xor_state(const RowState &s, int mask) {
    RowState o;
    o.m = __shfl_xor_sync(0xffffffffu, s.m, mask);
    o.S = __shfl_xor_sync(0xffffffffu, s.S, mask);
    o.best = __shfl_xor_sync(0xffffffffu, s.best, mask);
    o.z_at = __shfl_xor_sync(0xffffffffu, s.z_at, mask);
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

// ln x of a positive float-float x = hi + lo: ln hi + lo / hi (the next
// term, (lo / hi)^2 / 2, is below 2^-49).
__device__ __forceinline__ FF ln_of_ff(FF x) {
    const FF l = ln_ff(x.hi);
    return quick_two_sum(l.hi, l.lo + x.lo * __frcp_rn(x.hi));
}
// m ln 2 as float-float for an integer-valued float m: the fp32 product, its
// exact rounding error, and m times the part of ln 2 that fp32 drops.
__device__ __forceinline__ FF mul_ln2_ff(float m) {
    constexpr float kLn2Tail = -1.9046542999577683e-09f;  // ln 2 - fl(ln 2)
    const float p = m * kLn2;
    return quick_two_sum(p, fmaf(m, kLn2Tail, fmaf(m, kLn2, -p)));
}
// Sum of partial sums S_i 2^(m_i - m) (m the largest reference): each term is
// an exact power-of-two rescaling, added in float-float.
__device__ __forceinline__ FF add_scaled_partial(FF S, const RowState &p, float m) {
    if (p.m != -INFINITY && p.S > 0.f) S = ff_add(S, FF{scale_pow2(p.S, p.m - m), 0.f});
    return S;
}

// The natural-log log-sum-exp of the partial states (m_i, S_i) of one row, as
// float-float (about 44 bits): m ln 2 + ln sum_i S_i 2^(m_i - m), the partial
// sums rescaled exactly by their integer references.  Every lane of the warp
// calls it; lane i reads partials i, i + 32, ...  Returns -inf for an empty
// row.
__device__ __forceinline__ FF warp_lse_of_partials(const RowState *part, int n) {
    float m = -INFINITY;
    for (int i = threadIdx.x & 31; i < n; i += 32) m = fmaxf(m, part[i].m);
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, k));
    if (m == -INFINITY) return FF{-INFINITY, 0.f};
    FF S{0.f, 0.f};
    for (int i = threadIdx.x & 31; i < n; i += 32) S = add_scaled_partial(S, part[i], m);
#pragma unroll
    for (int k = 16; k > 0; k >>= 1)
        S = ff_add(S, FF{__shfl_xor_sync(0xffffffffu, S.hi, k), __shfl_xor_sync(0xffffffffu, S.lo, k)});
    return ff_add(mul_ln2_ff(m), ln_of_ff(S));
}
// The same for one thread reading all n partials in order.
__device__ __forceinline__ FF lse_of_partials(const RowState *part, int n) {
    float m = -INFINITY;
    for (int i = 0; i < n; ++i) m = fmaxf(m, part[i].m);
    if (m == -INFINITY) return FF{-INFINITY, 0.f};
    FF S{0.f, 0.f};
    for (int i = 0; i < n; ++i) S = add_scaled_partial(S, part[i], m);
    return ff_add(mul_ln2_ff(m), ln_of_ff(S));
}

__device__ __forceinline__ float term_exp2(float z, float c2h, float c2l, float m) {
    return fast_exp2(fmaf(z, c2l, fmaf(z, c2h, -m)));
}

// Online-softmax step with the logits z[0..N) of one row (c2 = (c2h, c2l)),
// against an integer reference m (log2 units) that may lag the maximum
// (terms above 1 are fine; a group whose sum leaves [0, 2^64] is redone
// against its own maximum, an exact power-of-two rescaling).  e[i] receives
// the terms 2^(z c2 - m) against the final m.
template <int N>
__device__ __forceinline__ void softmax_push_group(RowState &st, const float (&z)[N], float c2h, float c2l,
                                                   float (&e)[N]) {
    if (st.m == -INFINITY) {
        float zm = -INFINITY;
#pragma unroll
        for (int i = 0; i < N; ++i) zm = fmaxf(zm, z[i]);
        if (zm == -INFINITY) return;
        st.m = ceilf(zm * c2h);  // c2 > 0: the rounded product is monotone in z
    }
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        e[i] = term_exp2(z[i], c2h, c2l, st.m);
        acc += e[i];
    }
    if (!(acc <= 0x1p64f)) {
        float zm = -INFINITY;
#pragma unroll
        for (int i = 0; i < N; ++i) zm = fmaxf(zm, z[i]);
        const float nm = ceilf(fmaxf(st.m, zm * c2h));
        st.S = scale_pow2(st.S, st.m - nm);
        st.m = nm;
        acc = 0.f;
#pragma unroll
        for (int i = 0; i < N; ++i) {
            e[i] = term_exp2(z[i], c2h, c2l, st.m);
            acc += e[i];
        }
    }
    st.S += acc;
}

// Greedy step: the key is the logit itself (lowest id on exact ties).
__device__ __forceinline__ void argmax_push(RowState &st, float z, int v) {
    const unsigned long long w = key_word(FF{z, 0.f}, v);
    if (w > st.best) {
        st.best = w;
        st.z_at = z;
    }
    st.m = fmaxf(st.m, z);
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

// Final draw state (residual or bonus): the best key word (key_word) of a
// row segment, 0 = none.  A residual row whose entries all have p <= q
// (impossible in exact arithmetic after a rejection) keeps 0 here and is
// redrawn from p by the merge step.
struct ResidualState {
    unsigned long long best;
};

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

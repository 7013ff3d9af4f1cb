// Markov-head logits on the tcgen05 tensor cores, fused with sampling.
//
// Method: "DSpark, la bozza che sa quando fermarsi" (paithon.it), section
// "Un po' di autoregressione basta": position j draws from
// softmax((U_j + E_in[x_{j-1}] W_out^T) / T), a rank-r bias driven by the
// previous token.  The bias is a dense contraction (128 requests x 64 tokens x
// r per tile), so it runs on the tensor cores; everything after it -- base
// logits, temperature, online softmax, Philox Gumbel-max -- is fused into the
// TMEM epilogue so that each logit is produced and consumed on chip.
//
// Two uses share the kernel:
//  - draft: rows = 128 requests (a batch of at most 64 is replicated twice
//    over the 128 rows, each replica taking half of every tile's columns);
//    base-logit tiles come by TMA; one cooperative launch walks all block
//    positions, meeting the other CTAs of its row block at a bounded grid
//    barrier between positions, where each row's best (key, token) word gives
//    x_j for the next position's A operand.  Per-(request, segment) softmax
//    partials go to the workspace for draft_finalize (lse, log q);
//  - final draw of verification ("Les mathematiques derriere l'acceleration",
//    section "La garantie de l'echantillonnage par rejet", and "DeepSeek发布
//    DSpark", section "DSpark 是什么？"): each row is a request that either
//    rejected at position d (draw from max(0, p_d - q_d), q rebuilt from base
//    logits + Markov bias) or accepted its whole block (bonus draw from p_L);
//    other rows idle.  Target rows stream by cp.async into per-thread slots
//    three sub-slices ahead; base values are read only for lanes with a token
//    that passes the per-token test against p.
//
// CTA layout (one CTA per SM, 480 threads, ~200 KB shared memory):
//   warps 0-11  epilogue: warp w reads TMEM lanes 32*(w%4).. (its quadrant of
//               rows); the 8 sixteen-column sub-slices of each 128-column
//               tile are dealt round-robin to the quadrant's three warps;
//   warp 12     TMA producer: W_out chunks (128 tokens x 64 of r, 128-byte
//               swizzle, L2 evict-last) and base-logit tiles (two boxes of
//               128 requests x 64 tokens, evict-first);
//   warps 13-14 UMMA issuers for even / odd tiles (M=128, N=128, K=16 steps);
//               warp 13 also allocates TMEM.
// The A operand (the 128 gathered E_in rows, 128 x r bf16) is written once per
// position into TMEM (columns 384..) and read from there by the bias UMMAs,
// which leaves shared memory to the streams.  Rings: 8 W chunks (two tiles),
// 2 base tiles (tile slots), 3 TMEM accumulators of 128 columns.  Tiles are as
// wide as a single UMMA allows at this shape because every tcgen05.mma costs a
// roughly fixed issue time whatever its N: wide tiles cut the instructions per
// token.  In the draft the base-logit tile joins the contraction: after the
// r/16 bias steps, eight N=16 UMMAs multiply 16-token slices of the tile (128
// requests x 128 tokens, already in the K-major A layout as TMA writes it) by
// a 16 x 16 identity into the matching accumulator columns, so TMEM holds
// z = U + bias and the epilogue reads nothing from shared memory.  (U * 1 and
// U * 0 are exact; base logits must be finite, since inf * 0 would poison the
// other columns of its 16-wide step.)  Every wait is bounded; a timeout sets
// the timeout bit of the flag word and the CTA unwinds.
//
// Per-token Gumbel-max without a logarithm per token: token v can beat a key K
// only if E_v < 2^(s2_v - K) = e_v * 2^(m - K), where e_v = 2^(s2_v - m) is the
// softmax term already computed and E_v = -ln u_v >= 1 - u_v.  So the test
// (1 - u_v) < e_v * Q with Q = 2^(m - K) (with a rounding margin) rejects
// almost every token; only the survivors evaluate -ln u_v and a key.
#include <climits>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "device_common.cuh"
#include "internal.h"
#include "tc_primitives.cuh"

namespace dspark {
namespace {

using namespace tc;

constexpr int BM = 128;
constexpr int BN = 128;                  // tokens per tile: the UMMA N
#ifndef DSPARK_EPI_WARPS
#define DSPARK_EPI_WARPS 12
#endif
constexpr int kEpiWarps = DSPARK_EPI_WARPS;  // a multiple of 4: one group per TMEM lane quadrant
constexpr int kEpiPerQuad = kEpiWarps / 4;   // warps sharing a quadrant's 16-column sub-slices
constexpr int kProducerWarp = kEpiWarps;
constexpr int kMmaWarp = kEpiWarps + 1;      // and kMmaWarp + 1: even / odd tiles
constexpr int kThreads = (kEpiWarps + 3) * 32;
// registers per thread such that the warps of the busiest SM sub-partition fit its 16K
constexpr int kMaxRegs = (16384 / (32 * ((kEpiWarps + 3 + 3) / 4))) / 8 * 8 > 168
                             ? 168
                             : (16384 / (32 * ((kEpiWarps + 3 + 3) / 4))) / 8 * 8;
static_assert(kEpiWarps % 4 == 0 && kEpiPerQuad <= 8, "epilogue warps");
#ifndef DSPARK_W_STAGES
#define DSPARK_W_STAGES 8
#endif
#ifndef DSPARK_U_STAGES
#define DSPARK_U_STAGES 2
#endif
constexpr int kWStages = DSPARK_W_STAGES;  // W ring: one 64-wide K atom of one tile per stage
constexpr int kUStages = DSPARK_U_STAGES;  // tile slots: tile t fills slot t % kUStages
constexpr int kAccBufs = 3;
constexpr uint32_t kTmemCols = 512;      // 3 x 128 accumulator columns + A, power-of-two allocation
constexpr uint32_t kTmemA = kAccBufs * BN;  // A operand: columns 384.. (r/2 columns, <= 128)
constexpr uint32_t kWChunk = BN * 128;   // 128 tokens x 64 of r: 16 KB
constexpr uint32_t kUHalf = BM * 128;    // 128 requests x 64 tokens: 16 KB (one TMA box)
constexpr uint32_t kUBytes = 2 * kUHalf;
constexpr uint32_t kOffW = 0;
constexpr uint32_t kOffU = kOffW + kWStages * kWChunk;
// 16 x 16 bf16 identity in the B-operand layout: eight N = 16 UMMAs per tile
// add the base-logit tile (as an A operand) onto the bias accumulator
constexpr uint32_t kOffI = kOffU + kUStages * kUBytes;
// The final draw's target values: each epilogue thread owns kTargetAhead
// slots of 32 bytes (16 bf16) in the base-logit ring, which the final draw
// does not use; the low and high 16-byte halves lie in two arrays, so a warp's
// reads of one half are contiguous.
constexpr int kTargetAhead = 4;
constexpr uint32_t kTargetHalf = kTargetAhead * kEpiWarps * 32 * 16;
static_assert(2 * kTargetHalf <= kUStages * kUBytes, "target slots fit in the base-logit ring");
__device__ __forceinline__ uint32_t target_slot(uint32_t sbase, int k, int tid) {
    return sbase + kOffU + (uint32_t)(((k % kTargetAhead) * (kEpiWarps * 32) + tid) * 16);
}
constexpr uint32_t kIBytes = 16 * 128;
// per-row merge of the four column slices (the W ring keeps streaming the
// next block position meanwhile)
constexpr uint32_t kOffMerge = kOffI + kIBytes;
constexpr uint32_t kMergeBytes = BM * kEpiPerQuad * 32;
constexpr uint32_t kOffBar = kOffMerge + kMergeBytes;
constexpr int kNumBars = kWStages + 2 * kUStages + 2 * kAccBufs + 1 + 2;
static_assert(kNumBars * 8 <= 256, "barrier region");
constexpr uint32_t kOffMisc = kOffBar + 256;
constexpr uint32_t kMiscBytes = 16 + BM * 28;
constexpr uint32_t kSmemBytes = kOffMisc + kMiscBytes + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(kTmemA + 128 <= kTmemCols, "TMEM accumulators and A operand");

constexpr long long kSpinLimit = 4000000000LL;  // ~2 s of clock cycles
constexpr long long kDrainLimit = 200000000LL;  // ~0.1 s: copies and UMMAs in flight after a timeout
constexpr float kQMax = 0x1p126f;

struct TcParams {
    const __nv_bfloat16 *e_in;
    const __nv_bfloat16 *a_rows;  // draft, one position: A row of request b at a_rows + b r (else E_in[x_{j-1}])
    const __nv_bfloat16 *base;
    const __nv_bfloat16 *target;
    const int64_t *target_row0;  // final draw: packed target rows (nullptr: dense)
    int64_t n_target_rows;
    const int32_t *anchor;
    const int32_t *tokens;
    const float *temperature;
    const uint32_t *request_id;
    const int32_t *final_code;  // [B]: -1, or (kind << 16) | position
    const float2 *lse_t_row;    // [B] target lse of the rejected row, natural log, float-float
    const float *draft_lse;     // [B][G] natural log
    int B, G, V, r;
    int j, j_end;               // draft: block positions j .. j_end - 1 in this launch
    int nseg;
    int rep;                    // row replication for small batches: TMEM row i holds request m0 + i % (128 / rep)
    int pass;                   // final draw: odd passes walk the segment backwards
    PhiloxRoundKeys keys;
    RowState *part;             // draft: [G][B][nseg] softmax / key partials
    unsigned long long *best;   // draft: [G][B] row-wide best (key, token) words, see key_word
    unsigned int *grid_bar;     // draft, several positions: [row blocks] arrival counters of the barrier
    ResidualState *rpart;
    uint32_t *res_best;         // final draw: [B] row-wide best residual key (ordered encoding)
    uint32_t *flags;
    float *z_out;
};


// Grid-wide barrier between block positions (one thread per CTA; the launch
// is cooperative, so every CTA is resident).  Bounded: gives up after about
// `limit` cycles or when this CTA has aborted.
__device__ __forceinline__ bool grid_sync(unsigned int *ctr, unsigned int target, volatile int *abort,
                                          long long limit) {
    __threadfence();
    atomicAdd(ctr, 1u);
    if (!counter_wait(ctr, target, abort, limit)) return false;
    __threadfence();
    return true;
}

// Named barrier `id` over `nthreads` threads that also returns the OR of every
// participant's `pred`, so all of them take the same decision (a flag another
// warp may raise at any time, read once per thread, could otherwise differ).
__device__ __forceinline__ bool named_barrier_or(int id, int nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ int seg_begin(int s, int nseg, int V) {
    if (s >= nseg) return V;
    return (int)(((long long)s * V / nseg) & ~15LL);  // whole 16-token sub-slices
}

__device__ __forceinline__ bool uniform_wait(uint32_t bar, uint32_t parity, volatile int *abort) {
    bool ok = mbar_wait(bar, parity, abort, kSpinLimit);
    return __all_sync(0xffffffffu, ok);
}

// Element i (a compile-time constant after unrolling) of 16 packed bf16.
__device__ __forceinline__ float bf16_at(const uint4 &lo, const uint4 &hi, int i) {
    uint32_t wd;
    switch (i >> 1) {
        case 0: wd = lo.x; break;
        case 1: wd = lo.y; break;
        case 2: wd = lo.z; break;
        case 3: wd = lo.w; break;
        case 4: wd = hi.x; break;
        case 5: wd = hi.y; break;
        case 6: wd = hi.z; break;
        default: wd = hi.w; break;
    }
    return (i & 1) ? bf16_hi(wd) : bf16_lo(wd);
}

// 16 bf16 values starting at p (n valid; the rest read as 0).
__device__ __forceinline__ void load16_bf16(const __nv_bfloat16 *p, int n, uint4 &lo, uint4 &hi) {
    if (n >= 16) {
        lo = __ldg(reinterpret_cast<const uint4 *>(p));
        hi = __ldg(reinterpret_cast<const uint4 *>(p) + 1);
    } else {
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t a = (2 * i < n) ? (uint32_t)__bfloat16_as_ushort(p[2 * i]) : 0u;
            const uint32_t b = (2 * i + 1 < n) ? (uint32_t)__bfloat16_as_ushort(p[2 * i + 1]) : 0u;
            w[i] = a | (b << 16);
        }
        lo = make_uint4(w[0], w[1], w[2], w[3]);
        hi = make_uint4(w[4], w[5], w[6], w[7]);
    }
}

// Pairwise sum of 16 terms (short dependency chains).
__device__ __forceinline__ float sum16(const float (&e)[16]) {
    float s8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) s8[i] = e[2 * i] + e[2 * i + 1];
#pragma unroll
    for (int i = 0; i < 4; ++i) s8[i] += s8[i + 4];
    return (s8[0] + s8[2]) + (s8[1] + s8[3]);
}

// Word i (a compile-time constant after unrolling) of four Philox blocks.
__device__ __forceinline__ uint32_t word_at(const uint4 (&w)[4], int i) {
    const uint4 &b = w[i >> 2];
    switch (i & 3) {
        case 0: return b.x;
        case 1: return b.y;
        case 2: return b.z;
        default: return b.w;
    }
}

// The largest of 16 packed bf16 values (lo: elements 0-7, hi: 8-15), by
// packed maxima (exact: a maximum needs no rounding).
__device__ __forceinline__ float max16_bf16(const uint4 &lo, const uint4 &hi) {
    auto mx = [](uint32_t a, uint32_t b) {
        uint32_t d;
        asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
        return d;
    };
    const uint32_t m = mx(mx(mx(lo.x, lo.y), mx(lo.z, lo.w)), mx(mx(hi.x, hi.y), mx(hi.z, hi.w)));
    return fmaxf(bf16_lo(m), bf16_hi(m));
}

// The draft epilogue's paths for stored logits and greedy rows, out of line:
// they run only when logits are stored or a row has T = 0, and outside the
// loop they leave it smaller (measured on GB300, both together with per-lane
// accumulator hand-back: round 1.2-2.2 % shorter on four workloads).
// The 16 logits come in four float4s.
__device__ __noinline__ void store_z16(float *zo, float4 a, float4 b, float4 c, float4 d, int n) {
    const float z[16] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w, d.x, d.y, d.z, d.w};
    for (int i = 0; i < n; ++i) zo[i] = z[i];
}
// greedy rows: the row's argmax word, its logit and the running maximum
struct GreedyState {
    unsigned long long best;
    float z_at, m;
};
__device__ __noinline__ GreedyState argmax16(GreedyState g, float4 a, float4 b, float4 c, float4 d, int n, int v) {
    const float z[16] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w, d.x, d.y, d.z, d.w};
    for (int i = 0; i < n; ++i) {
        const unsigned long long w = key_word(FF{z[i], 0.f}, v + i);
        if (w > g.best) {
            g.best = w;
            g.z_at = z[i];
        }
        g.m = fmaxf(g.m, z[i]);
    }
    return g;
}

// Element i (a run-time index) of 16 values held in registers: a tree of
// selects on the bits of i, so the values stay in registers.
__device__ __forceinline__ float select16(const float (&z)[16], int i) {
    float a[8], b[4], c[2];
#pragma unroll
    for (int k = 0; k < 8; ++k) a[k] = (i & 8) ? z[k + 8] : z[k];
#pragma unroll
    for (int k = 0; k < 4; ++k) b[k] = (i & 4) ? a[k + 4] : a[k];
#pragma unroll
    for (int k = 0; k < 2; ++k) c[k] = (i & 2) ? b[k + 2] : b[k];
    return (i & 1) ? c[1] : c[0];
}
// Element i (a run-time index) of 16 raw 32-bit values.
__device__ __forceinline__ uint32_t select16(const uint32_t (&z)[16], int i) {
    uint32_t a[8], b[4], c[2];
#pragma unroll
    for (int k = 0; k < 8; ++k) a[k] = (i & 8) ? z[k + 8] : z[k];
#pragma unroll
    for (int k = 0; k < 4; ++k) b[k] = (i & 4) ? a[k + 4] : a[k];
#pragma unroll
    for (int k = 0; k < 2; ++k) c[k] = (i & 2) ? b[k + 2] : b[k];
    return (i & 1) ? c[1] : c[0];
}
// Element i (a run-time index) of 16 packed bf16.
__device__ __forceinline__ float select16_bf16(const uint4 &lo, const uint4 &hi, int i) {
    const uint4 a = (i & 8) ? hi : lo;
    const uint32_t b0 = (i & 4) ? a.z : a.x, b1 = (i & 4) ? a.w : a.y;
    const uint32_t wd = (i & 2) ? b1 : b0;
    return (i & 1) ? bf16_hi(wd) : bf16_lo(wd);
}
// Word i (a run-time index) of four Philox blocks.
__device__ __forceinline__ uint32_t select16(const uint4 (&w)[4], int i) {
    const uint4 a = (i & 8) ? ((i & 4) ? w[3] : w[2]) : ((i & 4) ? w[1] : w[0]);
    const uint32_t b0 = (i & 2) ? a.z : a.x, b1 = (i & 2) ? a.w : a.y;
    return (i & 1) ? b1 : b0;
}

// The largest of the 16 words (the smallest 1 - u of the sub-slice).
__device__ __forceinline__ uint32_t max_word16(const uint4 (&w)[4]) {
    uint32_t a = max(max(w[0].x, w[0].y), max(w[0].z, w[0].w));
    const uint32_t b = max(max(w[1].x, w[1].y), max(w[1].z, w[1].w));
    const uint32_t c = max(max(w[2].x, w[2].y), max(w[2].z, w[2].w));
    const uint32_t d = max(max(w[3].x, w[3].y), max(w[3].z, w[3].w));
    return max(max(a, b), max(c, d));
}

// A lane's running draw of one row in one block position: the two largest
// screened fp32 keys k = z c2 - log2(-ln u) (log2 units) with their logits,
// words and token ids.
struct Top2 {
    float k1, k2;
    float z1, z2;
    uint32_t w1, w2;
    int v1, v2;
};
__device__ __forceinline__ Top2 top2_init() { return Top2{-INFINITY, -INFINITY, 0.f, 0.f, 0u, 0u, -1, -1}; }

// Error bound of a screened key k (log2 units): log2(-ln u) within about
// 1e-5 (log2_neg_log_uniform_fast), the fp32 roundings of z c2 and of k.
__device__ __forceinline__ float screen_tol(float k) { return 2e-5f + 4e-7f * fabsf(k); }

// The screening factor for a threshold K2 in log2 units (see screen_q).
__device__ __forceinline__ float screen_q2(float m, float K2) {
    if (K2 == -INFINITY) return INFINITY;
    return fminf(fast_exp2(m - K2), kQMax) * (1.f + 4e-7f * (fabsf(K2) + fabsf(m) + 64.f));
}

// The smallest Gumbel noise a word can give, g(2^-24) = -ln(24 ln 2), in log2
// units and rounded down: every token's key is at least s2_v + kGminLog2, so a
// lane's largest scaled logit alone bounds the row's best key from below.
constexpr float kGminLog2 = -4.0563f;   // -2.81148 nats * log2(e) = -4.05615

// A published lower bound (natural log) in log2 units, rounded down.
__device__ __forceinline__ float lower_to_log2(float kn) {
    return (kn == -INFINITY) ? -INFINITY : fmaf(kn, kLog2e, -fabsf(kn) * 0x1p-21f);
}

// Raise the threshold K2 (log2 units) to a lower bound of the row's best key
// and publish it in natural log, rounded down, to the CTA's per-row word and
// the row-wide word's high half.
__device__ __forceinline__ void publish_lower(float &K2, float lower, unsigned long long *best, uint32_t *cta_best) {
    K2 = lower;
    const float kn = fmaf(lower, kLn2, -fabsf(lower) * 0x1p-21f);
    red_max_shared_u32(cta_best, key_to_ordered(kn));
    red_max_u64(best, (unsigned long long)key_to_ordered(kn) << 32);
}
// The bound from a scaled logit s2 alone: its token's key is at least
// s2 + kGminLog2 (less the rounding of s2 = z c2).
__device__ __forceinline__ void raise_floor(float &K2, float s2, unsigned long long *best, uint32_t *cta_best) {
    const float lower = s2 + kGminLog2 - 4e-7f * fabsf(s2);
    if (lower > K2) publish_lower(K2, lower, best, cta_best);
}

// Draft epilogue for the 16 logits z of one row (T > 0, c2 = (c2, c2l) =
// log2(e) / T), tokens v .. v + n - 1, with their draft-stream words w (word
// i of token v + i).  Every lane of the warp calls it together (it votes
// across the warp); `on` is false for rows that are greedy or inactive, which
// then change nothing.
//
// Per-token Gumbel-max: token v can reach a key above a threshold K only if
// E_v = -ln u_v < e^(s_v - K) = e_v Q / margin, where e_v = 2^(s2_v - m) is
// the softmax term already computed and Q = screen_q2(m, K log2 e).  Since
// E >= 1 - u, the test (1 - u_v) < e_v Q (conservative form f1 < fl(e Q + 1))
// never loses a token that can reach K.  Most sub-slices are decided by one
// test: the largest word of the 16 against the sub-slice's sum (sum >= every
// e_v).  A sub-slice that passes tests its tokens one by one and gives each
// survivor an fp32 key k (within screen_tol of the exact one); the lane keeps
// its two largest.  K is the largest lower bound known for the row: the
// lane's own k1 - screen_tol(k1), or one another lane published (in natural
// log, to the CTA's per-row word in shared memory and the row-wide word's high
// half in global memory).  The exact (float-float) keys are formed once, at
// the end of the position (draft_top2_word).
//
// The softmax keeps an integer reference m (log2 units) that may lag the
// maximum: terms 2^(z c2 - m) above 1 are fine, and a group whose sum exceeds
// 2^64 (or overflows) is redone against its own maximum.
__device__ __forceinline__ void draft_tokens16(RowState &st, Top2 &tp, float &Q, float &K2, const float (&z)[16],
                                               float c2, float c2l, int n, int v, bool on,
                                               unsigned long long *best, uint32_t *cta_best, const uint4 (&w)[4]) {
    const bool full = (n == 16);  // warp-uniform
    float e[16];
    float sum = 0.f;
    if (on) {
        if (st.m == -INFINITY) {
            // the first group of this thread's row: the reference is its maximum, rounded up
            float zm = -INFINITY;
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (full || i < n) zm = fmaxf(zm, z[i]);
            st.m = ceilf(zm * c2);  // c2 > 0: the rounded product is monotone in z
            raise_floor(K2, zm * c2, best, cta_best);
            Q = screen_q2(st.m, K2);
        }
        if (full) {
#pragma unroll
            for (int i = 0; i < 16; ++i) e[i] = term_exp2(z[i], c2, c2l, st.m);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) e[i] = (i < n) ? term_exp2(z[i], c2, c2l, st.m) : 0.f;
        }
        sum = sum16(e);
        if (!(sum <= 0x1p64f)) {  // far above the reference (or overflow): renormalise
            float zm = -INFINITY;
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (full || i < n) zm = fmaxf(zm, z[i]);
            const float cm = ceilf(fmaxf(st.m, zm * c2));
            st.S = scale_pow2(st.S, st.m - cm);
            st.m = cm;
            raise_floor(K2, zm * c2, best, cta_best);
            Q = screen_q2(st.m, K2);
#pragma unroll
            for (int i = 0; i < 16; ++i) e[i] = (full || i < n) ? term_exp2(z[i], c2, c2l, st.m) : 0.f;
            sum = sum16(e);
        }
        st.S += sum;
    }
    const bool grp = on && sum > 0.f && one_minus_uniform_plus_one(max_word16(w)) < fmaf(sum, Q, 1.f);
    if (!(__any_sync(0xffffffffu, grp) && grp)) return;
    // rare: the tokens one by one (e_v = 0 for tokens past n fails the test).
    // The per-token tests give a mask; only its tokens, in increasing order,
    // take a key (a lane has about four the first time, one or two later, and
    // the warp runs its lanes' largest count instead of all 16).
    const float k1_before = tp.k1;
    uint32_t mask = 0u;
#pragma unroll
    for (int i = 0; i < 16; ++i)
        if (one_minus_uniform_plus_one(word_at(w, i)) < fmaf(e[i], Q, 1.f)) mask |= 1u << i;
#pragma unroll 1
    while (mask) {
        const int i = __ffs(mask) - 1;
        mask &= mask - 1u;
        const float zi = select16(z, i);
        const uint32_t wi = select16(w, i);
        const float k = fmaf(zi, c2l, fmaf(zi, c2, -log2_neg_log_uniform_fast(wi)));
        if (k > tp.k2) {
            if (k > tp.k1) {
                tp.k2 = tp.k1;
                tp.z2 = tp.z1;
                tp.w2 = tp.w1;
                tp.v2 = tp.v1;
                tp.k1 = k;
                tp.z1 = zi;
                tp.w1 = wi;
                tp.v1 = v + i;
            } else {
                tp.k2 = k;
                tp.z2 = zi;
                tp.w2 = wi;
                tp.v2 = v + i;
            }
        }
    }
    if (tp.k1 > k1_before) {
        const float lower = tp.k1 - screen_tol(tp.k1);  // <= the exact key of token v1 (log2 units)
        if (lower > K2) {
            publish_lower(K2, lower, best, cta_best);
            Q = screen_q2(st.m, K2);
        }
    }
}

// The exact key word of a lane's draw: the float-float key of its best
// screened token, and of the second when the two fp32 keys are within their
// error bounds of each other (then the larger word wins).  0 if none.
__device__ __forceinline__ unsigned long long draft_top2_word(const Top2 &tp, float T, float rT, float *z_at) {
    unsigned long long wb = 0ull;
    if (tp.k1 > -INFINITY) {
        wb = key_word(ff_add(div_ff(tp.z1, T, rT), gumbel_ff(tp.w1)), tp.v1);
        *z_at = tp.z1;
        if (tp.k2 >= tp.k1 - screen_tol(tp.k1) - screen_tol(tp.k2)) {
            const unsigned long long w2 = key_word(ff_add(div_ff(tp.z2, T, rT), gumbel_ff(tp.w2)), tp.v2);
            if (w2 > wb) {
                wb = w2;
                *z_at = tp.z2;
            }
        }
    }
    return wb;
}

// A timed-out CTA, before its shared memory and TMEM are given up: the copies
// it armed must land (bytes armed but never issued are counted as landed) and
// the UMMAs it issued must finish; each wait is bounded again.  Out of line:
// the path runs only after a timeout.
// full0: the full_tile barrier of slot 0 (the slots' barriers are 8 bytes apart).
__device__ __noinline__ void drain_copies(uint32_t full0, int armed, uint32_t unissued, volatile int *never) {
    if (armed <= 0) return;
    const int last = armed - 1;
    if (unissued) mbar_complete_tx(full0 + 8u * (uint32_t)(last % kUStages), unissued);
    for (int t = armed > kUStages ? armed - kUStages : 0; t < armed; ++t)
        mbar_wait(full0 + 8u * (uint32_t)(t % kUStages), (uint32_t)(t / kUStages) & 1u, never, kDrainLimit);
}
__device__ __noinline__ void drain_ummas(uint32_t bar, volatile int *never) {
    umma_commit(bar);
    mbar_wait(bar, 0u, never, kDrainLimit);
}

// The warps of the busiest SM sub-partition share its 16K registers: kMaxRegs
// each (15 warps: 4 per sub-partition, 128 registers).
//
// The draft form walks block positions p.j .. p.j_end - 1 in one launch when
// the launch is cooperative: between positions every CTA publishes its rows'
// best (key, token) words and meets the others at a grid barrier; then the
// epilogue warps read x_j, gather the E_in rows of the next position into the
// TMEM A operand and release the MMA warps (a_ready), while the producer has
// already been streaming the next position's W_out and base-logit tiles.
// Tile, ring and accumulator counters run on across positions.
// kQuad: the four-replica form (batches of at most 32 requests), in which
// epilogue warps also pass the tiles where they have no sub-slice.
template <bool kFinal, bool kQuad>
__global__ void __maxnreg__(kMaxRegs)
markov_tc_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_u,
                 const __grid_constant__ TcParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int seg = blockIdx.x;
    const int m0 = blockIdx.y * BM;
    const int vb = seg_begin(seg, p.nseg, p.V);
    const int ve = seg_begin(seg + 1, p.nseg, p.V);
    const int ntiles = (ve - vb + BN - 1) / BN;
    const int npos = kFinal ? 1 : p.j_end - p.j;
    const int total = npos * ntiles;  // tiles of all positions, in order
    // Odd positions (odd passes of the final draw) walk the segment backwards:
    // each then starts on the W_out tiles the previous one touched last, which
    // are still in L2.
    auto tile_col = [&](int tg) {
        const int pi = tg / ntiles, t = tg - pi * ntiles;
        const bool reverse = (((kFinal ? p.pass : p.j + pi)) & 1) != 0;
        return vb + (reverse ? (ntiles - 1 - t) : t) * BN;
    };

    auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * i; };
    // full_tile(slot): every W chunk and the base-logit tile of one tile have
    // landed; empty_w(stage): a W chunk was read; slot_free(slot): every UMMA
    // of the slot's tile is done (its base tile is free and its full_tile
    // phase has been consumed, so the slot may be armed again); a_ready: the
    // A operand of the next position is in TMEM.
    auto empty_w = [&](int s) { return bar(s); };
    auto full_tile = [&](int s) { return bar(kWStages + s); };
    auto slot_free = [&](int s) { return bar(kWStages + kUStages + s); };
    auto tfull = [&](int a) { return bar(kWStages + 2 * kUStages + a); };
    auto tempty = [&](int a) { return bar(kWStages + 2 * kUStages + kAccBufs + a); };
    const uint32_t a_ready = bar(kWStages + 2 * kUStages + 2 * kAccBufs);
    // drain(i): every UMMA of issuer i is done (used only after a timeout)
    auto drain = [&](int i) { return bar(kWStages + 2 * kUStages + 2 * kAccBufs + 1 + i); };

    int *misc = reinterpret_cast<int *>(smem + kOffMisc);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(misc);
    volatile int *abort = misc + 1;
    volatile int *never = misc + 2;  // stays 0: the abort flag of the drain's waits
    int *row_prev = misc + 4;  // final draw: the row's previous token
    float *row_c2 = reinterpret_cast<float *>(misc + 4 + BM);
    uint32_t *row_rid = reinterpret_cast<uint32_t *>(misc + 4 + 2 * BM);
    int *row_code = misc + 4 + 3 * BM;  // final draw: kind << 16 | position; draft: temperature valid
    // draft: the best key of each row found in this CTA during the position
    // (ordered encoding, 0 = none), shared by the quadrant's warps
    uint32_t *row_kbest = reinterpret_cast<uint32_t *>(misc + 4 + 4 * BM);
    float *row_T = reinterpret_cast<float *>(misc + 4 + 5 * BM);  // the row's temperature
    float *row_c2l = reinterpret_cast<float *>(misc + 4 + 6 * BM);  // low part of c2 (c2_split)

    // one position of the recurrent head: launched as a programmatic
    // dependent of the state kernel, so the set-up and the first W_out and
    // base-logit tiles overlap it; its outputs are waited for (griddep_wait)
    // only where they are read, at the A operand build.  (No early trigger
    // for the next state kernel: its blocks would crowd onto the first SMs
    // this grid frees.)
    if (threadIdx.x == 0) {
        for (int s = 0; s < kWStages; ++s) mbar_init(empty_w(s), 1);  // released by the UMMAs
        for (int s = 0; s < kUStages; ++s) {
            mbar_init(full_tile(s), 1);
            mbar_init(slot_free(s), 1);
        }
        for (int a = 0; a < kAccBufs; ++a) {
            mbar_init(tfull(a), 1);
            // one arrival per lane and 16-column sub-slice each quadrant
            // processes; in the four-replica form one per epilogue warp and tile
            mbar_init(tempty(a), kQuad ? kEpiWarps : 32 * (32 / p.rep));
        }
        mbar_init(a_ready, kEpiWarps);
        mbar_init(drain(0), 1);
        mbar_init(drain(1), 1);
        *abort = 0;
        *never = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_desc(&map_w);
        if (!kFinal) tma_prefetch_desc(&map_u);
    }
    // the final draw is launched as a dependent of the decide pass: its set-up
    // above overlaps that pass, whose outputs are read from here on
    if (kFinal) griddep_wait();
    // Small batches (B <= 32 or 64) replicate their requests over the 128
    // TMEM rows, 4 or 2 times, and each replica (a set of lane quadrants)
    // processes its own share of every tile's columns: the epilogue then runs
    // on every SM sub-partition (a warp reads only its own lane quadrant).
    const int rows_q = BM / p.rep;  // distinct requests in the tile
    if (threadIdx.x < BM) {
        const int b = m0 + (int)threadIdx.x % rows_q;
        int prev = -1, code = 0;
        float c2 = 0.f, c2l = 0.f;
        uint32_t id = 0;
        if (b < p.B) {
            const float T = p.temperature[b];
            id = p.request_id ? p.request_id[b] : (uint32_t)b;
            const bool t_ok = T >= 0.f && !isinf(T);
            if (!kFinal) {
                if (p.j == 0 && seg == 0) {
                    const int x0 = p.anchor[b];
                    if (x0 < 0 || x0 >= p.V) atomicOr(p.flags, kFlagBadToken);
                    if (!t_ok) atomicOr(p.flags, kFlagBadTemperature);
                }
                code = t_ok ? 1 : 0;
                if (T > 0.f && t_ok) {
                    const float2 cs = c2_split(T);
                    c2 = cs.x;
                    c2l = cs.y;
                }
            } else {
                code = p.final_code[b];  // validated by the decide kernel
                if (code >= 0) {
                    const int d = code & 0xFFFF;
                    if ((code >> 16) == 1) prev = (d == 0) ? p.anchor[b] : p.tokens[(size_t)b * p.G + d - 1];
                    c2 = kLog2e / T;
                }
            }
        } else if (kFinal) {
            code = -1;
        }
        row_prev[threadIdx.x] = prev;
        row_c2[threadIdx.x] = c2;
        row_c2l[threadIdx.x] = c2l;
        row_rid[threadIdx.x] = id;
        row_code[threadIdx.x] = code;
        row_kbest[threadIdx.x] = 0u;
        row_T[threadIdx.x] = (b < p.B) ? p.temperature[b] : 1.f;
    }
    if (!kFinal && warp < kEpiWarps && threadIdx.x < 16 * 8) {
        // identity row n (16 rows of 128 bytes): a single 1.0 at k = n;
        // 16-byte chunk c of row n sits at position c ^ (n & 7)
        const int n = threadIdx.x >> 3, pos = threadIdx.x & 7, c = pos ^ (n & 7);
        const uint32_t one = (c == (n >> 3)) ? ((n & 1) ? 0x3F800000u : 0x00003F80u) : 0u;
        const int wsel = (n & 7) >> 1;
        st_shared_v4(sbase + kOffI + n * 128 + (pos << 4),
                     make_uint4(wsel == 0 ? one : 0u, wsel == 1 ? one : 0u, wsel == 2 ? one : 0u,
                                wsel == 3 ? one : 0u));
        fence_proxy_async_smem();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int n_katoms = (p.r + 63) >> 6;
    // producer lane 0: tiles whose full_tile phase was armed, and the bytes armed
    // for the last of them that were never issued (a timeout inside the tile)
    int armed = 0;
    uint32_t unissued = 0;

    if (warp == kProducerWarp) {
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_last();
            const uint64_t pol_u = policy_evict_first();
            bool ok = true;
            for (int tg = 0; tg < total && ok; ++tg) {
                const int v0 = tile_col(tg);
                const int jj = p.j + tg / ntiles;
                const int slot = tg % kUStages;
                // the second 64-token box lies past the vocabulary only at its end
                const bool two = v0 + 64 < p.V;
                const uint32_t u_bytes = kFinal ? 0u : (two ? kUBytes : kUHalf);
                for (int kb = 0; kb < n_katoms; ++kb) {
                    const int c = tg * n_katoms + kb;
                    const int ws = c % kWStages;
                    const uint32_t wph = (uint32_t)(c / kWStages) & 1u;
                    if (c >= kWStages && !mbar_wait(empty_w(ws), wph ^ 1u, abort, kSpinLimit)) {
                        ok = false;
                        break;
                    }
                    if (kb == 0) {
                        if (tg >= kUStages &&
                            !mbar_wait(slot_free(slot), ((uint32_t)(tg / kUStages) & 1u) ^ 1u, abort, kSpinLimit)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(full_tile(slot), n_katoms * kWChunk + u_bytes);
                        armed = tg + 1;
                        unissued = n_katoms * kWChunk + u_bytes;
                    }
                    tma_load_2d(sbase + kOffW + ws * kWChunk, &map_w, full_tile(slot), kb * 64, v0, pol_w);
                    unissued -= kWChunk;
                }
                if (ok && !kFinal) {
                    // one box of rows_q requests per replica (128-byte rows: the
                    // swizzle phase of a replica at a multiple of 8 rows is unchanged)
                    for (int k = 0; k < p.rep; ++k) {
                        const uint32_t dst = sbase + kOffU + slot * kUBytes + (uint32_t)(k * rows_q * 128);
                        tma_load_3d(dst, &map_u, full_tile(slot), v0, jj, m0, pol_u);
                        if (two) tma_load_3d(dst + kUHalf, &map_u, full_tile(slot), v0 + 64, jj, m0, pol_u);
                    }
                    unissued -= u_bytes;
                }
            }
            if (!ok) {
                *abort = 1;
                atomicOr(p.flags, kFlagTimeout);
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
        // two issuers, even and odd tiles: a tcgen05.mma costs a roughly fixed
        // issue time, so one thread alone cannot keep the tensor core busy
        // while the epilogue warps share its sub-partition
        if (lane == 0) {
            const int par = warp - kMmaWarp;
            const uint32_t idesc = idesc_bf16_f32(BM, BN);
            const uint32_t idesc16 = idesc_bf16_f32(BM, 16);
            const int ksteps = p.r >> 4;
            // descriptors step in 16-byte units in their low word: K-step s of a
            // 64-wide atom sits at byte 32 (s % 4) of each 128-byte swizzled row
            const uint64_t d_w = sw128_kmajor_desc(sbase + kOffW);
            const uint32_t w_lo0 = (uint32_t)d_w, desc_hi = (uint32_t)(d_w >> 32);
            const uint32_t u_lo0 = (uint32_t)sw128_kmajor_desc(sbase + kOffU);
            const uint32_t i_lo = (uint32_t)sw128_kmajor_desc(sbase + kOffI);
            bool ok = true;
            int last_pi = -1;
            for (int tg = par; tg < total; tg += 2) {
                const int pi = tg / ntiles;
                const int a = tg % kAccBufs;
                const int slot = tg % kUStages;
                // the A operand of this position is in TMEM.  Every phase of
                // a_ready is waited for in order, also those of positions with no
                // tile of this warp (one tile per segment): a parity wait more
                // than one phase ahead would see an older phase as complete.
                while (last_pi < pi && ok) {
                    ++last_pi;
                    ok = mbar_wait(a_ready, (uint32_t)last_pi & 1u, abort, kSpinLimit);
                }
                if (!ok) break;
                if ((tg >= kAccBufs &&
                     !mbar_wait(tempty(a), ((uint32_t)(tg / kAccBufs) & 1u) ^ 1u, abort, kSpinLimit)) ||
                    !mbar_wait(full_tile(slot), (uint32_t)(tg / kUStages) & 1u, abort, kSpinLimit)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + a * BN;
                for (int kb = 0; kb < n_katoms; ++kb) {
                    const int ws = (tg * n_katoms + kb) % kWStages;
                    const uint32_t w_lo = w_lo0 + ws * (kWChunk >> 4);
                    // K-step s = 4 kb + k4: A columns 8 s .. 8 s + 7 of the TMEM copy
                    const uint32_t a_tm = tmem_base + kTmemA + (uint32_t)(32 * kb);
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4)
                        if (4 * kb + k4 < ksteps)
                            umma_bf16_ts(d_tmem, a_tm + 8 * k4, w_lo + 2 * k4, desc_hi, idesc, (kb | k4) ? 1u : 0u);
                    umma_commit(empty_w(ws));
                }
                if (!kFinal) {
                    // + base-logit tile: columns 16 s .. 16 s + 15 get U x identity
                    const uint32_t u_lo = u_lo0 + slot * (kUBytes >> 4);
#pragma unroll
                    for (int s = 0; s < 8; ++s)
                        umma_bf16_w(d_tmem + 16 * s, u_lo + (s >> 2) * (kUHalf >> 4) + 2 * (s & 3), i_lo, desc_hi,
                                    idesc16, 1u);
                }
                umma_commit(slot_free(slot));
                umma_commit(tfull(a));
            }
            if (!ok) {
                *abort = 1;
                atomicOr(p.flags, kFlagTimeout);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ epilogue ----
        const int q = warp & 3, slice = warp >> 2;  // quadrant, index within the quadrant's warps
        const int row = q * 32 + lane;
        const int rq = row % rows_q;  // the request slot of this row (replicas share it)
        const int b = m0 + rq;
        // this quadrant's share of each tile's 8 column blocks: spt = 8 / rep
        // consecutive blocks from cb0; a replica spans 4 / rep whole quadrants
        // (rep is 1 or 2; kQuad: 4, one replica per quadrant)
        const int spt_sh = kQuad ? 1 : (p.rep == 2) ? 2 : 3;
        const int spt = 1 << spt_sh;
        const int cb0 = kQuad ? q * 2 : (p.rep == 2) ? (q >> 1) * 4 : 0;
        const float c2 = row_c2[row];
        const float c2l = row_c2l[row];
        const float Trow = row_T[row];
        const float rT = (Trow > 0.f) ? __frcp_rn(Trow) : 0.f;
        const uint32_t rid = row_rid[row];
        const int code = row_code[row];
        const int kind = kFinal ? (code >= 0 ? (code >> 16) : 0) : 0;
        const int fpos = kFinal ? (code & 0xFFFF) : 0;
        const uint32_t stream = kFinal ? (kind == 1 ? kStreamResidual : kStreamBonus) : kStreamDraft;

        bool ok = true;
        // With one or two replicas every epilogue warp has a sub-slice in every
        // tile (a quadrant's share is 8 or 4 sub-slices for kEpiPerQuad = 3
        // warps) and hands back each one.  With four replicas (kQuad) a
        // quadrant's share of a tile is two sub-slices for three warps, so every
        // warp takes part in every tile, in order: it waits for the tile's
        // accumulator and hands it back once (one arrival per warp), also for a
        // tile in which it has no sub-slice.  Either way the UMMAs never run more
        // than one phase of an accumulator ahead of any warp, and no parity wait
        // can alias.  waited_g: the last tile (counted over all positions) this
        // warp has waited for.
        int waited_g = -1;
        auto pass_tile = [&](int tw) {  // wait for tile tw and hand it straight back
            const bool r = uniform_wait(tfull(tw % kAccBufs), (uint32_t)(tw / kAccBufs) & 1u, abort);
            if (r && lane == 0) mbar_arrive(tempty(tw % kAccBufs));
            return r;
        };
        for (int pi = 0; pi < npos && ok; ++pi) {
            const int jj = kFinal ? 0 : p.j + pi;
            // ---- A operand of this position: TMEM lane = request row, K in
            // pairs per 32-bit column; the quadrant's warp `slice` writes the
            // 64-element K blocks slice, slice + kEpiPerQuad, .. of its rows: E_in[x_{j-1}] (Markov head), or the
            // request's own row of p.a_rows (the recurrent head's state h_j).
            // Every UMMA of the previous position is done: this warp has seen
            // the tfull of its last tile.
            int prev = -1;
            if (!kFinal && p.a_rows && pi == 0) griddep_wait();
            if (kFinal) {
                prev = row_prev[row];
            } else if (b < p.B && code) {
                if (jj == 0) {
                    prev = p.anchor[b];
                    if (prev < 0 || prev >= p.V) prev = -1;
                } else {
                    prev = word_token(load_relaxed_u64(p.best + (size_t)(jj - 1) * p.B + b));
                }
            }
            {
                const __nv_bfloat16 *a_src =
                    (!kFinal && p.a_rows) ? p.a_rows + (size_t)b * p.r : p.e_in + (size_t)max(prev, 0) * p.r;
#pragma unroll 1
                for (int k0 = slice * 64; k0 < p.r; k0 += kEpiPerQuad * 64) {
                    const int nk = min(64, p.r - k0);  // a multiple of 16
                    uint32_t av[32];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        uint4 val = make_uint4(0u, 0u, 0u, 0u);
                        if (prev >= 0 && 8 * i < nk)
                            val = __ldg(reinterpret_cast<const uint4 *>(a_src + k0) + i);
                        av[4 * i] = val.x;
                        av[4 * i + 1] = val.y;
                        av[4 * i + 2] = val.z;
                        av[4 * i + 3] = val.w;
                    }
                    tmem_st32(tmem_base + ((uint32_t)(q * 32) << 16) + kTmemA + (uint32_t)(k0 / 2), av);
                    tmem_st_wait();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(a_ready);
            }
            const bool active = kFinal ? (kind != 0) : (prev >= 0);
            // only rows that draw need words: a warp whose rows are all padding,
            // inactive or greedy skips the Philox blocks (warp-uniform)
            const bool need_words = __any_sync(0xffffffffu, active && c2 > 0.f);
            const uint32_t pos = kFinal ? (uint32_t)fpos : (uint32_t)jj;
            // the parts of Philox fixed by this request and position
            const PhiloxRow prow = philox_row(rid, pos, stream, p.keys);

            RowState st = row_state_init();
            float Q = kQMax;
            float K2 = -INFINITY;  // the largest lower bound of an achieved key of the row (log2 units)
            Top2 tp = top2_init();
            unsigned long long *best = (kFinal || b >= p.B) ? nullptr : p.best + (size_t)jj * p.B + b;
            uint32_t kg_next = 0u;  // "none"
            float kbest_r = -INFINITY;  // best residual key of the row known to this thread
            uint32_t kr_next = 0u;      // the row-wide word, loaded one sub-slice ahead ("none")
            uint32_t *res_best = (kFinal && active) ? p.res_best + b : nullptr;
            ResidualState rs{0ull};
            float lse_q2 = 0.f, lse_t2 = 0.f, lse_q = 0.f;
            FF lse_t{0.f, 0.f};
            const __nv_bfloat16 *urow = nullptr, *trow = nullptr;
            if (kFinal && active) {
                trow = target_row(p.target, p.target_row0, p.n_target_rows, b, p.G, fpos, p.V);  // checked by decide
                if (kind == 1) {
                    urow = p.base + ((size_t)b * p.G + fpos) * p.V;
                    lse_q = p.draft_lse[(size_t)b * p.G + fpos];
                    lse_q2 = lse_q * kLog2e;
                    const float2 lt = p.lse_t_row[b];
                    lse_t = FF{lt.x, lt.y};
                    lse_t2 = lt.x * kLog2e;
                } else {
                    lse_q2 = INFINITY;  // q = 0
                    lse_t2 = 0.f;       // unnormalised p: the same argmax
                }
            }
            // this warp's 16-token sub-slices of this position: sub-slice si is
            // column block si % 8 of tile si / 8; the quadrant's warps take every
            // kEpiPerQuad-th one (so no warp skips a tile)
            const bool rev_pos = (((kFinal ? p.pass : p.j + pi)) & 1) != 0;
            const int nsub = ntiles * spt;
            auto sub_col = [&](int si) {
                const int t = si >> spt_sh;
                return vb + (rev_pos ? (ntiles - 1 - t) : t) * BN + (cb0 + (si & (spt - 1))) * 16;
            };
            // final draw: this thread's target values arrive by cp.async into
            // its own slots of the (otherwise unused) base-logit ring,
            // kTargetAhead - 1 sub-slices ahead (its base values are read only
            // for the groups that pass the bound test).  One commit group per
            // sub-slice, empty where nothing is copied.
            auto prefetch_target = [&](int k) {
                const int sn = slice + k * kEpiPerQuad;
                if (active && sn < nsub) {
                    const int vn = sub_col(sn);
                    const int nn = min(16, ve - vn);
                    if (nn > 0) {
                        const uint32_t dst = target_slot(sbase, k, threadIdx.x);
                        cp_async_16(dst, trow + vn, 2 * min(nn, 8));
                        cp_async_16(dst + kTargetHalf, nn > 8 ? trow + vn + 8 : trow + vn, 2 * max(nn - 8, 0));
                    }
                }
                cp_async_commit();
            };
            if (kFinal) {
#pragma unroll
                for (int k = 0; k < kTargetAhead - 1; ++k) prefetch_target(k);
            }
            int waited = -1;  // the last tile whose accumulator this warp waited for
#pragma unroll 1
            for (int si = slice, k = 0; si < nsub && ok; si += kEpiPerQuad, ++k) {
                const int t = si >> spt_sh;
                const int tg = pi * ntiles + t;
                const int a = tg % kAccBufs;
                const uint32_t aph = (uint32_t)(tg / kAccBufs) & 1u;
                {
                    // The sub-slice's 16 token words (four Philox blocks, counters
                    // v / 4 .. v / 4 + 3) need nothing from the tensor cores.
                    uint4 w[4];
                    uint32_t acc[16];
                    const int vw = sub_col(si);
                    const uint32_t taddr =
                        tmem_base + ((uint32_t)(q * 32) << 16) + a * BN + (uint32_t)(cb0 + (si & (spt - 1))) * 16;
                    auto draw_words = [&]() {
                        if (need_words) {
                            philox_folded4((uint32_t)vw >> 2, prow, p.keys, w);
                        } else {
#pragma unroll
                            for (int g = 0; g < 4; ++g) w[g] = make_uint4(0u, 0u, 0u, 0u);
                        }
                    };
                    if constexpr (kQuad) {
                        // four replicas: one copy of the word code.  On a tile already
                        // waited for, the TMEM load goes first and the words are drawn
                        // under its latency; on a new tile the words are drawn while
                        // its UMMAs may still run, then the accumulator is waited for
                        // and loaded (largev round 531 -> 502 us; the same form in
                        // the one- and two-replica kernel was slower)
                        const bool new_tile = (t != waited);
                        if (!new_tile) tmem_ld16(taddr, acc);
                        draw_words();
                        if (new_tile) {
                            bool w_ok = true;
                            for (int tw = waited_g + 1; tw < tg && w_ok; ++tw) w_ok = pass_tile(tw);  // no sub-slice
                            if (!w_ok || !uniform_wait(tfull(a), aph, abort)) {
                                if (lane == 0) {
                                    *abort = 1;
                                    atomicOr(p.flags, kFlagTimeout);
                                }
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            waited = t;
                            waited_g = tg;
                            tmem_ld16(taddr, acc);
                        }
                    } else if (t != waited) {
                        // a new tile: draw the words while its UMMAs may still run
                        draw_words();
                        if (!uniform_wait(tfull(a), aph, abort)) {
                            if (lane == 0) {
                                *abort = 1;
                                atomicOr(p.flags, kFlagTimeout);
                            }
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        waited = t;
                        tmem_ld16(taddr, acc);
                    } else {
                        // the tile is ready: issue the TMEM load, draw under its latency
                        tmem_ld16(taddr, acc);
                        draw_words();
                    }
                    tmem_ld_wait16(acc);
                    // this sub-slice (kQuad: this warp's last of the tile) is in
                    // registers: hand its part of the accumulator back
                    if (!kQuad) {
                        // every lane hands back its own part once its TMEM load is
                        // done (no warp sync)
                        tc_fence_before();
                        mbar_arrive(tempty(a));
                    } else if (si + kEpiPerQuad >= nsub || ((si + kEpiPerQuad) >> spt_sh) != t) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(tempty(a));
                    }
                    const int v = vw;
                    const int n = min(16, ve - v);
                    if (!kFinal) {
                        if (n <= 0) continue;  // warp-uniform: n depends on the tile and slice only
                        float z[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) z[i] = __uint_as_float(acc[i]);
                        if (p.z_out && active)
                            store_z16(p.z_out + ((size_t)b * p.G + jj) * p.V + v, make_float4(z[0], z[1], z[2], z[3]),
                                      make_float4(z[4], z[5], z[6], z[7]), make_float4(z[8], z[9], z[10], z[11]),
                                      make_float4(z[12], z[13], z[14], z[15]), n);
                        if (active && c2 == 0.f) {
                            const GreedyState g = argmax16(GreedyState{st.best, st.z_at, st.m},
                                                           make_float4(z[0], z[1], z[2], z[3]),
                                                           make_float4(z[4], z[5], z[6], z[7]),
                                                           make_float4(z[8], z[9], z[10], z[11]),
                                                           make_float4(z[12], z[13], z[14], z[15]), n, v);
                            st.best = g.best;
                            st.z_at = g.z_at;
                            st.m = g.m;
                        }
                        const bool on = active && c2 > 0.f;
                        if (on) {
                            // the best key known for the row: this CTA's (shared memory,
                            // current) or the row-wide word's high half (global, loaded
                            // up to four sub-slices earlier)
                            const float kg = lower_to_log2(
                                ordered_to_key(max(kg_next, *(volatile uint32_t *)(row_kbest + rq))));
                            if (kg > K2) {
                                K2 = kg;
                                Q = screen_q2(st.m, K2);
                            }
                        }
                        draft_tokens16(st, tp, Q, K2, z, c2, c2l, n, v, on, best, row_kbest + rq, w);
                        // reload the row-wide word after this warp's first sub-slice of
                        // the position (by then every CTA has published its rows' first
                        // groups, so the threshold is tight from the second sub-slice
                        // on), then every fourth sub-slice, after this one's
                        // publications.  Measured on GB300: 227 us against 238 us with
                        // every fourth alone; every second, every eighth or a
                        // threshold four sub-slices older are slower, never is 10 %
                        // slower.
                        if (on && (si < kEpiPerQuad || ((si / kEpiPerQuad) & 3) == 3))
                            kg_next = load_relaxed(reinterpret_cast<const uint32_t *>(best) + 1);
                    } else {
                        // start the copy kTargetAhead - 1 sub-slices ahead (before any
                        // skip: the skipped sub-slice may come first when walking the
                        // segment backwards; its slot was read last sub-slice), then take
                        // this sub-slice's target values (packed bf16 pairs)
                        prefetch_target(k + kTargetAhead - 1);
                        if (n <= 0) continue;  // warp-uniform
                        cp_async_wait<kTargetAhead - 1>();
                        uint4 ct_lo, ct_hi;
                        {
                            const uint32_t src = target_slot(sbase, k, threadIdx.x);
                            ct_lo = ld_shared_v4(src);
                            ct_hi = ld_shared_v4(src + kTargetHalf);
                        }
                        // Per-token Gumbel-max (stream 2 residual, 3 bonus).  A residual
                        // row weighs token v by r_v = p_v - q_v where positive, with p
                        // and q normalised (reference 0); a bonus row by
                        // 2^(t_v c2 - tref) with the sub-slice's largest scaled logit as
                        // tref (q = 0: lse_q2 = +inf).  Token v can beat the best key K
                        // only if (1 - u_v) < r_v 2^(off - K), off = tref for bonus
                        // rows, 0 for residual rows.  The sub-slice is first tested
                        // with its largest word against a bound from its largest target
                        // logit alone: every r_v <= p_v <= 2^(t_max c2 - tref).
                        const bool bonus = (kind == 2);
                        float tm = -INFINITY;
                        if (n == 16) {
                            tm = max16_bf16(ct_lo, ct_hi);
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                if (i < n) tm = fmaxf(tm, bf16_at(ct_lo, ct_hi, i));
                        }
                        const float off = bonus ? tm * c2 : 0.f;
                        const float tref = bonus ? off : lse_t2;
                        if (active) {
                            // the row-wide best key (one sub-slice old) tightens the threshold
                            const float kg = ordered_to_key(kr_next);
                            if (kg > kbest_r) kbest_r = kg;
                        }
                        const float Qg = screen_q(off, kbest_r);
                        const float pmax = fast_exp2(fmaf(tm, c2, -tref));
                        const bool maybe = active && one_minus_uniform_plus_one(max_word16(w)) < fmaf(pmax, Qg, 1.f);
                        // the row-wide word for the next sub-slice (this thread's own
                        // publications below are already in kbest_r)
                        if (active) kr_next = load_relaxed(res_best);
                        if (!__any_sync(0xffffffffu, maybe)) continue;
                        // per token against p alone (r_v <= p_v, with a margin for the
                        // approximate exponential; exact for bonus rows): most lanes
                        // drop out here, before any base value is read
                        uint32_t pmask = 0u;
                        if (maybe) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                if (i < n) {
                                    const float pv = fast_exp2(fmaf(bf16_at(ct_lo, ct_hi, i), c2, -tref));
                                    if (one_minus_uniform_plus_one(word_at(w, i)) < fmaf(pv * (1.f + 1e-6f), Qg, 1.f))
                                        pmask |= 1u << i;
                                }
                            }
                        }
                        if (!__any_sync(0xffffffffu, pmask != 0u)) continue;
                        // the draft logits z = base + bias of this sub-slice (residual rows)
                        uint4 u_lo = make_uint4(0, 0, 0, 0), u_hi = u_lo;
                        if (pmask && kind == 1) load16_bf16(urow + v, n, u_lo, u_hi);
                        // then per token with an upper bound of r_v = p_v - q_v under the
                        // approximate exponentials (where p and q are close, most
                        // tokens stop here); the survivors form a mask
                        uint32_t mask = 0u;
                        if (pmask) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                if ((pmask >> i) & 1u) {
                                    const float zi = bf16_at(u_lo, u_hi, i) + __uint_as_float(acc[i]);
                                    const float pv = fast_exp2(fmaf(bf16_at(ct_lo, ct_hi, i), c2, -tref));
                                    const float qv = fast_exp2(fmaf(zi, c2, -lse_q2));
                                    const float ub = (pv - qv) + 4e-7f * (pv + qv);
                                    if (ub > 0.f && one_minus_uniform_plus_one(word_at(w, i)) < fmaf(ub, Qg, 1.f))
                                        mask |= 1u << i;
                                }
                            }
                        }
                        // a survivor's fp32 key (log2 units) from an upper bound of r_v
                        // under the approximate exponentials, so never below the true
                        // key by more than rounding; -inf where the bound is not
                        // positive (p <= q: no residual mass)
                        auto fp32_key = [&](int i, float &tb, float &zb, uint32_t &wb) {
                            tb = select16_bf16(ct_lo, ct_hi, i);
                            zb = select16_bf16(u_lo, u_hi, i) + __uint_as_float(select16(acc, i));
                            wb = select16(w, i);
                            const float pv = fast_exp2(fmaf(tb, c2, -tref));
                            const float qv = fast_exp2(fmaf(zb, c2, -lse_q2));
                            const float ub = (pv - qv) + 4e-7f * (pv + qv);
                            return ub > 0.f ? off + fast_log2(ub) - fast_log2(neg_log_uniform(wb)) : -INFINITY;
                        };
                        // the survivor with the largest fp32 key goes first, so that its
                        // float-float key raises the row's best before the others are
                        // tested against it (the largest key word wins, whatever the order)
                        int first = -1;
                        if (mask & (mask - 1u)) {
                            float kb = -INFINITY;
#pragma unroll 1
                            for (uint32_t m2 = mask; m2; m2 &= m2 - 1u) {
                                const int i = __ffs(m2) - 1;
                                float tb, zb;
                                uint32_t wb;
                                const float kk = fp32_key(i, tb, zb, wb);
                                if (kk > kb) {
                                    kb = kk;
                                    first = i;
                                }
                            }
                        }
#pragma unroll 1
                        while (mask) {
                            const int i = (first >= 0) ? first : __ffs(mask) - 1;
                            first = -1;
                            mask &= ~(1u << i);
                            float tb, zb;
                            uint32_t wb;
                            const float kk = fp32_key(i, tb, zb, wb);
                            const float K2 = kbest_r * kLog2e;
                            if (!(kk > K2 - key_tol2(kk, K2))) continue;
                            float key_hi;
                            const unsigned long long word =
                                final_key_word(tb, zb, wb, v + i, bonus, Trow, rT, lse_t, lse_q, &key_hi);
                            if (word > rs.best) {
                                rs.best = word;
                                if (key_hi >= kbest_r) {
                                    kbest_r = key_hi;
                                    red_max_u32(res_best, key_to_ordered(key_hi));
                                }
                            }
                        }
                    }
                }
            }
            // the position's last tiles in which this warp has no sub-slice (or all
            // of them, for a warp with none in this position)
            for (int tw = waited_g + 1; kQuad && ok && tw < (pi + 1) * ntiles; ++tw) {
                if (pass_tile(tw)) {
                    waited_g = tw;
                } else {
                    if (lane == 0) {
                        *abort = 1;
                        atomicOr(p.flags, kFlagTimeout);
                    }
                    ok = false;
                }
            }
            // no copy may still be landing in the target slots (a timed-out
            // warp leaves the loop early)
            if (kFinal) cp_async_wait_all();
            // merge the four column slices of each row
            if (!kFinal) {
                if (c2 > 0.f) {  // sampled rows: the exact key word of the lane's draw
                    float zb = 0.f;
                    st.best = draft_top2_word(tp, Trow, rT, &zb);
                    st.z_at = zb;
                }
                RowState *ms = reinterpret_cast<RowState *>(smem + kOffMerge);
                ms[row * kEpiPerQuad + slice] = st;
            } else {
                ResidualState *ms = reinterpret_cast<ResidualState *>(smem + kOffMerge);
                ms[row * kEpiPerQuad + slice] = rs;
            }
            asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
            // one thread per request merges its row's slices and replicas
            if (slice == 0 && row < rows_q && b < p.B) {
                if (!kFinal) {
                    const RowState *ms = reinterpret_cast<const RowState *>(smem + kOffMerge);
                    for (int k = 0; k < p.rep; ++k)
                        for (int s2 = (k == 0 ? 1 : 0); s2 < kEpiPerQuad; ++s2)
                            row_state_merge(st, ms[(row + k * rows_q) * kEpiPerQuad + s2]);
                    p.part[((size_t)jj * p.B + b) * p.nseg + seg] = st;
                    if (st.best) red_max_u64(best, st.best);
                    row_kbest[rq] = 0u;  // the next position's (every warp is past its last read)
                } else if (active) {
                    const ResidualState *ms = reinterpret_cast<const ResidualState *>(smem + kOffMerge);
                    for (int k = 0; k < p.rep; ++k)
                        for (int s2 = (k == 0 ? 1 : 0); s2 < kEpiPerQuad; ++s2)
                            rs.best = max(rs.best, ms[(row + k * rows_q) * kEpiPerQuad + s2].best);
                    p.rpart[(size_t)b * p.nseg + seg] = rs;
                }
            }
            if (!kFinal && pi + 1 < npos) {
                // every CTA of this row block has published its rows: x_j is final
                // (a row block needs only its own rows' words)
                asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
                if (threadIdx.x == 0 &&
                    !grid_sync(p.grid_bar + blockIdx.y, (unsigned int)(pi + 1) * gridDim.x, abort, kSpinLimit)) {
                    *abort = 1;
                    atomicOr(p.flags, kFlagTimeout);
                }
                // every epilogue warp leaves together if any part of the CTA gave up
                if (named_barrier_or(1, kEpiWarps * 32, *abort != 0)) ok = false;
                __threadfence();
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (*abort) {  // the same for every thread after the barrier
        if (lane == 0) {
            if (warp == kProducerWarp) drain_copies(full_tile(0), armed, unissued, never);
            if (warp == kMmaWarp || warp == kMmaWarp + 1) drain_ummas(drain(warp - kMmaWarp), never);
        }
        __syncwarp();
        tc_fence_before();
        __syncthreads();
    }
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ------------------------------------------------------------------ host ----
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

cudaError_t make_w_map(CUtensorMap *m, const void *w_out, int V, int r) {
    auto fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)r, (cuuint64_t)V};
    cuuint64_t strides[1] = {(cuuint64_t)r * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)BN};
    cuuint32_t estr[2] = {1, 1};
    CUresult res = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(w_out), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Base logits [B][G][V] as a 3-D tensor (V, G, B), boxes of 64 columns x
// 128 requests (box_rows: 128 / the row replication) in the 128-byte swizzled
// layout (two boxes per tile and replica).
cudaError_t make_u_map(CUtensorMap *m, const void *base, int B, int G, int V, int box_cols = 64, int box_rows = BM) {
    auto fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[3] = {(cuuint64_t)V, (cuuint64_t)G, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)V * 2, (cuuint64_t)G * V * 2};
    cuuint32_t box[3] = {(cuuint32_t)box_cols, 1, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    const bool tile = (box_cols == 64);
    // no L2 promotion: the base logits are read once, and promoted sectors
    // only crowd W_out out of L2 (cold-cache DRAM reads of a dspark5 draft
    // launch 554 -> 512 MB, same time)
    CUresult res = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, tile ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                      CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <bool kFinal, bool kQuad>
cudaError_t set_smem_attr() {
    static PerDeviceOnce once;
    return once.run([] {
        return cudaFuncSetAttribute(markov_tc_kernel<kFinal, kQuad>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kSmemBytes);
    });
}
// the kernel form for a row replication (four replicas: kQuad)
template <bool kFinal>
auto tc_kernel(int rep) -> decltype(&markov_tc_kernel<kFinal, false>) {
    return rep == 4 ? &markov_tc_kernel<kFinal, true> : &markov_tc_kernel<kFinal, false>;
}
template <bool kFinal>
cudaError_t set_smem_attrs(int rep) {
    return rep == 4 ? set_smem_attr<kFinal, true>() : set_smem_attr<kFinal, false>();
}

PhiloxRoundKeys round_keys(uint64_t seed) {
    PhiloxRoundKeys K;
    uint32_t k0 = (uint32_t)(seed & 0xFFFFFFFFu), k1 = (uint32_t)(seed >> 32);
    for (int r = 0; r < 10; ++r) {
        K.k0[r] = k0;
        K.k1[r] = k1;
        k0 += kPhiloxW0;
        k1 += kPhiloxW1;
    }
    return K;
}

}  // namespace

int tc_row_blocks(int B) { return (B + BM - 1) / BM; }

// Row replication of the tensor-core kernels: a batch of at most 64 requests
// fills the 128 accumulator rows twice, one of at most 32 four times, each
// replica taking its share of every tile's column blocks.  A replica spans
// whole TMEM lane quadrants (one TMEM load reads the same columns for all 32
// lanes of a warp), so at most 4.  A warp whose quadrant share of a tile holds
// no sub-slice for it still waits on that tile's accumulator phase.
int tc_row_replication(int B) { return B <= 32 ? 4 : (B <= 64 ? 2 : 1); }

int tc_segments(int B, int V) {
    const int mb = tc_row_blocks(B);
    int nseg = kNumSMs / mb;
    if (nseg < 1) nseg = 1;
    const int max_seg = V / BN;
    if (nseg > max_seg) nseg = max_seg < 1 ? 1 : max_seg;
    return nseg;
}

size_t tc_residual_state_bytes() { return sizeof(ResidualState); }

namespace {

// CTAs of the draft kernel that can be resident at once on the current device
// (0 if cooperative launches are unavailable).
int coop_capacity() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    static std::mutex mu;
    static int cached[64];
    static bool have[64];
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 64) return 0;
    if (!have[dev]) {
        int coop = 0, sms = 0, per_sm = 0;
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (coop && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, markov_tc_kernel<false, false>, kThreads,
                                                                 kSmemBytes) == cudaSuccess)
            cached[dev] = per_sm * sms;
        else
            cached[dev] = 0;
        cudaGetLastError();
        have[dev] = true;
    }
    return cached[dev];
}

}  // namespace

namespace {

cudaError_t draft_setup(const DraftArgs &a, const DraftPlan &pl, CUtensorMap *mw, CUtensorMap *mu, TcParams &p) {
    cudaError_t e = make_w_map(mw, a.w_out, a.V, a.r);
    if (e != cudaSuccess) return e;
    const int rep = tc_row_replication(a.B);
    if ((e = make_u_map(mu, a.base, a.B, a.G, a.V, 64, BM / rep)) != cudaSuccess) return e;
    if ((e = set_smem_attrs<false>(rep)) != cudaSuccess) return e;
    p = TcParams{};
    p.e_in = static_cast<const __nv_bfloat16 *>(a.e_in);
    p.base = static_cast<const __nv_bfloat16 *>(a.base);
    p.anchor = a.anchor;
    p.tokens = a.tokens;
    p.temperature = a.temperature;
    p.request_id = a.request_id;
    p.B = a.B;
    p.G = a.G;
    p.V = a.V;
    p.r = a.r;
    p.nseg = pl.nsplit;
    p.rep = rep;
    p.keys = round_keys(a.seed);
    p.part = reinterpret_cast<RowState *>(a.ws + pl.partial_offset);
    p.best = reinterpret_cast<unsigned long long *>(a.ws + pl.best_offset);
    p.grid_bar = reinterpret_cast<unsigned int *>(a.ws + pl.bar_offset);
    p.flags = reinterpret_cast<uint32_t *>(a.ws);
    p.z_out = a.z_out;
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_draft_tensor(const DraftArgs &a, const DraftPlan &pl, cudaStream_t s) {
    CUtensorMap mw, mu;
    TcParams p;
    cudaError_t e = draft_setup(a, pl, &mw, &mu, p);
    if (e != cudaSuccess) return e;
    const dim3 grid(pl.nsplit, pl.row_blocks);
    // all positions in one cooperative launch when every CTA fits at once
    if (a.G > 1 && (long)grid.x * grid.y <= (long)coop_capacity()) {
        p.j = 0;
        p.j_end = a.G;
        void *args[] = {(void *)&mw, (void *)&mu, (void *)&p};
        e = cudaLaunchCooperativeKernel((const void *)tc_kernel<false>(p.rep), grid, dim3(kThreads), args, kSmemBytes,
                                        s);
        if (e != cudaErrorCooperativeLaunchTooLarge) return e;
        cudaGetLastError();  // not resident after all: one launch per position
    }
    for (int j = 0; j < a.G; ++j) {
        p.j = j;
        p.j_end = j + 1;
        tc_kernel<false>(p.rep)<<<grid, kThreads, kSmemBytes, s>>>(mw, mu, p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_draft_tensor_rows(const DraftArgs &a, const DraftPlan &pl, int j, const void *a_rows,
                                     cudaStream_t s) {
    CUtensorMap mw, mu;
    TcParams p;
    cudaError_t e = draft_setup(a, pl, &mw, &mu, p);
    if (e != cudaSuccess) return e;
    p.a_rows = static_cast<const __nv_bfloat16 *>(a_rows);
    p.j = j;
    p.j_end = j + 1;
    // overlap the launch, barrier set-up and the first W_out / base-logit
    // tiles with the state kernel that writes a_rows
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(pl.nsplit, pl.row_blocks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr{};
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc_kernel<false>(p.rep), mw, mu, p);
}

cudaError_t launch_final_tensor(const FinalArgs &a, cudaStream_t s) {
    CUtensorMap mw;
    cudaError_t e = make_w_map(&mw, a.w_out, a.V, a.r);
    if (e != cudaSuccess) return e;
    const int rep = tc_row_replication(a.B);
    if ((e = set_smem_attrs<true>(rep)) != cudaSuccess) return e;
    TcParams p{};
    p.e_in = static_cast<const __nv_bfloat16 *>(a.e_in);
    p.base = static_cast<const __nv_bfloat16 *>(a.base);
    p.target = static_cast<const __nv_bfloat16 *>(a.target);
    p.target_row0 = a.target_row0;
    p.n_target_rows = a.n_target_rows;
    p.anchor = a.anchor;
    p.tokens = a.tokens;
    p.temperature = a.temperature;
    p.request_id = a.request_id;
    p.final_code = a.final_code;
    p.lse_t_row = a.lse_t_row;
    p.draft_lse = a.draft_lse;
    p.B = a.B;
    p.G = a.G;
    p.V = a.V;
    p.r = a.r;
    p.j = 0;
    p.rep = rep;
    p.pass = a.pass;
    p.nseg = a.nseg;
    p.keys = round_keys(a.seed);
    p.rpart = reinterpret_cast<ResidualState *>(a.rpart);
    p.res_best = a.res_best;
    p.flags = a.flags;
    // the final draw reads its base rows directly: map_u is unused
    return launch_dependent(tc_kernel<true>(rep), dim3(a.nseg, tc_row_blocks(a.B)), dim3(kThreads), kSmemBytes, s,
                            mw, mw, p);
}

}  // namespace dspark

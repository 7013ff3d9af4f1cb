// Confidence calibration and the load-aware prefix scheduler.
//
// Method: "DSpark, la bozza che sa quando fermarsi" (paithon.it), section
// "Verificare meglio, non di piu'": confidences c_{b,j} are rescaled with one
// temperature per block position, a_{b,j} = prod_{i<=j} c_{b,i} is the chance
// that the prefix up to j survives, and the scheduler admits the candidate
// tokens of all requests in decreasing a while Theta = tau * SPS(B) grows,
// stopping at the first candidate that does not raise it.
//
// The same page's section "Che cosa resta da verificare" says production drops
// the early stop (and works from confidences two rounds old, which is the
// caller's choice of input); "Verificare meglio, non di piu'" compares with a
// fixed confidence threshold.  Policies:
//  0  early stop (above);
//  1  no early stop: the admitted count with the largest Theta (first on ties);
//  2  threshold on a: L_b grows from L_min while a_{b,L_b} > threshold;
//  3  threshold on c: the same with the per-position confidence (a leading run).
//
// One block of 1024 threads (the work is at most a few thousand candidates):
//  1. c, a per request in fp32 (a fixed left-to-right product); policies 2-3
//     decide the lengths here and skip to 5;
//  2. tau_0 and the candidate list (a, j, b) for L_min <= j < L_max;
//  3. sort by (a desc, j asc, b asc): E <= 8 keys per thread in registers,
//     a bitonic network within each warp, then merge levels through shared
//     memory (a bitonic network in shared memory beyond 8192 candidates);
//  4. block prefix sum of a in float-float, Theta before / after each admission, and
//     the first candidate whose admission does not raise Theta (policy 0,
//     block min) or the count with the largest Theta (policy 1, block argmax);
//  5. scatter the admitted counts into the verify lengths, Theta of the result.
#include <algorithm>
#include <climits>

#include "device_common.cuh"
#include "internal.h"

namespace dspark {
namespace {

constexpr int kSchedThreads = 1024;
// keys per thread of the register sort, at most (more sort in shared memory)
constexpr int kSortRegE = 8;

// Sort key of a candidate: a >= 0 is fp32, so its bit pattern orders like
// its value; (~bits) puts larger a first, the payload j * B + b breaks ties
// by position, then request.
__device__ __forceinline__ unsigned long long cand_key(float a, int pay) {
    return ((unsigned long long)(~__float_as_uint(a)) << 32) | (unsigned int)pay;
}

// tau and Theta in float-float arithmetic (an unevaluated sum hi + lo of two
// floats, about 44 significant bits), on the fp32 pipes: GB300's fp64 rate
// would make this one-block kernel wait on its fp64 unit.
struct ff {
    float hi, lo;
};
__device__ __forceinline__ ff ff_make(float x) { return ff{x, 0.f}; }
// Knuth's two-sum of two floats, then renormalised (|lo| <= ulp(hi) / 2)
__device__ __forceinline__ ff ff_two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return ff{s, e};
}
__device__ __forceinline__ ff ff_fast_norm(float hi, float lo) {
    const float s = __fadd_rn(hi, lo);
    return ff{s, __fsub_rn(lo, __fsub_rn(s, hi))};
}
__device__ __forceinline__ ff ff_add(ff a, ff b) {
    const ff s = ff_two_sum(a.hi, b.hi);
    return ff_fast_norm(s.hi, __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo)));
}
__device__ __forceinline__ ff ff_add_f(ff a, float b) {
    const ff s = ff_two_sum(a.hi, b);
    return ff_fast_norm(s.hi, __fadd_rn(s.lo, a.lo));
}
// a * b for a float b: the product's rounding error from an FMA
__device__ __forceinline__ ff ff_mul_f(ff a, float b) {
    const float p = __fmul_rn(a.hi, b);
    const float e = __fmaf_rn(a.lo, b, __fmaf_rn(a.hi, b, -p));
    return ff_fast_norm(p, e);
}
__device__ __forceinline__ bool ff_gt(ff a, ff b) { return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo); }
__device__ __forceinline__ double ff_to_double(ff a) { return (double)a.hi + (double)a.lo; }
__device__ __forceinline__ ff shfl_xor_ff(ff v, int o) {
    return ff{__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
}
__device__ __forceinline__ ff shfl_up_ff(ff v, int o) {
    return ff{__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
}

__device__ ff block_sum(ff v, ff *red) {
    for (int o = 16; o > 0; o >>= 1) v = ff_add(v, shfl_xor_ff(v, o));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    ff t = (lane < (int)(blockDim.x >> 5)) ? red[lane] : ff_make(0.f);
    for (int o = 16; o > 0; o >>= 1) t = ff_add(t, shfl_xor_ff(t, o));
    return t;
}

// Exclusive prefix over threads of one float-float per thread.
__device__ ff block_exclusive_scan(ff v, ff *red) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    ff incl = v;
    for (int o = 1; o < 32; o <<= 1) {
        const ff n = shfl_up_ff(incl, o);
        if (lane >= o) incl = ff_add(incl, n);
    }
    __syncthreads();
    if (lane == 31) red[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const ff w = (lane < (int)(blockDim.x >> 5)) ? red[lane] : ff_make(0.f);
        ff wi = w;
        for (int o = 1; o < 32; o <<= 1) {
            const ff n = shfl_up_ff(wi, o);
            if (lane >= o) wi = ff_add(wi, n);
        }
        // exclusive prefix of the warp totals: the inclusive one of the lane before
        const ff ex = shfl_up_ff(wi, 1);
        red[lane] = (lane == 0) ? ff_make(0.f) : ex;
    }
    __syncthreads();
    // exclusive within the warp: the inclusive value of the lane before
    const ff before = shfl_up_ff(incl, 1);
    return ff_add(red[warp], lane == 0 ? ff_make(0.f) : before);
}

// Block-wide argmax of (value, index): the larger value, on equal values the
// smaller index.  Every thread gets the result.
__device__ void block_argmax(ff &v, int &n, ff *redv, int *redn) {
    for (int o = 16; o > 0; o >>= 1) {
        const ff v2 = shfl_xor_ff(v, o);
        const int n2 = __shfl_xor_sync(0xffffffffu, n, o);
        if (ff_gt(v2, v) || (v2.hi == v.hi && v2.lo == v.lo && n2 < n)) {
            v = v2;
            n = n2;
        }
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) {
        redv[warp] = v;
        redn[warp] = n;
    }
    __syncthreads();
    v = (lane < (int)(blockDim.x >> 5)) ? redv[lane] : ff{-INFINITY, 0.f};
    n = (lane < (int)(blockDim.x >> 5)) ? redn[lane] : INT_MAX;
    for (int o = 16; o > 0; o >>= 1) {
        const ff v2 = shfl_xor_ff(v, o);
        const int n2 = __shfl_xor_sync(0xffffffffu, n, o);
        if (ff_gt(v2, v) || (v2.hi == v.hi && v2.lo == v.lo && n2 < n)) {
            v = v2;
            n = n2;
        }
    }
}

__device__ __forceinline__ void prefetch_l1(const float *p) { asm volatile("prefetch.global.L1 [%0];" ::"l"(p)); }

// (a, b) <- (min, max) when up, else (max, min)
__device__ __forceinline__ void cmpx(unsigned long long &a, unsigned long long &b, bool up) {
    const unsigned long long lo = min(a, b), hi = max(a, b);
    a = up ? lo : hi;
    b = up ? hi : lo;
}

// Ascending sort of key[0 .. E * blockDim.x) (padding included), E consecutive
// keys per thread (thread t holds keys t E .. t E + E - 1):
//  1. each warp sorts its 32 E keys in registers with a bitonic network
//     (partners within a thread swapped in registers, across lanes by
//     shuffle), every warp's run ascending;
//  2. five merge levels through shared memory join the 32 runs: at run length
//     L each thread finds where its E outputs start on the merge path of its
//     pair of runs (a binary search over the diagonal, ties taken from the
//     first run) and merges E keys from there.
// key[] holds the sorted keys on return.
template <int E>
__device__ void sort_keys(unsigned long long *key) {
    constexpr int n = E * kSchedThreads;
    const int t = threadIdx.x, lane = t & 31;
    unsigned long long v[E];
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = key[t * E + e];
    // 1. bitonic sort of the warp's run (index lane E + e within the run)
#pragma unroll
    for (int k = 2; k <= 32 * E; k <<= 1) {
#pragma unroll
        for (int jj = k >> 1; jj >= E; jj >>= 1) {
            const int d = jj / E;  // partner lane distance
            const bool take_min = (((lane * E) & k) == 0) == ((lane & d) == 0);
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const unsigned long long o = __shfl_xor_sync(0xffffffffu, v[e], d);
                v[e] = take_min ? min(v[e], o) : max(v[e], o);
            }
        }
#pragma unroll
        for (int jl = E >> 1; jl >= 1; jl >>= 1) {
            if (jl < k) {
#pragma unroll
                for (int e = 0; e < E; ++e)
                    if ((e & jl) == 0) cmpx(v[e], v[e | jl], ((lane * E + e) & k) == 0);
            }
        }
    }
    // 2. merge levels
#pragma unroll 1
    for (int L = 32 * E; L < n; L <<= 1) {
        __syncthreads();  // the previous level's reads are done
#pragma unroll
        for (int e = 0; e < E; ++e) key[t * E + e] = v[e];
        __syncthreads();
        const int base = (t * E) & ~(2 * L - 1);  // the pair of runs [base, base + L), [base + L, base + 2 L)
        const int diag = t * E - base;
        const unsigned long long *ra = key + base, *rb = key + base + L;
        int lo = max(0, diag - L), hi = min(diag, L);
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (ra[mid] <= rb[diag - 1 - mid]) lo = mid + 1;
            else hi = mid;
        }
        int i = lo, j = diag - lo;
        unsigned long long ka = ra[min(i, L - 1)], kb = rb[min(j, L - 1)];
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const bool take_a = j >= L || (i < L && ka <= kb);
            v[e] = take_a ? ka : kb;
            if (e + 1 < E) {
                if (take_a) ka = ra[min(++i, L - 1)];
                else kb = rb[min(++j, L - 1)];
            }
        }
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < E; ++e) key[t * E + e] = v[e];
    __syncthreads();
}

// A bitonic network on keys in shared memory, one compare-exchange per thread
// and loop step, a block barrier per stage: for more than kSortRegE keys per
// thread, where the register form would spill.
__device__ void bitonic_sort_shared(unsigned long long *key, int n) {
    for (int k = 2; k <= n; k <<= 1) {
        for (int jj = k >> 1; jj > 0; jj >>= 1) {
            for (int i = threadIdx.x; i < n; i += blockDim.x) {
                const int ixj = i ^ jj;
                if (ixj > i) {
                    const unsigned long long ki = key[i], kx = key[ixj];
                    const bool up = (i & k) == 0;
                    if (up ? (kx < ki) : (ki < kx)) {
                        key[i] = kx;
                        key[ixj] = ki;
                    }
                }
            }
            __syncthreads();
        }
    }
}

__global__ void __launch_bounds__(kSchedThreads)
schedule_kernel(const float *__restrict__ conf_logits, const float *__restrict__ pos_temp,
                const float *__restrict__ sps, int B, int G, int L_min, int L_max, int npow2, int policy,
                float threshold, float *__restrict__ conf, float *__restrict__ cum_conf,
                int32_t *__restrict__ verify_len, double *__restrict__ theta_out,
                uint32_t *__restrict__ flags) {
    griddep_wait();  // a programmatic dependent: the previous launch's writes are visible after this
    extern __shared__ unsigned long long smem[];
    // the sort runs over nsort keys: the candidates' power of two, at least one per thread
    const int nsort = max(npow2, kSchedThreads);
    unsigned long long *key = smem;                       // [nsort] sort keys
    int *len_s = reinterpret_cast<int *>(key + nsort);    // [B]
    __shared__ ff red[32];
    __shared__ int redn[32];
    __shared__ float pt_s[kMaxG];  // position temperatures
    __shared__ int first_fail;
    __shared__ int bad_temp;

    const int tid = threadIdx.x;
    const int width = L_max - L_min;
    const int ncand = B * width;
    if (tid == 0) {
        first_fail = ncand;
        bad_temp = 0;
    }
    // the call's flag words start clear (this block is their only writer)
    if (tid < (int)(kFlagBytes / sizeof(uint32_t))) flags[tid] = 0u;
    __syncthreads();
    for (int j = tid; j < G; j += blockDim.x) {
        const float T = pos_temp[j];
        pt_s[j] = T;
        if (!(T > 0.f) || isinf(T)) atomicOr(&bad_temp, 1);
    }
    __syncthreads();
    if (bad_temp) {
        if (tid == 0) atomicOr(flags, kFlagBadPosTemp);
        for (int b = tid; b < B; b += blockDim.x) verify_len[b] = L_min;
        for (int i = tid; i < B * G; i += blockDim.x) {
            conf[i] = __int_as_float(0x7fc00000);
            cum_conf[i] = __int_as_float(0x7fc00000);
        }
        if (tid == 0 && theta_out) *theta_out = __longlong_as_double(0x7ff8000000000000LL);
        return;
    }

    // 1-2. calibrated confidences, prefix products, tau_0, candidates (policies
    // 2-3: the lengths, tau and the batch tokens of the result)
    ff tau_part = ff_make(0.f), tok_part = ff_make(0.f);
    for (int b = tid; b < B; b += blockDim.x) {
        float prod = 1.f;
        ff t = ff_make(1.f);
        int L = L_min;
        bool run = true;
        const float *lrow = conf_logits + (size_t)b * G;
        // the row's logits eight at a time (the loads in flight together)
        for (int j0 = 0; j0 < G; j0 += 8) {
            float lg[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) lg[u] = (j0 + u < G) ? lrow[j0 + u] : 0.f;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int j = j0 + u;
                if (j >= G) break;
                const float c = 1.f / (1.f + expf(-lg[u] / pt_s[j]));
                prod *= c;
                conf[(size_t)b * G + j] = c;
                cum_conf[(size_t)b * G + j] = prod;
                if (policy >= 2) {
                    if (run && j >= L_min && j < L_max) {
                        run = (policy == 2 ? prod : c) > threshold;
                        if (run) L = j + 1;
                    }
                    if (j < L) t = ff_add_f(t, prod);
                } else {
                    if (j < L_min) t = ff_add_f(t, prod);
                    if (j >= L_min && j < L_max) key[b * width + (j - L_min)] = cand_key(prod, j * B + b);
                }
            }
        }
        tau_part = ff_add(tau_part, t);
        len_s[b] = L;
        tok_part = ff_add_f(tok_part, (float)(L + 1));
    }
    if (policy >= 2) {
        const ff tau = block_sum(tau_part, red);
        const ff tok = block_sum(tok_part, red);  // an integer below 2^24: exact
        for (int b = tid; b < B; b += blockDim.x) verify_len[b] = len_s[b];
        if (tid == 0 && theta_out) *theta_out = ff_to_double(tau) * (double)sps[(long)tok.hi];
        return;
    }
    for (int i = ncand + tid; i < nsort; i += blockDim.x) key[i] = ~0ull;
    const ff tau0 = block_sum(tau_part, red);
    __syncthreads();

    // 3. bitonic sort: highest priority first (ascending keys)
    switch (nsort / kSchedThreads) {
        case 1: sort_keys<1>(key); break;
        case 2: sort_keys<2>(key); break;
        case 4: sort_keys<4>(key); break;
        case kSortRegE: sort_keys<kSortRegE>(key); break;
        default: bitonic_sort_shared(key, nsort); break;
    }

    // 4. prefix sums and the first admission that does not raise Theta
    const long n0 = (long)B * (L_min + 1);
    const int per = (ncand + blockDim.x - 1) / blockDim.x;
    const int lo = min(ncand, tid * per), hi = min(ncand, lo + per);
    // this thread's entries of the SPS table into L1 while the scan runs
    for (int i = lo; i < hi; ++i) prefetch_l1(sps + n0 + i + 1);
    if (lo < hi) prefetch_l1(sps + n0 + lo);
    auto a_of = [&](int i) { return __uint_as_float(~(unsigned int)(key[i] >> 32)); };
    ff local = ff_make(0.f);
    for (int i = lo; i < hi; ++i) local = ff_add_f(local, a_of(i));
    const ff before = block_exclusive_scan(local, red);
    ff run = ff_add(tau0, before);  // tau before candidate lo
    int nstar;
    if (policy == 0) {
        for (int i = lo; i < hi; ++i) {
            const float a = a_of(i);
            const ff th_before = ff_mul_f(run, sps[n0 + i]);
            const ff next = ff_add_f(run, a);
            const ff th_after = ff_mul_f(next, sps[n0 + i + 1]);
            if (!ff_gt(th_after, th_before)) {
                atomicMin(&first_fail, i);
                break;
            }
            run = next;
        }
        __syncthreads();
        nstar = first_fail;
    } else {
        // Theta after admitting the first n candidates, n = 0 .. ncand
        ff bv = (tid == 0) ? ff_mul_f(tau0, sps[n0]) : ff{-INFINITY, 0.f};
        int bn = (tid == 0) ? 0 : INT_MAX;
        for (int i = lo; i < hi; ++i) {
            run = ff_add_f(run, a_of(i));
            const ff th = ff_mul_f(run, sps[n0 + i + 1]);
            if (ff_gt(th, bv)) {
                bv = th;
                bn = i + 1;
            }
        }
        block_argmax(bv, bn, red, redn);
        nstar = bn;
        __syncthreads();
    }
    // tau after the admitted prefix, for Theta
    ff adm = ff_make(0.f);
    for (int i = lo; i < min(hi, nstar); ++i) adm = ff_add_f(adm, a_of(i));
    const ff tau_final = ff_add(tau0, block_sum(adm, red));

    // 5. verify lengths
    for (int i = tid; i < nstar; i += blockDim.x) atomicAdd(&len_s[(int)(key[i] & 0xFFFFFFFFu) % B], 1);
    __syncthreads();
    for (int b = tid; b < B; b += blockDim.x) verify_len[b] = len_s[b];
    if (tid == 0 && theta_out) *theta_out = ff_to_double(tau_final) * (double)sps[n0 + nstar];
}

}  // namespace

size_t schedule_smem_bytes(int B, int G, int L_min, int L_max) {
    (void)G;
    const long ncand = (long)B * (L_max - L_min);
    long npow2 = 1;
    while (npow2 < ncand) npow2 <<= 1;
    return (size_t)std::max(npow2, (long)kSchedThreads) * sizeof(unsigned long long) + sizeof(int) * (size_t)B;
}

cudaError_t launch_schedule(const ScheduleArgs &a, cudaStream_t s) {
    // (policies 2-3 do not sort, but one launch shape serves all)
    const long ncand = (long)a.B * (a.L_max - a.L_min);
    int npow2 = 1;
    while (npow2 < ncand) npow2 <<= 1;
    const size_t smem = schedule_smem_bytes(a.B, a.G, a.L_min, a.L_max);
    // the dynamic shared-memory limit is raised once per device, to the most
    // the entry points accept
    static PerDeviceOnce attr;
    cudaError_t e = attr.run([] {
        return cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kScheduleMaxSmem);
    });
    if (e != cudaSuccess) return e;
    if (smem > (size_t)kScheduleMaxSmem) return cudaErrorInvalidValue;
    // a programmatic dependent of the launch before it (the kernel waits for
    // that launch before its first access)
    return launch_dependent(schedule_kernel, dim3(1), dim3(kSchedThreads), smem, s, a.conf_logits, a.pos_temp,
                            a.sps, a.B, a.G, a.L_min, a.L_max, npow2, a.policy, a.threshold, a.conf, a.cum_conf,
                            a.verify_len, a.theta_out, reinterpret_cast<uint32_t *>(a.ws));
}

}  // namespace dspark

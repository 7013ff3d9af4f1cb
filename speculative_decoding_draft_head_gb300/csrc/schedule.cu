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
//  3. bitonic sort in shared memory by (a desc, j asc, b asc);
//  4. block prefix sum of a in float-float, Theta before / after each admission, and
//     the first candidate whose admission does not raise Theta (policy 0,
//     block min) or the count with the largest Theta (policy 1, block argmax);
//  5. scatter the admitted counts into the verify lengths, Theta of the result.
#include <climits>

#include "device_common.cuh"
#include "internal.h"

namespace dspark {
namespace {

constexpr int kSchedThreads = 1024;

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

__global__ void __launch_bounds__(kSchedThreads)
schedule_kernel(const float *__restrict__ conf_logits, const float *__restrict__ pos_temp,
                const float *__restrict__ sps, int B, int G, int L_min, int L_max, int npow2, int policy,
                float threshold, float *__restrict__ conf, float *__restrict__ cum_conf,
                int32_t *__restrict__ verify_len, double *__restrict__ theta_out,
                uint32_t *__restrict__ flags) {
    extern __shared__ unsigned long long smem[];
    unsigned long long *key = smem;                       // [npow2] sort keys
    int *len_s = reinterpret_cast<int *>(key + npow2);    // [B]
    __shared__ ff red[32];
    __shared__ int redn[32];
    __shared__ unsigned long long xch[kSchedThreads];  // register-sort exchange
    __shared__ int first_fail;
    __shared__ int bad_temp;

    const int tid = threadIdx.x;
    const int width = L_max - L_min;
    const int ncand = B * width;
    if (tid == 0) {
        first_fail = ncand;
        bad_temp = 0;
    }
    __syncthreads();
    for (int j = tid; j < G; j += blockDim.x) {
        const float T = pos_temp[j];
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
        for (int j = 0; j < G; ++j) {
            const float l = conf_logits[(size_t)b * G + j];
            const float c = 1.f / (1.f + expf(-l / pos_temp[j]));
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
    for (int i = ncand + tid; i < npow2; i += blockDim.x) key[i] = ~0ull;
    const ff tau0 = block_sum(tau_part, red);
    __syncthreads();

    // 3. bitonic sort: highest priority first (ascending keys)
    if (npow2 <= kSchedThreads) {
        // one key per thread (padding sorts last): partners closer than a warp
        // are exchanged by shuffle, the others through shared memory
        unsigned long long kv = (tid < npow2) ? key[tid] : ~0ull;
        for (int k = 2; k <= kSchedThreads; k <<= 1) {
            for (int jj = k >> 1; jj > 0; jj >>= 1) {
                unsigned long long other;
                if (jj >= 32) {
                    __syncthreads();
                    xch[tid] = kv;
                    __syncthreads();
                    other = xch[tid ^ jj];
                } else {
                    other = __shfl_xor_sync(0xffffffffu, kv, jj);
                }
                const bool up = (tid & k) == 0, lower = (tid & jj) == 0;
                kv = (up == lower) ? min(kv, other) : max(kv, other);
            }
        }
        __syncthreads();
        if (tid < npow2) key[tid] = kv;
        __syncthreads();
    } else {
        for (int k = 2; k <= npow2; k <<= 1) {
            for (int jj = k >> 1; jj > 0; jj >>= 1) {
                for (int i = tid; i < npow2; i += blockDim.x) {
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

    // 4. prefix sums and the first admission that does not raise Theta
    const long n0 = (long)B * (L_min + 1);
    const int per = (ncand + blockDim.x - 1) / blockDim.x;
    const int lo = min(ncand, tid * per), hi = min(ncand, lo + per);
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
    return (size_t)npow2 * sizeof(unsigned long long) + sizeof(int) * (size_t)B;
}

cudaError_t launch_schedule(const ScheduleArgs &a, cudaStream_t s) {
    // (policies 2-3 do not sort, but one launch shape serves all)
    const long ncand = (long)a.B * (a.L_max - a.L_min);
    int npow2 = 1;
    while (npow2 < ncand) npow2 <<= 1;
    const size_t smem = schedule_smem_bytes(a.B, a.G, a.L_min, a.L_max);
    cudaError_t e = cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    schedule_kernel<<<1, kSchedThreads, smem, s>>>(a.conf_logits, a.pos_temp, a.sps, a.B, a.G, a.L_min,
                                                    a.L_max, npow2, a.policy, a.threshold, a.conf, a.cum_conf,
                                                    a.verify_len, a.theta_out, reinterpret_cast<uint32_t *>(a.ws));
    return cudaGetLastError();
}

}  // namespace dspark

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
//  4. block prefix sum of a in fp64, Theta before / after each admission, and
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

__device__ double block_sum(double v, double *red) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    double t = (lane < (int)(blockDim.x >> 5)) ? red[lane] : 0.0;
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    return t;
}

// Exclusive prefix over threads of one double per thread.
__device__ double block_exclusive_scan(double v, double *red) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    double incl = v;
    for (int o = 1; o < 32; o <<= 1) {
        const double n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    __syncthreads();
    if (lane == 31) red[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        double w = (lane < (int)(blockDim.x >> 5)) ? red[lane] : 0.0;
        double wi = w;
        for (int o = 1; o < 32; o <<= 1) {
            const double n = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += n;
        }
        red[lane] = wi - w;  // exclusive prefix of warp totals
    }
    __syncthreads();
    return red[warp] + (incl - v);
}

// Block-wide argmax of (value, index): the larger value, on equal values the
// smaller index.  Every thread gets the result.
__device__ void block_argmax(double &v, int &n, double *redv, int *redn) {
    for (int o = 16; o > 0; o >>= 1) {
        const double v2 = __shfl_xor_sync(0xffffffffu, v, o);
        const int n2 = __shfl_xor_sync(0xffffffffu, n, o);
        if (v2 > v || (v2 == v && n2 < n)) {
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
    v = (lane < (int)(blockDim.x >> 5)) ? redv[lane] : -INFINITY;
    n = (lane < (int)(blockDim.x >> 5)) ? redn[lane] : INT_MAX;
    for (int o = 16; o > 0; o >>= 1) {
        const double v2 = __shfl_xor_sync(0xffffffffu, v, o);
        const int n2 = __shfl_xor_sync(0xffffffffu, n, o);
        if (v2 > v || (v2 == v && n2 < n)) {
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
    __shared__ double red[32];
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
    double tau_part = 0.0, tok_part = 0.0;
    for (int b = tid; b < B; b += blockDim.x) {
        float prod = 1.f;
        double t = 1.0;
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
                if (j < L) t += (double)prod;
            } else {
                if (j < L_min) t += (double)prod;
                if (j >= L_min && j < L_max) key[b * width + (j - L_min)] = cand_key(prod, j * B + b);
            }
        }
        tau_part += t;
        len_s[b] = L;
        tok_part += (double)(L + 1);
    }
    if (policy >= 2) {
        const double tau = block_sum(tau_part, red);
        const double tok = block_sum(tok_part, red);
        for (int b = tid; b < B; b += blockDim.x) verify_len[b] = len_s[b];
        if (tid == 0 && theta_out) *theta_out = tau * (double)sps[(long)tok];
        return;
    }
    for (int i = ncand + tid; i < npow2; i += blockDim.x) key[i] = ~0ull;
    const double tau0 = block_sum(tau_part, red);
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
    auto a_of = [&](int i) { return (double)__uint_as_float(~(unsigned int)(key[i] >> 32)); };
    double local = 0.0;
    for (int i = lo; i < hi; ++i) local += a_of(i);
    const double before = block_exclusive_scan(local, red);
    double run = tau0 + before;  // tau before candidate lo
    int nstar;
    if (policy == 0) {
        for (int i = lo; i < hi; ++i) {
            const double a = a_of(i);
            const double th_before = run * (double)sps[n0 + i];
            const double th_after = (run + a) * (double)sps[n0 + i + 1];
            if (!(th_after > th_before)) {
                atomicMin(&first_fail, i);
                break;
            }
            run += a;
        }
        __syncthreads();
        nstar = first_fail;
    } else {
        // Theta after admitting the first n candidates, n = 0 .. ncand
        double bv = (tid == 0) ? tau0 * (double)sps[n0] : -INFINITY;
        int bn = (tid == 0) ? 0 : INT_MAX;
        for (int i = lo; i < hi; ++i) {
            run += a_of(i);
            const double th = run * (double)sps[n0 + i + 1];
            if (th > bv) {
                bv = th;
                bn = i + 1;
            }
        }
        block_argmax(bv, bn, red, redn);
        nstar = bn;
        __syncthreads();
    }
    // tau after the admitted prefix, for Theta
    double adm = 0.0;
    for (int i = lo; i < min(hi, nstar); ++i) adm += a_of(i);
    const double tau_final = tau0 + block_sum(adm, red);

    // 5. verify lengths
    for (int i = tid; i < nstar; i += blockDim.x) atomicAdd(&len_s[(int)(key[i] & 0xFFFFFFFFu) % B], 1);
    __syncthreads();
    for (int b = tid; b < B; b += blockDim.x) verify_len[b] = len_s[b];
    if (tid == 0 && theta_out) *theta_out = tau_final * (double)sps[n0 + nstar];
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

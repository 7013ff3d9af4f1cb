// Confidence calibration and the load-aware prefix scheduler.
//
// Method: "DSpark, la bozza che sa quando fermarsi" (paithon.it), section
// "Verificare meglio, non di piu'": confidences c_{b,j} are rescaled with one
// temperature per block position, a_{b,j} = prod_{i<=j} c_{b,i} is the chance
// that the prefix up to j survives, and the scheduler admits the candidate
// tokens of all requests in decreasing a while Theta = tau * SPS(B) grows,
// stopping at the first candidate that does not raise it.
//
// One block of 1024 threads (the work is at most a few thousand candidates):
//  1. c, a per request in fp64 (a fixed left-to-right product), fp32 copies out;
//  2. tau_0 and the candidate list (a, j, b) for L_min <= j < L_max;
//  3. bitonic sort in shared memory by (a desc, j asc, b asc);
//  4. block prefix sum of a, Theta before / after each admission, the first
//     candidate whose admission does not raise Theta (block min);
//  5. scatter the admitted counts into the verify lengths.
#include <climits>

#include "device_common.cuh"
#include "internal.h"

namespace dspark {
namespace {

constexpr int kSchedThreads = 1024;

__device__ __forceinline__ bool cand_before(double ka, int pa, double kb, int pb) {
    return ka > kb || (ka == kb && pa < pb);
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

__global__ void __launch_bounds__(kSchedThreads)
schedule_kernel(const float *__restrict__ conf_logits, const float *__restrict__ pos_temp,
                const float *__restrict__ sps, int B, int G, int L_min, int L_max, int npow2,
                float *__restrict__ conf, float *__restrict__ cum_conf,
                int32_t *__restrict__ verify_len, double *__restrict__ theta_out,
                uint32_t *__restrict__ flags) {
    extern __shared__ double smem[];
    double *key = smem;                                   // [npow2]
    int *pay = reinterpret_cast<int *>(key + npow2);      // [npow2]: j * B + b
    int *len_s = pay + npow2;                             // [B]
    __shared__ double red[32];
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

    // 1-2. calibrated confidences, prefix products, tau_0, candidates
    double tau_part = 0.0;
    for (int b = tid; b < B; b += blockDim.x) {
        double prod = 1.0;
        double t = 1.0;
        for (int j = 0; j < G; ++j) {
            const double l = (double)conf_logits[(size_t)b * G + j];
            const double c = 1.0 / (1.0 + exp(-l / (double)pos_temp[j]));
            prod *= c;
            conf[(size_t)b * G + j] = (float)c;
            cum_conf[(size_t)b * G + j] = (float)prod;
            if (j < L_min) t += prod;
            if (j >= L_min && j < L_max) {
                const int i = b * width + (j - L_min);
                key[i] = prod;
                pay[i] = j * B + b;
            }
        }
        tau_part += t;
        len_s[b] = L_min;
    }
    for (int i = ncand + tid; i < npow2; i += blockDim.x) {
        key[i] = -1.0;
        pay[i] = INT_MAX;
    }
    const double tau0 = block_sum(tau_part, red);
    __syncthreads();

    // 3. bitonic sort: highest priority first
    for (int k = 2; k <= npow2; k <<= 1) {
        for (int jj = k >> 1; jj > 0; jj >>= 1) {
            for (int i = tid; i < npow2; i += blockDim.x) {
                const int ixj = i ^ jj;
                if (ixj > i) {
                    const double ki = key[i], kx = key[ixj];
                    const int pi = pay[i], px = pay[ixj];
                    const bool up = (i & k) == 0;
                    const bool swap = up ? cand_before(kx, px, ki, pi) : cand_before(ki, pi, kx, px);
                    if (swap) {
                        key[i] = kx; key[ixj] = ki;
                        pay[i] = px; pay[ixj] = pi;
                    }
                }
            }
            __syncthreads();
        }
    }

    // 4. prefix sums and the first admission that does not raise Theta
    const long n0 = (long)B * (L_min + 1);
    const int per = (ncand + blockDim.x - 1) / blockDim.x;
    const int lo = min(ncand, tid * per), hi = min(ncand, lo + per);
    double local = 0.0;
    for (int i = lo; i < hi; ++i) local += key[i];
    const double before = block_exclusive_scan(local, red);
    double run = tau0 + before;  // tau before candidate lo
    for (int i = lo; i < hi; ++i) {
        const double th_before = run * (double)sps[n0 + i];
        const double th_after = (run + key[i]) * (double)sps[n0 + i + 1];
        if (!(th_after > th_before)) {
            atomicMin(&first_fail, i);
            break;
        }
        run += key[i];
    }
    __syncthreads();
    const int nstar = first_fail;
    // tau after the admitted prefix, for Theta
    double adm = 0.0;
    for (int i = lo; i < min(hi, nstar); ++i) adm += key[i];
    const double tau_final = tau0 + block_sum(adm, red);

    // 5. verify lengths
    for (int i = tid; i < nstar; i += blockDim.x) atomicAdd(&len_s[pay[i] % B], 1);
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
    return (size_t)npow2 * (sizeof(double) + sizeof(int)) + sizeof(int) * (size_t)B;
}

cudaError_t launch_schedule(const ScheduleArgs &a, cudaStream_t s) {
    const long ncand = (long)a.B * (a.L_max - a.L_min);
    int npow2 = 1;
    while (npow2 < ncand) npow2 <<= 1;
    const size_t smem = schedule_smem_bytes(a.B, a.G, a.L_min, a.L_max);
    cudaError_t e = cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    schedule_kernel<<<1, kSchedThreads, smem, s>>>(a.conf_logits, a.pos_temp, a.sps, a.B, a.G, a.L_min,
                                                    a.L_max, npow2, a.conf, a.cum_conf, a.verify_len,
                                                    a.theta_out, reinterpret_cast<uint32_t *>(a.ws));
    return cudaGetLastError();
}

}  // namespace dspark

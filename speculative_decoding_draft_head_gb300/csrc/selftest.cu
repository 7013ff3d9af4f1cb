// Self-tests: the bounded waits every kernel of the library relies on, and the
// device's rate for the draw's random words.
//
// Bounded waits: one block waits, with the production helpers and a short
// limit, on an mbarrier phase that no thread completes and on a global counter
// that no thread increments.  Both must give up and report it; the context
// stays usable (nothing faults, traps or spins without a limit).
//
// Random words: a full grid draws Philox4x32-10 blocks with the library's own
// folded form (philox_folded4, the draft's per-token words), nothing else, and
// reports the blocks per second: the ALU roof of the per-token Gumbel-max
// draw, measured on the device that runs it.
#include "device_common.cuh"
#include "internal.h"
#include "tc_primitives.cuh"

namespace dspark {

__device__ unsigned int g_selftest_counter;  // never incremented
__device__ uint32_t g_selftest_result;

namespace {

__global__ void bounded_wait_probe_kernel(long long limit_cycles) {
    __shared__ __align__(8) unsigned long long mbar;
    __shared__ int abort;
    if (threadIdx.x == 0) {
        tc::mbar_init(tc::smem_u32(&mbar), 1);
        abort = 0;
        tc::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const bool mbar_done = tc::mbar_wait(tc::smem_u32(&mbar), 0u, &abort, limit_cycles);
        const bool counter_done = counter_wait(&g_selftest_counter, 1u, &abort, limit_cycles);
        g_selftest_result = (mbar_done ? 0u : 1u) | (counter_done ? 0u : 2u);
    }
}

constexpr int kRateThreads = 512;

__global__ void __launch_bounds__(kRateThreads) philox_rate_kernel(uint32_t *sink, int iters, PhiloxRoundKeys K) {
    const uint32_t gid = blockIdx.x * blockDim.x + threadIdx.x;
    const PhiloxRow R = philox_row(gid, 1u, kStreamDraft, K);
    uint32_t acc = 0u;
    uint32_t x = gid << 12;
    for (int it = 0; it < iters; ++it) {
        uint4 w[4];
        philox_folded4(x, R, K, w);
#pragma unroll
        for (int g = 0; g < 4; ++g) acc ^= (w[g].x ^ w[g].y) ^ (w[g].z ^ w[g].w);
        x += 4u;
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, m);
    if ((threadIdx.x & 31) == 0) sink[gid >> 5] = acc;  // keeps the words live
}

}  // namespace

size_t philox_probe_sink_bytes(int sms) { return (size_t)sms * 4 * (kRateThreads / 32) * sizeof(uint32_t); }

cudaError_t run_philox_probe(void *sink, int sms, int iters, double *blocks_per_s, cudaStream_t s) {
    PhiloxRoundKeys K;
    uint32_t k0 = 0x12345678u, k1 = 0x9abcdef0u;
    for (int r = 0; r < 10; ++r) {
        K.k0[r] = k0;
        K.k1[r] = k1;
        k0 += kPhiloxW0;
        k1 += kPhiloxW1;
    }
    const int blocks = sms * 4;  // 2048 threads per SM
    cudaEvent_t e0, e1;
    cudaError_t e = cudaEventCreate(&e0);
    if (e != cudaSuccess) return e;
    if ((e = cudaEventCreate(&e1)) != cudaSuccess) {
        cudaEventDestroy(e0);
        return e;
    }
    float ms = 0.f;
    philox_rate_kernel<<<blocks, kRateThreads, 0, s>>>(static_cast<uint32_t *>(sink), 8, K);  // warm-up
    e = cudaEventRecord(e0, s);
    if (e == cudaSuccess) {
        philox_rate_kernel<<<blocks, kRateThreads, 0, s>>>(static_cast<uint32_t *>(sink), iters, K);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaEventRecord(e1, s);
    if (e == cudaSuccess) e = cudaEventSynchronize(e1);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (e != cudaSuccess) return e;
    *blocks_per_s = (double)blocks * kRateThreads * (double)iters * 4.0 / ((double)ms * 1e-3);
    return cudaSuccess;
}

cudaError_t run_bounded_wait_probe(unsigned int limit_us, uint32_t *result, cudaStream_t s) {
    int dev = 0, khz = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev);
    if (e != cudaSuccess) return e;
    const uint32_t zero = 0u, unset = 0xFFFFFFFFu;
    if ((e = cudaMemcpyToSymbolAsync(g_selftest_counter, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s)) !=
        cudaSuccess)
        return e;
    if ((e = cudaMemcpyToSymbolAsync(g_selftest_result, &unset, sizeof(unset), 0, cudaMemcpyHostToDevice, s)) !=
        cudaSuccess)
        return e;
    const long long limit_cycles = (long long)limit_us * (long long)(khz > 0 ? khz : 2000000) / 1000;
    bounded_wait_probe_kernel<<<1, 32, 0, s>>>(limit_cycles);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = cudaMemcpyFromSymbolAsync(result, g_selftest_result, sizeof(uint32_t), 0, cudaMemcpyDeviceToHost, s)) !=
        cudaSuccess)
        return e;
    return cudaStreamSynchronize(s);
}

}  // namespace dspark

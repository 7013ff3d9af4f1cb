// Self-test of the bounded waits every kernel of the library relies on.
//
// One block waits, with the production helpers and a short limit, on an
// mbarrier phase that no thread completes and on a global counter that no
// thread increments.  Both must give up and report it; the context stays
// usable (nothing faults, traps or spins without a limit).
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

}  // namespace

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

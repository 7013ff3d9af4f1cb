// Packing the target rows that verification reads.
//
// "DSpark, la bozza che sa quando fermarsi" (paithon.it), section "Verificare
// meglio, non di piu'": the verify lengths L_b chosen by the scheduler size the
// target's batch, sum_b (L_b + 1) rows.  dspark_pack_target gathers rows
// 0 .. L_b of every request from a dense [B][G+1][V] target, which may live in
// device memory or in pinned host memory mapped into the device's address
// space (the gather then moves exactly the rows verification reads across the
// host link), into the packed layout of dspark_verify_packed.
//
// Two launches, both driven by the device-side verify lengths (no host round
// trip): a one-block scan writes each request's first packed row and the row
// count, then one block per (request, row) copies the rows with 16-byte loads.
#include "device_common.cuh"
#include "internal.h"

namespace dspark {
namespace {

constexpr int kScanThreads = 1024;
constexpr int kCopyThreads = 256;

// rows a request contributes: 0 .. L_b, none for an invalid length (the
// verification flags it and reads no row of it)
__device__ __forceinline__ int packed_rows(const int32_t *verify_len, int b, int G) {
    const int L = verify_len ? verify_len[b] : G;
    return (L < 0 || L > G) ? 0 : L + 1;
}

__global__ void __launch_bounds__(kScanThreads)
pack_scan_kernel(const int32_t *__restrict__ verify_len, int B, int G, int64_t *__restrict__ row0,
                 int64_t *__restrict__ n_rows) {
    __shared__ int64_t warp_sum[kScanThreads / 32];
    __shared__ int64_t carry;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < B; base += kScanThreads) {
        const int b = base + threadIdx.x;
        const int64_t x = (b < B) ? packed_rows(verify_len, b, G) : 0;
        // inclusive scan within the warp, then across the warps
        int64_t v = x;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, v, d);
            if (lane >= d) v += y;
        }
        if (lane == 31) warp_sum[warp] = v;
        __syncthreads();
        if (warp == 0) {
            int64_t w = warp_sum[lane];
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int64_t y = __shfl_up_sync(0xffffffffu, w, d);
                if (lane >= d) w += y;
            }
            warp_sum[lane] = w;  // inclusive over warps
        }
        __syncthreads();
        const int64_t before = carry + (warp > 0 ? warp_sum[warp - 1] : 0) + (v - x);
        if (b < B) row0[b] = before;
        __syncthreads();
        if (threadIdx.x == kScanThreads - 1) carry = before + x;
        __syncthreads();
    }
    if (threadIdx.x == 0 && n_rows) *n_rows = carry;
}

// one block per (request, row slot): copies row j of request b when j <= L_b
// (requests along x: their count may pass the 65535 limit of y)
__global__ void __launch_bounds__(kCopyThreads)
pack_copy_kernel(const unsigned char *__restrict__ src, const int32_t *__restrict__ verify_len,
                 const int64_t *__restrict__ row0, int G, size_t row_bytes, unsigned char *__restrict__ dst) {
    const int b = blockIdx.x, j = blockIdx.y;
    if (j >= packed_rows(verify_len, b, G)) return;
    const uint4 *s = reinterpret_cast<const uint4 *>(src + ((size_t)b * (G + 1) + j) * row_bytes);
    uint4 *d = reinterpret_cast<uint4 *>(dst + (size_t)(row0[b] + j) * row_bytes);
    const size_t n = row_bytes / 16;
    size_t i = threadIdx.x;
    for (; i + 3 * kCopyThreads < n; i += 4 * kCopyThreads) {  // four loads in flight
        const uint4 a0 = s[i], a1 = s[i + kCopyThreads], a2 = s[i + 2 * kCopyThreads], a3 = s[i + 3 * kCopyThreads];
        d[i] = a0;
        d[i + kCopyThreads] = a1;
        d[i + 2 * kCopyThreads] = a2;
        d[i + 3 * kCopyThreads] = a3;
    }
    for (; i < n; i += kCopyThreads) d[i] = s[i];
}

}  // namespace

cudaError_t launch_pack_target(const void *src, const int32_t *verify_len, int B, int G, int V, size_t elem_bytes,
                               void *dst, int64_t *row0, int64_t *n_rows, cudaStream_t s) {
    pack_scan_kernel<<<1, kScanThreads, 0, s>>>(verify_len, B, G, row0, n_rows);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    pack_copy_kernel<<<dim3(B, G + 1), kCopyThreads, 0, s>>>(static_cast<const unsigned char *>(src), verify_len,
                                                             row0, G, (size_t)V * elem_bytes,
                                                             static_cast<unsigned char *>(dst));
    return cudaGetLastError();
}

}  // namespace dspark

// dspark_verify_noalloc: the verification entry point for callers that cannot
// allocate device memory.
//
// Some callers have no way to hand the library a scratch buffer: an inference
// runtime whose device memory is planned up front and handed out only to
// tensors, a plugin invoked from inside another framework's execution context
// where cudaMalloc is not allowed, or a foreign-function caller with no
// allocator binding at all.  For them this entry point runs the same kernels
// as dspark_verify with the scratch memory taken from a fixed array that lives
// in this library's device image.
//
// The array is a file-scope __device__ variable of kNoAllocScratchBytes; every
// GPU that loads the library holds it until the process exits.  In host code
// its name is only a host-side stand-in, so its device address is looked up
// once per device with cudaGetSymbolAddress (on the first call on that device,
// with that device current) and cached for the life of the process (a
// cudaDeviceReset invalidates it).  Make that first call before any stream
// capture begins.  All calls share the array and it keeps the previous
// call's contents: the flag word is cleared on every call, and two calls whose
// work overlaps on the GPU (different streams, or different host threads
// without ordering) race on it.  Requests whose verify workspace would exceed
// the array are rejected with DSPARK_ERR_UNSUPPORTED.  Nothing here calls
// cudaMalloc, cudaFree or any allocating routine.
#include <cstdio>
#include <mutex>

#include "internal.h"

namespace dspark {
namespace {

constexpr size_t kNoAllocScratchBytes = DSPARK_NOALLOC_SCRATCH_BYTES;  // 4 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_verify_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (set-up on first use).
cudaError_t scratch_address(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_verify_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace dspark

using namespace dspark;

extern "C" {

dspark_status dspark_verify_noalloc(
    const void *target_logits, const void *base_logits, const void *e_in, const void *w_out,
    const float *draft_logits, const int32_t *anchor, const int32_t *draft_tokens,
    const float *draft_lse, const float *draft_logq, const int32_t *verify_len,
    const float *temperature, const uint32_t *request_id, int B, int G, int V, int r,
    dspark_dtype dtype, uint64_t seed, int32_t *accept_len, int32_t *out_tokens, int32_t *num_out,
    float *target_lse, float *logp_sel, void *stream) {
    // the argument errors dspark_verify would report come first
    const dspark_status st = verify_check_args(target_logits, base_logits, e_in, w_out, draft_logits, anchor,
                                               draft_tokens, draft_lse, draft_logq, temperature, B, G, V, r, dtype,
                                               accept_len, out_tokens, num_out);
    if (st != DSPARK_OK) return st;
    const size_t need = plan_verify(B, G, V, r, dtype).ws_bytes;
    if (need > kNoAllocScratchBytes)
        return set_last_error(DSPARK_ERR_UNSUPPORTED,
                              "verify needs %zu bytes of scratch, more than the fixed %zu-byte array",
                              need, kNoAllocScratchBytes);
    void *scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess)
        return set_last_error(DSPARK_ERR_CUDA, "cudaGetSymbolAddress of the scratch array: %s",
                              cudaGetErrorString(e));
    // dspark_verify clears the flag word at the head of the scratch and
    // launches the same kernels as with a caller-owned workspace.
    return dspark_verify(target_logits, base_logits, e_in, w_out, draft_logits, anchor, draft_tokens,
                         draft_lse, draft_logq, verify_len, temperature, request_id, B, G, V, r, dtype,
                         seed, accept_len, out_tokens, num_out, target_lse, logp_sel, scratch, need,
                         stream);
}

dspark_status dspark_read_noalloc_flags(void *stream, uint32_t *flags) {
    if (!flags) return set_last_error(DSPARK_ERR_INVALID_ARG, "flags is NULL");
    void *scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e == cudaSuccess) return dspark_read_device_flags(scratch, stream, flags);
    return set_last_error(DSPARK_ERR_CUDA, "cudaGetSymbolAddress of the scratch array: %s", cudaGetErrorString(e));
}

}  // extern "C"

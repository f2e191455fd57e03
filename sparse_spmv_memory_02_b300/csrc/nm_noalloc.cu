// nm_pack_noalloc: the pack entry point for callers that must not allocate
// device memory.
//
// nm_pack needs four bytes of scratch (the count of groups whose mask does
// not keep exactly N) and obtains them with cudaMallocAsync.  Some callers
// cannot let a library allocate: a serving engine that has reserved nearly
// all device memory up front for its own pools (a stray allocation fails or
// fragments them), a runtime whose memory budget is fixed before start-up,
// or code that must not risk the implicit device synchronisation an
// allocation or free can bring.  This variant runs the same pack kernel but
// counts into a fixed array compiled into the library instead.
//
// The scratch array lives in this file; its device address is looked up
// once per device (cudaGetSymbolAddress on the first call made with that
// device current) and cached, so the library must not be called on a device
// again after cudaDeviceReset.  The array is shared by every call on a
// device and keeps the last call's contents, so each call clears it first;
// two calls that overlap on the GPU (for example on two streams) race on it.
// Like nm_pack, the call synchronises its stream, so a capturing stream is
// refused.
#include <cuda_runtime.h>

#include <climits>
#include <cstdio>
#include <mutex>

#include "nm.h"
#include "nm_internal.h"

namespace {

// One 32-bit counter is used; the array is padded to 256 bytes.
constexpr int kScratchWords = NM_NOALLOC_SCRATCH_BYTES / 4;
static __device__ __align__(256) unsigned int g_noalloc_scratch[kScratchWords];

constexpr int kMaxDevices = 64;
unsigned int *g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mutex;

nm_status noalloc_fail(nm_status st, const char *msg)
{
    nm::set_last_error(msg);
    return st;
}

// Device address of the scratch array on the current device (set-up on first use).
cudaError_t scratch_for_current_device(unsigned int **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = static_cast<unsigned int *>(p);
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" nm_status nm_pack_noalloc(const void *W, const uint8_t *mask, int64_t rows, int64_t K,
                                     int N, int M, void *values, uint32_t *masks,
                                     nm_stream_t stream)
{
    nm::set_last_error("");
    if (M != 4 && M != 8) return noalloc_fail(NM_ERR_UNSUPPORTED, "M must be 4 or 8");
    if (N < 1 || N > M) return noalloc_fail(NM_ERR_UNSUPPORTED, "need 1 <= N <= M");
    if (rows < 0 || K < 0 || rows > INT_MAX || K > INT_MAX)
        return noalloc_fail(NM_ERR_INVALID_ARG, "rows and K must be in [0, INT_MAX]");
    if (K % M != 0) return noalloc_fail(NM_ERR_INVALID_ARG, "K must be a multiple of M");
    if (rows == 0 || K == 0) return NM_OK;
    if ((rows * (K / M)) > static_cast<int64_t>(NM_PACK_NOALLOC_MAX_GROUPS))
        return noalloc_fail(NM_ERR_INVALID_ARG,
                            "too many groups for the 32-bit scratch counter "
                            "(rows*K/M must be <= NM_PACK_NOALLOC_MAX_GROUPS)");
    if (!W || !mask || !values || !masks)
        return noalloc_fail(NM_ERR_INVALID_ARG, "W, mask, values and masks must be non-NULL");
    if (reinterpret_cast<uintptr_t>(W) % 2 != 0)
        return noalloc_fail(NM_ERR_INVALID_ARG, "W must be 2-byte aligned");
    if (reinterpret_cast<uintptr_t>(values) % 16 != 0 ||
        reinterpret_cast<uintptr_t>(masks) % 16 != 0)
        return noalloc_fail(NM_ERR_INVALID_ARG, "values and masks must be 16-byte aligned");

    // The call synchronises its stream to read the counter back, which a
    // capturing stream forbids: refuse it before any work is queued, so the
    // caller's capture stays valid.
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cap);
    if (e != cudaSuccess) return noalloc_fail(NM_ERR_CUDA, cudaGetErrorString(e));
    if (cap != cudaStreamCaptureStatusNone)
        return noalloc_fail(NM_ERR_INVALID_ARG,
                            "nm_pack_noalloc synchronises its stream and cannot be captured");

    unsigned int *d_bad = nullptr;
    e = scratch_for_current_device(&d_bad);
    if (e != cudaSuccess) return noalloc_fail(NM_ERR_CUDA, cudaGetErrorString(e));
    unsigned int h_bad = 0;
    e = cudaMemsetAsync(d_bad, 0, sizeof(unsigned int), s);
    if (e == cudaSuccess)
        e = nm::launch_pack(static_cast<const uint16_t *>(W), mask, rows, K, N, M,
                            static_cast<uint16_t *>(values), masks, d_bad, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(&h_bad, d_bad, sizeof(unsigned int), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return noalloc_fail(NM_ERR_CUDA, cudaGetErrorString(e));
    if (h_bad != 0) {
        char msg[128];
        snprintf(msg, sizeof(msg), "%u group(s) do not keep exactly N=%d of M=%d", h_bad, N, M);
        return noalloc_fail(NM_ERR_BAD_MASK, msg);
    }
    return NM_OK;
}

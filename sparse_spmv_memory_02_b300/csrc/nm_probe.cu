// Read-only HBM stream (include/nm_probe.h): the rate the SpMV kernels'
// weight stream is measured against.  One CTA of 1024 threads per SM; each
// thread keeps four independent 16-byte loads in flight and folds what it
// read into one word.
#include <cuda_runtime.h>

#include <cstdio>

#include "nm.h"
#include "nm_device.cuh"
#include "nm_internal.h"
#include "nm_probe.h"

namespace nm {
namespace {

constexpr int kProbeThreads = 1024;

__global__ void __launch_bounds__(kProbeThreads)
nm_probe_read_kernel(const uint4 *buf, size_t n16, uint32_t *sink)
{
    // Thread t reads units t, t + T, t + 2T, t + 3T of each block of 4T
    // units (T threads in the grid): every warp-wide load is 512 contiguous
    // bytes and each thread has four loads in flight.
    uint32_t acc = 0;
    const size_t T = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t base = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; base < n16;
         base += 4 * T) {
        uint4 v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const size_t idx = base + q * T;
            v[q] = idx < n16 ? ld_stream_v4(buf + idx) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) acc ^= v[q].x ^ v[q].y ^ v[q].z ^ v[q].w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
    if ((threadIdx.x & 31) == 0) atomicXor(sink, acc);
}

}  // namespace
}  // namespace nm

extern "C" nm_status nm_probe_read_stream(const void *buf, size_t bytes, uint32_t *sink,
                                          nm_stream_t stream)
{
    nm::set_last_error("");
    if (bytes == 0) return NM_OK;
    if (!buf || !sink) {
        nm::set_last_error("buf and sink must be non-NULL");
        return NM_ERR_INVALID_ARG;
    }
    if (reinterpret_cast<uintptr_t>(buf) % 16 != 0 || reinterpret_cast<uintptr_t>(sink) % 4 != 0 ||
        bytes % 16 != 0) {
        nm::set_last_error("buf must be 16-byte aligned, sink 4-byte aligned, bytes a multiple of 16");
        return NM_ERR_INVALID_ARG;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int nsm = nm::sm_count();
    if (nsm <= 0) {
        nm::set_last_error("no CUDA device");
        return NM_ERR_CUDA;
    }
    cudaError_t e = cudaMemsetAsync(sink, 0, sizeof(uint32_t), s);
    if (e == cudaSuccess) {
        nm::nm_probe_read_kernel<<<nsm, nm::kProbeThreads, 0, s>>>(
            static_cast<const uint4 *>(buf), bytes / 16, sink);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof(msg), "nm_probe_read_stream: %s", cudaGetErrorString(e));
        nm::set_last_error(msg);
        return NM_ERR_CUDA;
    }
    return NM_OK;
}

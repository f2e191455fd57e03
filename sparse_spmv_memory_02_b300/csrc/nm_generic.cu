// Scalar N:M kernels: SpMV for every valid pattern and K (the vectorised
// kernel needs 8 % N == 0 and K a multiple of its chunk span), and the
// pack / unpack kernels that produce and invert the packed layout.
//
// Layout (bitmask indexing with fixed-step traversal, "SparseDecoding:
// Decoding-Aware Pruning for Accurate and Efficient LLM Inference",
// Abstract): bit k%32 of mask word k/32 of a row is the keep bit of position
// k; the N kept values of group g sit at values[row][g*N .. g*N+N-1] in
// increasing k.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "nm_device.cuh"
#include "nm_internal.h"

namespace nm {

int sm_count()
{
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (dev >= 0 && dev < 64) {
        int v = cache[dev].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    if (dev >= 0 && dev < 64) cache[dev].store(v, std::memory_order_relaxed);
    return v;
}

// ---------------------------------------------------------------- SpMV

struct GenericArgs {
    const uint16_t *values;
    const uint32_t *masks;
    const __half *x;
    void *y;
    int64_t rows, K, ldx, ldy;
    int N, M;
    int y_f32;
};

// One warp per row; lane l walks groups l, l+32, ...: it reads the group's M
// mask bits, and for the j-th set bit the value at g*N + j.
template <int B>
__global__ void __launch_bounds__(256) nm_spmv_generic_kernel(const GenericArgs a)
{
    const int warps = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t groups = a.K / a.M;
    const int64_t Lv = groups * a.N;
    const int64_t Wm = (a.K + 31) / 32;
    const uint32_t full = (1u << a.M) - 1u;
    for (int64_t row = static_cast<int64_t>(blockIdx.x) * warps + warp; row < a.rows;
         row += static_cast<int64_t>(gridDim.x) * warps) {
        float acc[B];
#pragma unroll
        for (int b = 0; b < B; ++b) acc[b] = 0.f;
        for (int64_t g = lane; g < groups; g += 32) {
            const int64_t k0 = g * a.M;
            const uint32_t bits = (a.masks[row * Wm + k0 / 32] >> (k0 % 32)) & full;
            const uint16_t *vg = a.values + row * Lv + g * a.N;
            int j = 0;
            for (int q = 0; q < a.M; ++q) {
                if (((bits >> q) & 1u) && j < a.N) {
                    const float w = __half2float(__ushort_as_half(vg[j]));
                    ++j;
#pragma unroll
                    for (int b = 0; b < B; ++b)
                        acc[b] = fmaf(w, __half2float(a.x[b * a.ldx + k0 + q]), acc[b]);
                }
            }
        }
#pragma unroll
        for (int b = 0; b < B; ++b) {
            float v = acc[b];
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) store_y(a.y, b * a.ldy + row, v, a.y_f32 != 0);
        }
    }
}

template <int B>
static cudaError_t launch_generic_b(const GenericArgs &a, cudaStream_t s)
{
    const int threads = 256;
    const int nsm = sm_count();
    if (nsm <= 0) return cudaErrorInvalidDevice;
    const int64_t warps_needed = a.rows;
    int64_t grid = (warps_needed + 7) / 8;
    const int64_t cap = static_cast<int64_t>(nsm) * 8;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    nm_spmv_generic_kernel<B><<<static_cast<int>(grid), threads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_generic(const SpmvProblem &p, cudaStream_t s)
{
    GenericArgs a;
    a.values = static_cast<const uint16_t *>(p.values);
    a.masks = p.masks;
    a.x = static_cast<const __half *>(p.x);
    a.y = p.y;
    a.rows = p.rows;
    a.K = p.K;
    a.ldx = p.ldx;
    a.ldy = p.ldy;
    a.N = p.N;
    a.M = p.M;
    a.y_f32 = p.y_f32 ? 1 : 0;
    switch (p.batch) {
    case 1: return launch_generic_b<1>(a, s);
    case 2: return launch_generic_b<2>(a, s);
    case 3: return launch_generic_b<3>(a, s);
    case 4: return launch_generic_b<4>(a, s);
    case 5: return launch_generic_b<5>(a, s);
    case 6: return launch_generic_b<6>(a, s);
    case 7: return launch_generic_b<7>(a, s);
    case 8: return launch_generic_b<8>(a, s);
    default: return cudaErrorInvalidValue;
    }
}

// ---------------------------------------------------------------- pack

// One thread per (row, mask word): the word's 32/M groups (fewer in the last
// word of a row when K % 32 != 0).  Kept fp16 bit patterns are copied in
// increasing k to the group's N slots; a group with fewer than N set bits
// gets +0.0 in its missing slots, and any group without exactly N set bits
// is counted in *bad.
__global__ void __launch_bounds__(256)
nm_pack_kernel(const uint16_t *__restrict__ W, const uint8_t *__restrict__ mask, int64_t rows,
               int64_t K, int N, int M, uint16_t *__restrict__ values,
               uint32_t *__restrict__ masks, unsigned int *__restrict__ bad)
{
    const int64_t Wm = (K + 31) / 32;
    const int64_t total = rows * Wm;
    const int64_t Lv = (K / M) * N;
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
         t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = t / Wm;
        const int64_t w = t - r * Wm;
        const int64_t k0 = w * 32;
        const int64_t kend = (k0 + 32 < K) ? k0 + 32 : K;
        uint32_t word = 0;
        unsigned int nbad = 0;
        for (int64_t gk = k0; gk < kend; gk += M) {
            uint16_t *vg = values + r * Lv + (gk / M) * N;
            int kept = 0;
            for (int q = 0; q < M; ++q) {
                const int64_t k = gk + q;
                if (mask[r * K + k] != 0) {
                    word |= 1u << (k - k0);
                    if (kept < N) vg[kept] = W[r * K + k];
                    ++kept;
                }
            }
            for (int j = kept; j < N; ++j) vg[j] = 0;
            nbad += (kept != N) ? 1u : 0u;
        }
        masks[r * Wm + w] = word;
        if (nbad) atomicAdd(bad, nbad);
    }
}

// Inverse: dropped positions become +0.0; the j-th set bit of a group takes
// value j (at most N per group).
__global__ void __launch_bounds__(256)
nm_unpack_kernel(const uint16_t *__restrict__ values, const uint32_t *__restrict__ masks,
                 int64_t rows, int64_t K, int N, int M, uint16_t *__restrict__ W)
{
    const int64_t Wm = (K + 31) / 32;
    const int64_t total = rows * Wm;
    const int64_t Lv = (K / M) * N;
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
         t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = t / Wm;
        const int64_t w = t - r * Wm;
        const int64_t k0 = w * 32;
        const int64_t kend = (k0 + 32 < K) ? k0 + 32 : K;
        const uint32_t word = masks[r * Wm + w];
        for (int64_t gk = k0; gk < kend; gk += M) {
            const uint16_t *vg = values + r * Lv + (gk / M) * N;
            int j = 0;
            for (int q = 0; q < M; ++q) {
                const int64_t k = gk + q;
                if (((word >> (k - k0)) & 1u) && j < N) {
                    W[r * K + k] = vg[j];
                    ++j;
                } else {
                    W[r * K + k] = 0;
                }
            }
        }
    }
}

static int64_t grid_for(int64_t work, int threads)
{
    const int nsm = sm_count();
    int64_t grid = (work + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(nsm > 0 ? nsm : 148) * 16;
    if (grid > cap) grid = cap;
    return grid < 1 ? 1 : grid;
}

cudaError_t launch_pack(const uint16_t *W, const uint8_t *mask, int64_t rows, int64_t K, int N,
                        int M, uint16_t *values, uint32_t *masks, unsigned int *bad,
                        cudaStream_t s)
{
    const int64_t work = rows * ((K + 31) / 32);
    nm_pack_kernel<<<static_cast<int>(grid_for(work, 256)), 256, 0, s>>>(W, mask, rows, K, N, M,
                                                                         values, masks, bad);
    return cudaGetLastError();
}

cudaError_t launch_unpack(const uint16_t *values, const uint32_t *masks, int64_t rows, int64_t K,
                          int N, int M, uint16_t *W, cudaStream_t s)
{
    const int64_t work = rows * ((K + 31) / 32);
    nm_unpack_kernel<<<static_cast<int>(grid_for(work, 256)), 256, 0, s>>>(values, masks, rows, K,
                                                                           N, M, W);
    return cudaGetLastError();
}

}  // namespace nm

// N:M mask selection from scores, and selection fused with packing.
//
// The step before nm_pack in a pruning flow: in every group of M consecutive
// weights along K keep the N of largest score, where the score of weight
// (r, k) is |w| (magnitude pruning) or |w| * scale[k] with a per-input-channel
// scale such as the norm of input feature k over calibration activations
// (the importance measure of the Wanda family of training-free pruning
// methods, which the bedrocknews summary of arXiv 2610.12327v1 names as the
// baseline SparseDecoding improves on: weight magnitude weighted by
// activation statistics).  The pages do not fix the score; these are the
// two plain readings.
//
// Rule (shared with the oracle): position q of a group is kept iff fewer
// than N positions beat it, q' beating q when s(q') > s(q), or s(q') == s(q)
// and q' < q.  Without NaN scores exactly N positions are kept.  Scores are
// fp32: |w| converted exactly from fp16, times scale[k] rounded to nearest.
//
// Both kernels are plain streams (2 bytes of W read per weight; 1 byte of
// mask, or the packed bytes, written): one thread per group (selection) or
// per 32-position mask word (fused), with aligned vector loads of W and of
// the scales.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "nm_device.cuh"
#include "nm_internal.h"

namespace nm {

namespace {

template <int M> struct GroupVec;
template <> struct GroupVec<4> { using type = uint2; };  // 4 fp16
template <> struct GroupVec<8> { using type = uint4; };  // 8 fp16

// Scores of one group of M weights (fp16 bits in `w`) starting at column k.
template <int M>
__device__ __forceinline__ void group_scores(const typename GroupVec<M>::type &w,
                                             const float *__restrict__ scale, int64_t k,
                                             float (&s)[M])
{
    const uint32_t *wv = reinterpret_cast<const uint32_t *>(&w);
#pragma unroll
    for (int q = 0; q < M; ++q) {
        const uint16_t bits = static_cast<uint16_t>(wv[q / 2] >> (16 * (q & 1)));
        s[q] = fabsf(__half2float(__ushort_as_half(bits)));
    }
    if (scale) {
        float f[M];
        if constexpr (M == 4) {
            const float4 a = *reinterpret_cast<const float4 *>(scale + k);
            f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        } else {
            const float4 a = *reinterpret_cast<const float4 *>(scale + k);
            const float4 b = *reinterpret_cast<const float4 *>(scale + k + 4);
            f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
            f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
        }
#pragma unroll
        for (int q = 0; q < M; ++q) s[q] = __fmul_rn(s[q], f[q]);
    }
}

// Bit q set iff position q is kept (fewer than N positions beat it).
template <int M>
__device__ __forceinline__ uint32_t group_keep(const float (&s)[M], int N)
{
    uint32_t keep = 0;
#pragma unroll
    for (int q = 0; q < M; ++q) {
        int beaten = 0;
#pragma unroll
        for (int q2 = 0; q2 < M; ++q2)
            if (q2 != q) beaten += (s[q2] > s[q] || (s[q2] == s[q] && q2 < q)) ? 1 : 0;
        keep |= (beaten < N ? 1u : 0u) << q;
    }
    return keep;
}

// Each thread takes kU = 32 / M groups per sweep (group indices t,
// t + stride, ..., so that for every u the warp's loads are consecutive),
// issuing all of their loads before the first selection: 64 bytes of W in
// flight per thread.
template <int M> constexpr int kGroupsPerSweep = 32 / M;

// (row, group) of a flat group index, advanced by a fixed stride without a
// 64-bit division per step (the stride's own row/group split is taken once).
struct RowPos {
    int64_t r, g;
};
__device__ __forceinline__ void advance(RowPos &p, int64_t rs, int64_t gs, int64_t per_row)
{
    p.g += gs;
    p.r += rs;
    if (p.g >= per_row) {
        p.g -= per_row;
        ++p.r;
    }
}

template <int M>
__device__ __forceinline__ void store_group_mask(uint8_t *dst, uint32_t keep)
{
    // byte q = bit q of keep
    const uint32_t lo = (keep & 1u) | ((keep & 2u) << 7) | ((keep & 4u) << 14) | ((keep & 8u) << 21);
    if constexpr (M == 4) {
        *reinterpret_cast<uint32_t *>(dst) = lo;
    } else {
        const uint32_t h = keep >> 4;
        const uint32_t hi = (h & 1u) | ((h & 2u) << 7) | ((h & 4u) << 14) | ((h & 8u) << 21);
        *reinterpret_cast<uint2 *>(dst) = make_uint2(lo, hi);
    }
}

template <int M>
__global__ void __launch_bounds__(256)
nm_select_kernel(const uint16_t *__restrict__ W, const float *__restrict__ scale, int64_t rows,
                 int64_t K, int N, uint8_t *__restrict__ mask)
{
    using V = typename GroupVec<M>::type;
    constexpr int kU = kGroupsPerSweep<M>;
    const int64_t gpr = K / M;  // groups per row
    const int64_t total = rows * gpr;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t rs = stride / gpr, gs = stride - (stride / gpr) * gpr;
    const int64_t tfirst = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    RowPos pos = {tfirst / gpr, tfirst - (tfirst / gpr) * gpr};
    for (int64_t t0 = tfirst; t0 < total; t0 += kU * stride) {
        V w[kU];
        int64_t k[kU];  // column of each group (for its scales)
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t t = t0 + u * stride;
            k[u] = pos.g * M;
            advance(pos, rs, gs, gpr);
            if (t < total) w[u] = *reinterpret_cast<const V *>(W + t * M);  // group t at t*M
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t t = t0 + u * stride;
            if (t < total) {
                float s[M];
                group_scores<M>(w[u], scale, k[u], s);
                store_group_mask<M>(mask + t * M, group_keep<M>(s, N));
            }
        }
    }
}

// Fused selection and packing.  Thread t handles one group of a row whose
// groups are counted in whole mask words (gpad = ceil(K/32) * 32/M slots a
// row, slots past K/M idle), so the 32/M lanes of one mask word are adjacent
// and aligned in the warp: they OR their keep bits together with shuffles
// and the first of them writes the word, while each writes its N kept
// values next to its neighbours'.
template <int M>
__global__ void __launch_bounds__(256)
nm_prune_pack_kernel(const uint16_t *__restrict__ W, const float *__restrict__ scale,
                     int64_t rows, int64_t K, int N, uint16_t *__restrict__ values,
                     uint32_t *__restrict__ masks)
{
    using V = typename GroupVec<M>::type;
    constexpr int kU = kGroupsPerSweep<M>;
    constexpr int GW = 32 / M;  // groups per mask word (lanes per word)
    const int64_t gpr = K / M;
    const int64_t Wm = (K + 31) / 32;
    const int64_t gpad = Wm * GW;
    const int64_t total = rows * gpad;  // a multiple of GW
    const int64_t Lv = gpr * N;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;  // a multiple of 32
    const int lane = threadIdx.x & 31;
    // the sweep's trip count is the same for all lanes of a warp (warps
    // start at multiples of 32 and total is a multiple of GW): the
    // shuffles below see whole segments
    const int64_t rs = stride / gpad, gs = stride - (stride / gpad) * gpad;
    const int64_t tfirst = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    RowPos pos = {tfirst / gpad, tfirst - (tfirst / gpad) * gpad};
    for (int64_t t0 = tfirst; t0 - lane < total; t0 += kU * stride) {
        V w[kU];
        RowPos at[kU];
        bool live[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t t = t0 + u * stride;
            at[u] = pos;
            advance(pos, rs, gs, gpad);
            live[u] = t < total && at[u].g < gpr;
            if (live[u]) w[u] = *reinterpret_cast<const V *>(W + at[u].r * K + at[u].g * M);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t t = t0 + u * stride;
            const int64_t r = at[u].r;
            const int64_t g = at[u].g;
            uint32_t keep = 0;
            if (live[u]) {
                float s[M];
                group_scores<M>(w[u], scale, g * M, s);
                keep = group_keep<M>(s, N);
                // the first N kept values, in increasing k, packed into
                // lo (slots 0-3) and hi (slots 4-7); slots past the kept
                // ones stay +0.0 (only with NaN scores)
                const uint32_t *wv = reinterpret_cast<const uint32_t *>(&w[u]);
                uint64_t lo = 0, hi = 0;
                int kept = 0;
#pragma unroll
                for (int q = 0; q < M; ++q) {
                    if (((keep >> q) & 1u) && kept < N) {
                        const uint64_t v = (wv[q / 2] >> (16 * (q & 1))) & 0xFFFFu;
                        if (kept < 4) lo |= v << (16 * kept);
                        else hi |= v << (16 * (kept - 4));
                        ++kept;
                    }
                }
                uint16_t *vout = values + r * Lv + g * N;  // aligned to 2N bytes for N = 1, 2, 4, 8
                if (N == 2) {
                    *reinterpret_cast<uint32_t *>(vout) = static_cast<uint32_t>(lo);
                } else if (N == 4) {
                    *reinterpret_cast<uint2 *>(vout) =
                        make_uint2(static_cast<uint32_t>(lo), static_cast<uint32_t>(lo >> 32));
                } else if (N == 8) {
                    *reinterpret_cast<uint4 *>(vout) =
                        make_uint4(static_cast<uint32_t>(lo), static_cast<uint32_t>(lo >> 32),
                                   static_cast<uint32_t>(hi), static_cast<uint32_t>(hi >> 32));
                } else {
                    for (int j = 0; j < N; ++j)
                        vout[j] = static_cast<uint16_t>(j < 4 ? lo >> (16 * j) : hi >> (16 * (j - 4)));
                }
            }
            // mask word of the segment: group j of the word owns bits j*M..
            uint32_t word = keep << ((lane % GW) * M);
#pragma unroll
            for (int o = 1; o < GW; o <<= 1) word |= __shfl_xor_sync(0xffffffffu, word, o);
            if (t < total && lane % GW == 0) masks[r * Wm + g / GW] = word;
        }
    }
}

int64_t select_grid(int64_t work)
{
    const int64_t want = (work + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sm_count() > 0 ? sm_count() : 148) * 8;
    return want < 1 ? 1 : (want < cap ? want : cap);
}

}  // namespace

cudaError_t launch_select(const uint16_t *W, const float *scale, int64_t rows, int64_t K, int N,
                          int M, uint8_t *mask, cudaStream_t s)
{
    const int64_t work = rows * (K / M);
    const int grid = static_cast<int>(select_grid(work));
    if (M == 4)
        nm_select_kernel<4><<<grid, 256, 0, s>>>(W, scale, rows, K, N, mask);
    else
        nm_select_kernel<8><<<grid, 256, 0, s>>>(W, scale, rows, K, N, mask);
    return cudaGetLastError();
}

// Empty kernel: a stream-ordered boundary that a programmatic dependent
// launch after it cannot cross (see launch_prune_pack).
__global__ void nm_stream_fence_kernel() {}

cudaError_t launch_prune_pack(const uint16_t *W, const float *scale, int64_t rows, int64_t K,
                              int N, int M, uint16_t *values, uint32_t *masks, cudaStream_t s)
{
    const int64_t work = rows * ((K + 31) / 32);
    const int grid = static_cast<int>(select_grid(work));
    if (M == 4)
        nm_prune_pack_kernel<4><<<grid, 256, 0, s>>>(W, scale, rows, K, N, values, masks);
    else
        nm_prune_pack_kernel<8><<<grid, 256, 0, s>>>(W, scale, rows, K, N, values, masks);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // The packed arrays just written are what an SpMV launched next on this
    // stream reads, and the SpMV kernels start copying weights before their
    // dependence wait (programmatic dependent launch).  An ordinary launch
    // between the two starts only once the pack has completed and its writes
    // are visible, and the SpMV can overlap only that launch.
    nm_stream_fence_kernel<<<1, 32, 0, s>>>();
    return cudaGetLastError();
}

}  // namespace nm

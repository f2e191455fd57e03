// Decode-only calibration accumulation H += X^T X on the fifth-generation
// tensor cores (tcgen05), for sm_103a.
//
// SparseDecoding builds its pruning calibration matrices from the layer
// inputs X (tokens x features) collected while the dense model generates,
// with the prefill excluded ("SparseDecoding: Decoding-Aware Pruning for
// Accurate and Efficient LLM Inference", Abstract; "SparseDecoding Makes LLM
// Pruning Aware of Generation", the decoding-aware calibration paragraph):
// the Hessian-style matrix of a layer is the sum over generated tokens t of
// x_t x_t^T.  The caller feeds only decode-step activations; this kernel
// adds one batch of them, H[i][j] += sum_t X[t][i] X[t][j], in fp32.
//
// It is a dense contraction over tokens, so it runs on tcgen05.mma (fp16
// operands, fp32 accumulator in tensor memory):
//   * one CTA per 128 x 128 tile of H on or above the diagonal (H is
//     symmetric; the CTA also adds its tile's transpose below it); 4 warps;
//   * warp 0 lane 0 streams 64-token slabs of X with TMA: for the tile's
//     rows i0..i0+127 and columns j0..j0+127 the slab X[t0:t0+64][i0:i0+128]
//     (operand A) and X[t0:t0+64][j0:j0+128] (operand B), each as two
//     64-feature boxes with 128-byte swizzle, into a ring of stages;
//   * warp 1 lane 0 issues the MMAs, M = N = 128, K = 16 tokens each, with
//     both operands feature-major (the tokens are the contraction dimension
//     and X is token-major in memory) and commits each stage back to the
//     producer;
//   * all four warps read the accumulator out of tensor memory (warp w owns
//     lanes 32w..32w+31, i.e. rows i0+32w..), stage it in shared memory and
//     add it and its transpose into H with coalesced reductions
//     (red.global.add.f32), so each element of H is read-modified-written
//     once per call and never re-read by the kernel.
// Every mbarrier wait is bounded (nm_pipe.cuh): a stalled pipeline sets the
// error word, drains what it issued and releases its tensor memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "nm_internal.h"
#include "nm_pipe.cuh"

namespace nm {

namespace {

constexpr int kTile = 128;        // rows and columns of H per CTA
constexpr int kSlab = 64;         // tokens per stage
constexpr int kStages = 3;
constexpr int kHalfBytes = 64 * kSlab * 2;        // one 64-feature box: 8 KB
constexpr int kOperandBytes = 2 * kHalfBytes;     // 128 features: 16 KB
constexpr int kStageBytes = 2 * kOperandBytes;    // A and B: 32 KB
constexpr int kSmemBytes = 1024 + kStages * kStageBytes + 256;
constexpr int kTmemCols = 128;

struct CalibArgs {
    float *H;
    int64_t ldh;
    int K, T;
    int tiles_per_row;       // ceil(K / 128)
    uint32_t idesc;          // tcgen05 instruction descriptor
    uint64_t desc_hi;        // shared-memory descriptor without its address field
    unsigned int *err;
};

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` once every tcgen05.mma issued so far by this thread has
// completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns of this warp's 32 lanes of tensor memory.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void red_add(float *p, float v)
{
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

__global__ void __launch_bounds__(128, 2)
nm_calib_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CalibArgs a)
{
    extern __shared__ uint8_t calib_smem_raw[];
    // 128-byte swizzled tiles need 1024-byte aligned atoms
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(calib_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes);
    uint64_t *empty = full + kStages;
    uint64_t *acc_bar = empty + kStages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_bar + 1);
    volatile int *failed = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // H is symmetric: CTA b takes the b-th tile (ti, tj) with tj >= ti in
    // row-major order and also adds its transpose to tile (tj, ti).
    int ti = 0, rem = static_cast<int>(blockIdx.x);
    while (rem >= a.tiles_per_row - ti) {
        rem -= a.tiles_per_row - ti;
        ++ti;
    }
    const int tj = ti + rem;
    const int i0 = ti * kTile, j0 = tj * kTile;
    const int nslab = (a.T + kSlab - 1) / kSlab;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_bar, 1);
        *failed = 0;
        mbar_fence_init();
    }
    if (warp == 0) {  // the accumulator: 128 lanes x 128 fp32 columns
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------- TMA producer
        int issued = 0;
        for (int k = 0; k < nslab && !*failed; ++k) {
            const int s = k % kStages;
            if (k >= kStages && !mbar_wait(&empty[s], ((k / kStages) - 1) & 1)) {
                *failed = 1;
                atomicOr(a.err, kDevErrPipeTimeout);
                break;
            }
            uint8_t *st = smem + s * kStageBytes;
            mbar_arrive_expect_tx(&full[s], kStageBytes);
            const int t0 = k * kSlab;
            tma_load_2d(st, &tmx, i0, t0, &full[s]);
            tma_load_2d(st + kHalfBytes, &tmx, i0 + 64, t0, &full[s]);
            tma_load_2d(st + kOperandBytes, &tmx, j0, t0, &full[s]);
            tma_load_2d(st + kOperandBytes + kHalfBytes, &tmx, j0 + 64, t0, &full[s]);
            ++issued;
        }
        // copies still landing in this CTA's stages must finish before it exits
        for (int k = (issued > kStages ? issued - kStages : 0); k < issued; ++k)
            if (!mbar_wait(&full[k % kStages], (k / kStages) & 1)) break;
    } else if (warp == 1 && lane == 0) {
        // ---------------------------------------------- MMA issuer
        for (int k = 0; k < nslab; ++k) {
            const int s = k % kStages;
            if (*failed) break;
            if (!mbar_wait(&full[s], (k / kStages) & 1)) {
                *failed = 1;
                atomicOr(a.err, kDevErrPipeTimeout);
                break;
            }
            tc_fence_after();
            const uint32_t a_base = smem_addr(smem + s * kStageBytes);
            const uint32_t b_base = a_base + kOperandBytes;
#pragma unroll
            for (int kk = 0; kk < kSlab / 16; ++kk) {
                // 16 tokens = two 8-row swizzle atoms (1024 bytes each)
                const uint64_t ad = a.desc_hi | ((a_base + kk * 2048) >> 4);
                const uint64_t bd = a.desc_hi | ((b_base + kk * 2048) >> 4);
                mma_f16(tmem, ad, bd, a.idesc, (k | kk) != 0 ? 1u : 0u);
            }
            mma_commit(&empty[s]);  // the stage is free once these MMAs have read it
        }
        mma_commit(acc_bar);  // the accumulator is final once all MMAs complete
    }

    // -------------------------------------------------- epilogue (all warps)
    __syncwarp();
    // tcgen05.ld is warp-wide: the decision to read out must be uniform
    const bool ok = __all_sync(0xffffffffu, mbar_wait(acc_bar, 0)) != 0;
    if (!ok && lane == 0) atomicOr(a.err, kDevErrPipeTimeout);
    // the same decision in every warp: the staging below has CTA barriers
    const bool go = __syncthreads_and(ok && *failed == 0 && nslab > 0) != 0;
    tc_fence_after();
    if (go) {
        // The tile goes through shared memory (the stages are free: every
        // TMA load has landed and every MMA has read its operands), rows
        // padded to 129 floats, so that both H[i0 + r][j0 + c] and the
        // mirrored H[j0 + c][i0 + r] are added with coalesced reductions
        // (32 consecutive floats of H per warp instruction) and without bank
        // conflicts on either side.
        float *stg = reinterpret_cast<float *>(smem);
        constexpr int kPitch = kTile + 1;
        const int r = 32 * warp + lane;
#pragma unroll 1
        for (int c0 = 0; c0 < kTile; c0 += 32) {
            float v[32];
            tmem_ld32(tmem + (static_cast<uint32_t>(32 * warp) << 16) + c0, v);
#pragma unroll
            for (int q = 0; q < 32; ++q) stg[r * kPitch + c0 + q] = v[q];
        }
        __syncthreads();
        for (int rr = warp; rr < kTile && i0 + rr < a.K; rr += 4) {
            float *hp = a.H + static_cast<int64_t>(i0 + rr) * a.ldh + j0;
            for (int c = lane; c < kTile && j0 + c < a.K; c += 32) red_add(hp + c, stg[rr * kPitch + c]);
        }
        if (tj != ti) {
            for (int c = warp; c < kTile && j0 + c < a.K; c += 4) {
                float *hp = a.H + static_cast<int64_t>(j0 + c) * a.ldh + i0;
                for (int rr = lane; rr < kTile && i0 + rr < a.K; rr += 32)
                    red_add(hp + rr, stg[rr * kPitch + c]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda).
using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                 const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                 const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_tiled()
{
    static std::once_flag once;
    static EncodeTiled fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
    });
    return fn;
}

}  // namespace

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator, fp16 A
// and B, both MN-major (bits 15 and 16), N / 8 at bit 17, M / 16 at bit 24.
uint32_t calib_idesc()
{
    return (1u << 4) | (0u << 7) | (0u << 10) | (1u << 15) | (1u << 16) |
           (static_cast<uint32_t>(kTile >> 3) << 17) | (static_cast<uint32_t>(kTile >> 4) << 24);
}

// Shared-memory descriptor fields other than the start address, for an
// MN-major operand of 128-byte swizzled atoms (64 features x 8 tokens, 1024
// bytes): the next 64 features at `lbo` bytes (the second TMA box), the next
// 8 tokens at `sbo` bytes; version 1 (bit 46), layout 2 = 128-byte swizzle
// (bits 61-63).
uint64_t calib_desc_hi(uint32_t lbo, uint32_t sbo)
{
    return (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

cudaError_t launch_calib(const uint16_t *X, int64_t T, int64_t K, int64_t ldx, float *H,
                         int64_t ldh, unsigned int *err, uint32_t idesc, uint64_t desc_hi,
                         cudaStream_t s)
{
    EncodeTiled enc = encode_tiled();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap map;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(T)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldx) * 2};
    const cuuint32_t box[2] = {64, kSlab};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t *>(X), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    static std::atomic<int> smem_set{0};
    if (!smem_set.load(std::memory_order_relaxed)) {
        cudaError_t e = cudaFuncSetAttribute(nm_calib_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemBytes);
        if (e != cudaSuccess) return e;
        smem_set.store(1, std::memory_order_relaxed);
    }
    CalibArgs a;
    a.H = H;
    a.ldh = ldh;
    a.K = static_cast<int>(K);
    a.T = static_cast<int>(T);
    a.tiles_per_row = static_cast<int>((K + kTile - 1) / kTile);
    a.idesc = idesc;
    a.desc_hi = desc_hi;
    a.err = err;
    const int64_t tiles = static_cast<int64_t>(a.tiles_per_row) * (a.tiles_per_row + 1) / 2;
    if (tiles > 0x7fffffff) return cudaErrorInvalidValue;
    nm_calib_kernel<<<static_cast<unsigned int>(tiles), 128, kSmemBytes, s>>>(map, a);
    return cudaGetLastError();
}

}  // namespace nm

// 2:4 sparse x dense products for 2 to 32 vectors on the fifth-generation
// tensor cores (tcgen05), for sm_103a.  The library routes a 2:4 product
// here where that is faster than the CUDA-core row kernel (from batch 2-5 by
// layer size, takes_tensor_cores in nm_api.cu) and for every batch above 8.
//
// The same N:M product as the streaming kernels ("SparseDecoding:
// Decoding-Aware Pruning for Accurate and Efficient LLM Inference",
// Abstract: bitmask indexing, fixed-step traversal), for the regime where
// the batch makes the CUDA-core kernel instruction-bound (8 x B products and
// their x gathers per 16-byte chunk): the packed weights are still streamed
// from HBM exactly once and the tensor cores do the multiply.  Two kernels:
// nm_spmm_sp_kernel (the default, further below) takes the packed values as
// the sparse A operand of tcgen05.mma.sp; nm_spmm_tc_kernel (tuning key
// tc_sp=0, described here) expands each CTA's rows to dense fp16 in tensor
// memory first.
//
//   * One CTA per SM, rows split evenly over the CTAs (at most 256 rows a
//     CTA: two 128-row MMA tiles, the second possibly partial).
//   * Warp 16 lane 0 streams 128-position slabs by TMA into a ring of up to
//     16 stages: the CTA's rows' packed values (64 fp16 a row, 128-byte
//     swizzled), their mask words (4 a row) and x (the batch rows, 128-byte
//     swizzled, the MMA's B operand).
//   * Warps 0-15 expand the slab: every 2:4 group's value pair goes to its
//     two mask positions, zeros to the others (two byte permutes per group
//     with selectors from a 16-entry table), and the dense row is stored into
//     tensor memory (lane = row, two fp16 a column) as the MMA's A operand.
//     Warp 4h + q serves lanes 32q..32q+31; with two tiles h / 2 picks the
//     tile and h % 2 the half of the slab, with one tile h picks the quarter.
//   * Warps 17-20 (lane 0) issue tcgen05.mma (M = 128 per tile, N = the
//     batch padded to 16 or 32, K = 16 positions, A from tensor memory, fp32
//     accumulators in tensor memory), each a quarter of the slab's MMAs into
//     its own accumulator, and commit once a slab.
//   * Warps 0-15 read the accumulators (lane = row, column = vector) and
//     round them into y.
// Rows of a tile past the CTA's rows are never written: an MMA row depends
// on its own A row only, and those accumulator rows are not stored.
// Every mbarrier wait is bounded; a timeout sets the error word, the kernel
// drains what it issued, releases its tensor memory and returns.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "nm_bulk.cuh"  // bulk_tuning()
#include "nm_device.cuh"
#include "nm_internal.h"
#include "nm_pipe.cuh"
#include "nm_tc_expand.cuh"

namespace nm {

namespace {

constexpr int kSlabPos = 128;        // K positions per slab
constexpr int kMaxRows = 256;        // rows per CTA (two M tiles)
constexpr int kTileM = 128;
constexpr int kMaxStages = 16;
constexpr int kMaxABufs = 7;         // A buffers in tensor memory
constexpr int kExpWarps = 16;
constexpr int kMmaWarps = 4;         // MMA issuers, each with its own accumulator
constexpr int kThreads = 32 * (kExpWarps + 1 + kMmaWarps);
constexpr uint32_t kTmemCols = 512;  // accumulators [0, 4 Np <= 128), A buffers from 128
constexpr uint32_t kAColBase = 128;

// Wait without suspending the thread: the expanders and the MMA issuer hand
// A buffers back and forth every slab, so a wake-up delay there is paid on
// every slab.  Bounded like mbar_wait.
__device__ __forceinline__ bool mbar_spin(uint64_t *bar, uint32_t parity)
{
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0;; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(smem_addr(bar)), "r"(parity)
            : "memory");
        if (done) return true;
        if ((i & 63u) == 63u && global_ns() - t0 > kWaitLimitNs) return false;
    }
}

struct TcArgs {
    void *y;
    int64_t ldy;
    int rows, K, batch, Np;   // Np: batch padded to a multiple of 16
    int row_base, row_extra;  // CTA c owns row_base rows (+1 if c < row_extra)
    int y_f32;
    uint32_t idesc;
    uint64_t desc_hi;         // K-major, 128-byte swizzle, SBO 1024
    int box_rows;             // rows a values / masks box carries (max rows a CTA)
    int S;                    // ring stages
    int off_m, off_x;         // masks and x inside a stage
    int stage_bytes, x_bytes, off_bar;
    int x3d;                  // 1: x map is 3-D (one copy a slab), 0: 2-D (two copies)
    unsigned int *err;
};

__device__ __forceinline__ void tma3d(void *dst, const CUtensorMap *map, int x, int y, int z,
                                      uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma2d(void *dst, const CUtensorMap *map, int x, int y,
                                      uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// As tma2d, with an L2 cache policy (createpolicy) for the bytes read.
__device__ __forceinline__ void tma2d_hint(void *dst, const CUtensorMap *map, int x, int y,
                                           uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// D[tmem_d] (+)= A[tmem_a] * B[b_desc]: A in tensor memory, B in shared memory.
__device__ __forceinline__ void mma_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
        "r"(tmem_a), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void commit_to(uint64_t *bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_addr(bar))
        : "memory");
}

// 16 fp32 columns of this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 32-bit columns into this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, "
        "%10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
nm_spmm_tc_kernel(const __grid_constant__ CUtensorMap tm_vals,
                  const __grid_constant__ CUtensorMap tm_masks,
                  const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ TcArgs a)
{
    // Used as declared (not re-aligned through an integer), so every pointer
    // below stays visibly in shared memory and the compiler emits shared-
    // space loads.  The 128-byte-swizzled copies need the 1024-byte
    // alignment: checked, and the kernel does nothing without it.
    extern __shared__ __align__(1024) uint8_t tc_smem_raw[];
    uint8_t *smem = tc_smem_raw;
    if (smem_addr(tc_smem_raw) & 1023u) {
        if (threadIdx.x == 0) atomicOr(a.err, kDevErrSmemAlign);
        return;
    }
    // [stage]: values | masks (off_m) | x (off_x); then barriers and the table
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + a.off_bar);
    uint64_t *full = bars;                        // [S] TMA -> expanders, MMA
    // done[j % Q]: the MMAs of slab j have completed (one commit a slab).
    // That frees slab j's stage for the producer and its A buffer for the
    // expanders: the MMAs were issued only after every expander had read
    // the stage.  Q exceeds both ring depths, so no waiter can miss a phase.
    uint64_t *done = full + kMaxStages;           // [Q] MMA -> producer, expanders
    uint64_t *afull = done + kMaxStages + 1;      // [nbuf] expanders -> MMA
    uint64_t *acc = afull + kMaxABufs;            // MMA -> epilogue
    uint2 *sel_tab = reinterpret_cast<uint2 *>(acc + 1);  // [16]: both words' selectors
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sel_tab + 16);
    volatile int *failed = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const int r_begin = cta * a.row_base + min(cta, a.row_extra);
    const int r_count = a.row_base + (cta < a.row_extra ? 1 : 0);
    const int ntile = (r_count + kTileM - 1) / kTileM;  // 1 or 2
    const int nslab = a.K / kSlabPos;
    const int S = a.S;
    // A buffers: ntile x 64 columns each after the accumulators' 64
    const uint32_t buf_cols = static_cast<uint32_t>(ntile) * 64u;
    const int nbuf = min(kMaxABufs, static_cast<int>((kTmemCols - kAColBase) / buf_cols));
    const int Q = max(S, nbuf) + 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
        for (int j = 0; j < Q; ++j) mbar_init(&done[j], kMmaWarps);  // one commit an issuer
        for (int d = 0; d < nbuf; ++d) mbar_init(&afull[d], kExpWarps);  // one arrive a warp
        mbar_init(acc, kMmaWarps);
        *failed = 0;
        mbar_fence_init();
    }
    if (threadIdx.x < 16) {
        const uint32_t sel = expand_sel(threadIdx.x);
        sel_tab[threadIdx.x] = make_uint2(sel & 0xFFFFu, sel >> 16);
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;

    if (warp == kExpWarps) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_map(&tm_vals);
            prefetch_map(&tm_masks);
            prefetch_map(&tm_x);
            const int slab0 = static_cast<int>((static_cast<int64_t>(cta) * nslab) / gridDim.x);
            int issued = 0;
            // ring positions kept as running counters (no divisions in the
            // loop): stage s of slab k, and the done[] slot / parity of slab
            // k - S whose MMAs must have freed stage s
            int s = 0, qw = 0;
            uint32_t pw = 0;
            for (int k = 0; k < nslab && !*failed; ++k) {
                if (k >= S) {
                    if (!mbar_wait(&done[qw], pw)) {
                        *failed = 1;
                        atomicOr(a.err, kDevErrPipeTimeout);
                        break;
                    }
                    if (++qw == Q) {
                        qw = 0;
                        pw ^= 1u;
                    }
                }
                uint8_t *st = smem + s * a.stage_bytes;
                // CTAs start at different slabs (the sum is order-free), so
                // they do not all read the same x lines at the same moment
                int ks = k + slab0;
                if (ks >= nslab) ks -= nslab;
                // a box always lands whole (rows past the matrix read as zeros)
                mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(
                                                    a.box_rows * (128 + 16) + a.x_bytes));
                tma2d(st, &tm_vals, ks * 64, r_begin, &full[s]);
                tma2d(st + a.off_m, &tm_masks, ks * 4, r_begin, &full[s]);
                // x: both 64-position boxes of the slab
                if (a.x3d) {
                    tma3d(st + a.off_x, &tm_x, 0, 0, 2 * ks, &full[s]);
                } else {
                    tma2d(st + a.off_x, &tm_x, ks * kSlabPos, 0, &full[s]);
                    tma2d(st + a.off_x + a.x_bytes / 2, &tm_x, ks * kSlabPos + 64, 0, &full[s]);
                }
                ++issued;
                if (++s == S) s = 0;
            }
            for (int k = (issued > S ? issued - S : 0); k < issued; ++k)
                if (!mbar_wait(&full[k % S], (k / S) & 1)) break;
        }
    } else if (warp > kExpWarps) {
        // ------------------------------------------------ MMA issuers
        // A thread waits ~120 cycles on each tcgen05.mma it issues, whatever
        // N is, while several issuing threads proceed in parallel, so four
        // issuers split a slab: with two tiles issuer i takes tile i / 2 and
        // K steps 4 (i % 2) .. +3, with one tile K steps 2i, 2i + 1.  Each
        // accumulates into its own columns (i * Np); the epilogue adds the
        // partial sums.
        const int mi = warp - kExpWarps - 1;
        const int t = ntile == 2 ? (mi >> 1) : 0;
        const int kk0 = ntile == 2 ? 4 * (mi & 1) : 2 * mi;
        const int nkk = ntile == 2 ? 4 : 2;
        const uint32_t dcol = tmem + static_cast<uint32_t>(mi * a.Np);
        if (lane == 0) {
            int s = 0, d = 0, qd = 0;
            uint32_t ps = 0, pd = 0;  // parities of full[s] and afull[d]
            const uint32_t xstage0 = smem_addr(smem + a.off_x);
            for (int k = 0; k < nslab; ++k) {
                if (*failed) break;
                if (!mbar_spin(&full[s], ps) || !mbar_spin(&afull[d], pd)) {
                    *failed = 1;
                    atomicOr(a.err, kDevErrPipeTimeout);
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t xb = xstage0 + static_cast<uint32_t>(s * a.stage_bytes);
                const uint32_t ta = tmem + kAColBase + d * buf_cols + t * 64;
                for (int kk = kk0; kk < kk0 + nkk; ++kk) {
                    // x: 64-position box kk / 4, 32-byte step kk % 4 inside it
                    const uint32_t boff = (kk >> 2) * (a.x_bytes / 2) + (kk & 3) * 32;
                    mma_ts(dcol, ta + kk * 8, a.desc_hi | ((xb + boff) >> 4), a.idesc,
                           (k > 0 || kk > kk0) ? 1u : 0u);
                }
                commit_to(&done[qd]);
                if (++s == S) {
                    s = 0;
                    ps ^= 1u;
                }
                if (++d == nbuf) {
                    d = 0;
                    pd ^= 1u;
                }
                if (++qd == Q) qd = 0;
            }
            commit_to(acc);
        }
    } else {
        // ------------------------------------------------ expanders (warps 0-15)
        const int q = warp & 3;
        // warp = 4 h + q: lanes 32q.. of a tile; with two tiles, h / 2 is
        // the tile and h % 2 the half of the slab, with one, h the quarter
        const int h = warp >> 2;
        const int tile = ntile == 2 ? (h >> 1) : 0;
        const int c_lo = ntile == 2 ? 8 * (h & 1) : 4 * h;
        const int nc4 = ntile == 2 ? 2 : 1;            // groups of 4 chunks
        const int rr = tile * kTileM + 32 * q + lane;  // row of this lane in the CTA
        const bool warp_live = tile * kTileM + 32 * q < r_count;
        const int rs = rr < r_count ? rr : 0;          // lanes past the rows read row 0
        const int vc_lo = c_lo >> 1;  // first 16-byte value chunk (16 positions) of the share
        int s = 0, d = 0, qn = 0;
        uint32_t ps = 0, pn = 0;  // parities of full[s] and of done[qn] (slab k - nbuf)
        for (int k = 0; k < nslab; ++k) {
            // lane 0 polls for the warp
            int ok = 0;
            if (lane == 0)
                ok = !*failed && mbar_spin(&full[s], ps) && (k < nbuf || mbar_spin(&done[qn], pn));
            ok = __shfl_sync(0xffffffffu, ok, 0);
            __syncwarp();
            if (!ok) {
                if (lane == 0 && !*failed) {
                    *failed = 1;
                    atomicOr(a.err, kDevErrPipeTimeout);
                }
                break;
            }
            if (k >= nbuf && ++qn == Q) {
                qn = 0;
                pn ^= 1u;
            }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            if (warp_live) {
                const uint8_t *st = smem + s * a.stage_bytes;
                // the values box lands 128-byte swizzled: 16-byte chunk j of
                // row r at r * 128 + ((j ^ (r % 8)) * 16)
                const uint8_t *vrow = st + rs * 128;
                const uint4 m4 = *reinterpret_cast<const uint4 *>(st + a.off_m + rs * 16);
                const uint32_t ta = tmem + (static_cast<uint32_t>(32 * q) << 16) + kAColBase +
                                    d * buf_cols + tile * 64 + c_lo * 4;
                for (int g4 = 0; g4 < nc4; ++g4) {
                    // 32 positions = one mask word = two 16-byte value chunks
                    const int g = (c_lo >> 2) + g4;
                    const uint32_t mword = g == 0 ? m4.x : g == 1 ? m4.y : g == 2 ? m4.z : m4.w;
                    uint32_t w[16];
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        // value chunk vc: groups 4 vc .. 4 vc + 3, one value
                        // pair (word) each, loaded once
                        const int vc = vc_lo + 2 * g4 + h2;
                        const uint4 vv =
                            *reinterpret_cast<const uint4 *>(vrow + ((vc ^ (rs & 7)) << 4));
                        const uint32_t vw[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
                        for (int qq = 0; qq < 4; ++qq) {
                            // group 4 h2 + qq of the word: its two dense words
                            const uint2 e = sel_tab[(mword >> (16 * h2 + 4 * qq)) & 15u];
                            w[8 * h2 + 2 * qq] = prmt(vw[qq], 0u, e.x);
                            w[8 * h2 + 2 * qq + 1] = prmt(vw[qq], 0u, e.y);
                        }
                    }
                    tmem_st16(ta + 16 * g4, w);
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            }
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&afull[d]);
            if (++s == S) {
                s = 0;
                ps ^= 1u;
            }
            if (++d == nbuf) d = 0;
        }
    }

    // ---------------------------------------------------- epilogue
    __syncwarp();
    bool ok = true;
    if (warp < kExpWarps) ok = __all_sync(0xffffffffu, mbar_wait(acc, 0)) != 0;
    if (!ok && lane == 0) atomicOr(a.err, kDevErrPipeTimeout);
    const bool go = __syncthreads_and(ok && *failed == 0) != 0;
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    // warp = 4 h + q reads lanes 32q.. of tile h / 2 (two tiles) or 0, from
    // column 16 * (h % 2) or 16 * h in steps of 32 or 64
    const int eh = warp >> 2;
    const int b_lo = ntile == 2 ? 16 * (eh & 1) : 16 * eh;
    if (go && warp < kExpWarps && b_lo < a.Np) {
        const int q = warp & 3;
        const int tile = ntile == 2 ? (eh >> 1) : 0;
        const int b_step = ntile == 2 ? 32 : 64;
        const int row = tile * kTileM + 32 * q + lane;
        // the tile's partial sums: issuers 2 tile, 2 tile + 1 (two tiles) or 0-3
        const int p0 = ntile == 2 ? 2 * tile : 0;
        const int np = ntile == 2 ? 2 : 4;
        for (int b0 = b_lo; b0 < a.Np; b0 += b_step) {
            float v[16];
            const uint32_t lanes = static_cast<uint32_t>(32 * q) << 16;
            tmem_ld16(tmem + lanes + p0 * a.Np + b0, v);
            for (int pi = 1; pi < np; ++pi) {
                float w[16];
                tmem_ld16(tmem + lanes + (p0 + pi) * a.Np + b0, w);
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] += w[j];
            }
            if (row < r_count) {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (b0 + j < a.batch)
                        store_y(a.y, (b0 + j) * a.ldy + r_begin + row, v[j], a.y_f32 != 0);
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

// ------------------------------------------------------------------------
// The same product with the packed values as the sparse A operand of
// tcgen05.mma.sp: the 2:4 layout already is the compressed matrix the sparse
// tensor cores take (two values a group of four, in increasing k), so
// nothing is expanded.  Per 128-position slab:
//   * warps 8-10 (lane 0) copy by TMA the CTA's values ({64 values, rows}
//     box, 128-byte swizzle: the K-major A operand as it lands), its mask
//     words and x (as in the kernel above), one warp each;
//   * warps 0-7 (warp w: tile w / 4, rows 32 (w % 4) ..) turn each row's four
//     mask words into four metadata words (sp_meta_word: one per MMA of 32
//     positions) and store them into tensor memory, rows r and r + 8 of each
//     16-row block sharing lanes r and r + 8 (sp_meta_lane_word).  That layout
//     was read off the GPU: with one-hot x and w = position + 1, the product
//     shows which kept value each row multiplies with each x position, and
//     for all 4096 groups of a 128 x 128 slab with random masks it matched
//     this interleave exactly (one column per MMA, lane = row, placed
//     group g of every row at the lane and nibble predicted for only half of
//     them);
//   * warps 11-14 (lane 0) issue tcgen05.mma.sp (M = 128, N = batch padded to
//     16 or 32, K = 32 positions = 16 values, fp32 accumulators), each into
//     its own accumulator columns, and commit once a slab;
//   * warps 0-7 read the accumulators, add the issuers' partial sums and
//     round into y.
// A launch covers one matrix or a group of up to 8 with the same K and
// batch: each matrix's rows are spread evenly over its row units, and the
// units of all matrices are numbered in order.  A unit is one CTA, or with
// the K split one cluster of 2, 4 or 8 CTAs sharing a unit's one or two
// 128-row tiles, each streaming a share of K's slabs; ranks 1.. send their
// fp32 sums to rank 0 (st.async into its shared memory, counted on an
// mbarrier), which adds them in rank order.  sp_group_plan picks the layout.
constexpr int kSpConvWarps = 8;
constexpr int kSpProdWarp = 8;        // warps 8-10: producers
constexpr int kSpProdWarps = 3;
constexpr int kSpMmaWarps = 4;        // warps 11-14: MMA issuers
constexpr int kSpThreads = 32 * (kSpConvWarps + kSpProdWarps + kSpMmaWarps);
constexpr int kSpMaxStages = 32;      // ring stages (a stage holds only the rows it loads)
constexpr int kSpMaxMetaBufs = 12;    // metadata buffers (ntile x 4 MMAs each)
constexpr int kSpMaxAccSets = 4;      // accumulator sets an issuer rotates over, slab by slab
constexpr uint32_t kSpTmemCols = 512; // most columns a CTA allocates: accumulators, then metadata
// Tensor memory: issuer i's accumulator set j at column (i * nacc + j) * Np
// (4 issuers); from meta_base, each MMA's metadata word in its own column,
// 8-column aligned: meta_base + 8 * ((d * ntile + t) * 4 + kk) for buffer d,
// tile t, MMA kk.
__host__ __device__ constexpr uint32_t sp_meta_col(uint32_t meta_base, int ntile, int d, int t,
                                                   int kk)
{
    return meta_base + 8u * static_cast<uint32_t>((d * ntile + t) * 4 + kk);
}

constexpr int kSpMaxGroup = 8;         // matrices one launch may stream (a group's)

// One matrix of a launch: its rows are spread evenly over its row units
// [unit_begin, unit_begin + units) (CTAs, or clusters with the K split);
// its boxes carry box_rows rows.
struct SpMat {
    void *y;
    int64_t ldy;
    int row_base, row_extra;   // rows of unit u: row_base (+1 if u < row_extra)
    int unit_begin;            // first unit (units of all matrices in order)
    int box_rows;
    int x3d;                   // 1: x through the 3-D map
};

// The tensor maps of each matrix (values, mask words, x).
struct SpMaps {
    CUtensorMap v[kSpMaxGroup];
    CUtensorMap m[kSpMaxGroup];
    CUtensorMap x[kSpMaxGroup];
};

struct SpArgs {
    SpMat mat[kSpMaxGroup];
    int nmat;
    int total_units;          // row units of all matrices (grid = total_units * ksplit)
    int K, batch, Np;
    int y_f32;
    uint32_t idesc;           // tcgen05 instruction descriptor, sparse bit set
    uint64_t desc_hi;         // K-major, 128-byte swizzle, SBO 1024 (A and B)
    int ntile;                // 128-row MMA tiles a CTA (1 or 2)
    int S;                    // ring stages
    int off_m, off_x;         // masks and x inside a stage (values at 0, ntile * 16 KB)
    int stage_bytes, x_bytes, off_bar;
    int meta_mode;            // sp_meta_word mode
    int ksplit;               // CTAs (one cluster) sharing a unit of rows, each a part of K
                              // (1: no split, rows split evenly over the CTAs)
    int off_part;             // K split: rank 0's region for ranks 1..'s sums, [r - 1][row][cols]
    int split_cols;           // K split: columns summed across the cluster (8, 16 or 32 >= batch)
    uint32_t tmem_cols;       // tensor-memory columns allocated (256 or 512)
    int spin;                 // 1: metadata warps and MMA issuers spin on their barriers
    int meta_sel;             // 1: an MMA's metadata word is column kk of the buffer's
                              // group, chosen by the descriptor's sparsity selector
    int nacc;                 // accumulator sets per issuer (independent chains of MMAs)
    int nmbuf;                // metadata buffers in tensor memory
    uint32_t meta_base;       // first metadata column (after 4 * nacc * Np accumulators)
    unsigned int *err;
};

// D[tmem_d] (+)= A[a_desc] * B[b_desc], A 2:4-sparse with metadata at tmem_e.
// The cluster barrier in two halves: every thread of every CTA of the cluster
// arrives (release) and later waits (acquire); what a CTA wrote to shared
// memory before its arrive is visible to the others after their wait.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }

// The shared::cluster address of this CTA's shared address `a` in CTA `rank`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t a, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}

// Four floats into another CTA's shared memory (16-byte aligned shared::cluster
// address); the 16 bytes complete on that CTA's mbarrier `bar` (its
// shared::cluster address).
__device__ __forceinline__ void st_async_v4(uint32_t addr, float a0, float a1, float a2, float a3,
                                            uint32_t bar)
{
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
        ::"r"(addr), "f"(a0), "f"(a1), "f"(a2), "f"(a3), "r"(bar)
        : "memory");
}

// Eight fp32 columns of this warp's 32 tensor-memory lanes, without waiting
// (tmem_wait_ld before the registers are read).
__device__ __forceinline__ void tmem_ld8_nowait(uint32_t taddr, uint32_t (&r)[8])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// The metadata warps' and MMA issuers' waits: spinning (tuning key sp_spin=1,
// the default) or suspending until the phase completes.
__device__ __forceinline__ bool sp_wait(uint64_t *bar, uint32_t parity, int spin)
{
    return spin ? mbar_spin(bar, parity) : mbar_wait(bar, parity);
}

__device__ __forceinline__ void mma_sp_ss(uint32_t tmem_d, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t tmem_e, uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "tcgen05.mma.sp.cta_group::1.kind::f16 [%0], %1, %2, [%3], %4, p;\n\t}" ::"r"(tmem_d),
        "l"(a_desc), "l"(b_desc), "r"(tmem_e), "r"(idesc), "r"(accumulate)
        : "memory");
}

// One 32-bit column into this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t r0)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(r0)
                 : "memory");
}

// Four consecutive 32-bit columns into this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t r0, uint32_t r1, uint32_t r2,
                                         uint32_t r3)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
                 "r"(r0), "r"(r1), "r"(r2), "r"(r3)
                 : "memory");
}

__global__ void __launch_bounds__(kSpThreads, 1)
nm_spmm_sp_kernel(const __grid_constant__ SpMaps maps, const __grid_constant__ SpArgs a)
{
    extern __shared__ __align__(1024) uint8_t sp_smem_raw[];
    uint8_t *smem = sp_smem_raw;
    // every operand region starts 1024-byte aligned (swizzled boxes, MMA
    // descriptors), the metadata columns fit the allocation and every
    // matrix's boxes fit the stages' tiles: else nothing (the same for all
    // CTAs, before any barrier)
    bool bad_mat = a.nmat < 1 || a.nmat > kSpMaxGroup || a.total_units < 1 ||
                   gridDim.x != static_cast<unsigned>(a.total_units * a.ksplit);
    for (int i = 0; i < a.nmat && !bad_mat; ++i)
        bad_mat = a.mat[i].box_rows < 1 || a.mat[i].box_rows > kTileM * a.ntile ||
                  a.mat[i].row_base + (a.mat[i].row_extra ? 1 : 0) > a.mat[i].box_rows ||
                  a.mat[i].unit_begin < 0 || a.mat[i].unit_begin >= a.total_units;
    if (bad_mat || ((smem_addr(sp_smem_raw) | a.stage_bytes | a.off_m | a.off_x) & 1023u) ||
        a.S < 2 || a.S > kSpMaxStages ||
        a.nmbuf < 1 || a.nmbuf > kSpMaxMetaBufs || a.nacc < 1 || a.nacc > kSpMaxAccSets ||
        a.meta_base < static_cast<uint32_t>(4 * a.nacc * a.Np) ||
        (a.tmem_cols != 256 && a.tmem_cols != kSpTmemCols) ||
        sp_meta_col(a.meta_base, a.ntile, a.nmbuf - 1, a.ntile - 1, 3) >= a.tmem_cols ||
        (a.ksplit > 1 &&
         (a.ksplit > 8 ||
          (a.split_cols != 8 && a.split_cols != 16 && a.split_cols != 32) ||
          a.batch > a.split_cols || a.split_cols > a.Np ||
          a.K / kSlabPos < a.ksplit || (a.off_part & 15) ||
          a.off_part + (a.ksplit - 1) * kTileM * a.ntile * a.split_cols * 4 > a.off_bar))) {
        if (threadIdx.x == 0) atomicOr(a.err, kDevErrSmemAlign);
        return;
    }
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + a.off_bar);
    // a stage's three copies complete on their own barriers: values and x
    // (-> MMA), mask words (-> metadata warps)
    uint64_t *fullv = bars;                      // [S]
    uint64_t *fullm = fullv + kSpMaxStages;      // [S]
    uint64_t *fullx = fullm + kSpMaxStages;      // [S]
    uint64_t *done = fullx + kSpMaxStages;       // [Q] MMA -> producers, metadata warps
    uint64_t *mfull = done + kSpMaxStages + 1;   // [nmbuf] metadata warps -> MMA
    uint64_t *acc = mfull + kSpMaxMetaBufs;      // MMA -> epilogue
    uint64_t *part = acc + 1;                    // K split, rank 0: ranks 1..'s sums landed
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(part + 1);
    volatile int *failed = reinterpret_cast<volatile int *>(tmem_slot + 1);

    // Programmatic dependent launch: the next kernel in the stream may start
    // its own prologue and weight copies now; this one reads x and writes y
    // only after the previous kernel has completed (griddepcontrol.wait in
    // the x producer and before the epilogue).
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    // K split: the a.ksplit consecutive CTAs of a cluster share one unit of
    // rows (one or two 128-row tiles), CTA `rank` taking slabs [slab_lo,
    // slab_lo + nslab).  Rows are spread evenly over the units (CTAs without
    // the split).
    const int rank = a.ksplit > 1 ? cta % a.ksplit : 0;
    const int unit = cta / a.ksplit;
    int mi = 0;  // the matrix of this unit (units of a matrix are consecutive)
    while (mi + 1 < a.nmat && unit >= a.mat[mi + 1].unit_begin) ++mi;
    const SpMat &mt = a.mat[mi];
    const int lu = unit - mt.unit_begin;  // unit within the matrix
    const int r_begin = lu * mt.row_base + min(lu, mt.row_extra);
    const int r_count = mt.row_base + (lu < mt.row_extra ? 1 : 0);
    const int ntile = (r_count + kTileM - 1) / kTileM;  // this CTA's tiles (<= a.ntile)
    const int nconv = 4 * ntile;                        // metadata warps at work
    const int nslab_all = a.K / kSlabPos;
    const int slab_lo = static_cast<int>(static_cast<int64_t>(rank) * nslab_all / a.ksplit);
    const int nslab =
        static_cast<int>(static_cast<int64_t>(rank + 1) * nslab_all / a.ksplit) - slab_lo;
    const int S = a.S;
    const int NB = a.nmbuf;
    const int Q = max(S, NB) + 1;  // exceeds both ring depths

    // the tensor maps' descriptors start on their way now
    const CUtensorMap *tm_vals = &maps.v[mi], *tm_masks = &maps.m[mi], *tm_x = &maps.x[mi];
    if (warp == kSpProdWarp && lane < 3) prefetch_map(lane == 0 ? tm_vals : lane == 1 ? tm_masks : tm_x);
    // one thread a barrier (Q exceeds S and NB)
    if (static_cast<int>(threadIdx.x) < Q) {
        const int i = threadIdx.x;
        if (i < S) {
            mbar_init(&fullv[i], 1);
            mbar_init(&fullm[i], 1);
            mbar_init(&fullx[i], 1);
        }
        mbar_init(&done[i], kSpMmaWarps);  // one commit an issuer
        if (i < NB) mbar_init(&mfull[i], nconv);
        if (i == 0) {
            mbar_init(acc, kSpMmaWarps);
            mbar_init(part, 1);
            *failed = 0;
        }
        mbar_fence_init();
        // rank 0 of a split expects ranks 1..'s sums: split_cols floats for
        // each row of its tiles (the ranks of a cluster share the unit, so
        // its tiles)
        if (i == 0 && a.ksplit > 1 && rank == 0)
            mbar_arrive_expect_tx(
                part, static_cast<uint32_t>((a.ksplit - 1) * nconv * 32 * a.split_cols * 4));
    }
    // the cluster's barriers are initialised before any CTA of it writes to
    // another (the matching wait is in the epilogue)
    if (a.ksplit > 1) cluster_arrive();
    __syncthreads();

    // Tensor memory: warp 0 allocates it while the producers start their
    // copies; the other warps that use it meet on barrier 2.
    const bool producer = warp >= kSpProdWarp && warp < kSpProdWarp + kSpProdWarps;
    uint32_t tmem = 0;
    if (!producer) {
        if (warp == 0) {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_addr(tmem_slot)),
                         "r"(a.tmem_cols)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        named_barrier_sync(2, kSpThreads - 32 * kSpProdWarps);
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        tmem = *tmem_slot;
    }

    if (producer) {
        // ------------------------------------------------ TMA producers
        // Three warps, one copy each a slab (values, mask words, x): issuing a
        // tensor copy blocks the issuing thread for a while, and the three
        // issue in parallel.  Each arrives on the stage's barrier with its
        // own byte count on its own barrier.
        const int role = warp - kSpProdWarp;
        uint64_t *full = role == 0 ? fullv : role == 1 ? fullm : fullx;
        if (role == 2) pdl_wait();  // x may be the previous kernel's output
        if (lane == 0) {
            // the weights are read once: evict them first, so that they do
            // not push x (read by every CTA) out of L2
            const uint64_t pol = l2_evict_first_policy();
            const int slab0 = static_cast<int>((static_cast<int64_t>(cta) * nslab) / gridDim.x) %
                              max(nslab, 1);
            const uint32_t box_rows = static_cast<uint32_t>(mt.box_rows);
            const uint32_t tx = role == 0 ? box_rows * 128u
                              : role == 1 ? box_rows * 16u
                                          : static_cast<uint32_t>(a.x_bytes);
            int issued = 0, s = 0, qw = 0;
            uint32_t pw = 0;
            for (int k = 0; k < nslab && !*failed; ++k) {
                if (k >= S) {
                    if (!mbar_wait(&done[qw], pw)) {
                        *failed = 1;
                        atomicOr(a.err, kDevErrPipeTimeout);
                        break;
                    }
                    if (++qw == Q) {
                        qw = 0;
                        pw ^= 1u;
                    }
                }
                uint8_t *st = smem + s * a.stage_bytes;
                int ks = k + slab0;
                if (ks >= nslab) ks -= nslab;
                ks += slab_lo;
                mbar_arrive_expect_tx(&full[s], tx);
                if (role == 0) {
                    tma2d_hint(st, tm_vals, ks * 64, r_begin, &full[s], pol);
                } else if (role == 1) {
                    tma2d_hint(st + a.off_m, tm_masks, ks * 4, r_begin, &full[s], pol);
                } else if (mt.x3d) {
                    tma3d(st + a.off_x, tm_x, 0, 0, 2 * ks, &full[s]);
                } else {
                    tma2d(st + a.off_x, tm_x, ks * kSlabPos, 0, &full[s]);
                    tma2d(st + a.off_x + a.x_bytes / 2, tm_x, ks * kSlabPos + 64, 0, &full[s]);
                }
                ++issued;
                if (++s == S) s = 0;
            }
            // before the CTA can exit, every copy this thread issued must have
            // landed
            for (int k = (issued > S ? issued - S : 0); k < issued; ++k)
                if (!mbar_wait(&full[k % S], (k / S) & 1)) break;
        }
    } else if (warp >= kSpProdWarp + kSpProdWarps) {
        // ------------------------------------------------ MMA issuers
        // Issuer i: with two tiles, tile i / 2 and MMAs 2 (i % 2), +1 of the
        // slab; with one tile, MMA i.  Each accumulates into its own sets.
        const int mi = warp - kSpProdWarp - kSpProdWarps;
        const int t = ntile == 2 ? (mi >> 1) : 0;
        const int kk0 = ntile == 2 ? 2 * (mi & 1) : mi;
        const int nkk = ntile == 2 ? 2 : 1;
        const uint32_t dcol0 = tmem + static_cast<uint32_t>(mi * a.nacc * a.Np);
        if (lane == 0) {
            int s = 0, d = 0, qd = 0, ka = 0;  // ka: accumulator set of slab k
            uint32_t ps = 0, pd = 0;
            const uint32_t stage0 = smem_addr(smem);
            for (int k = 0; k < nslab; ++k) {
                if (*failed) break;
                if (!sp_wait(&fullv[s], ps, a.spin) || !sp_wait(&fullx[s], ps, a.spin) ||
                    !sp_wait(&mfull[d], pd, a.spin)) {
                    *failed = 1;
                    atomicOr(a.err, kDevErrPipeTimeout);
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t st = stage0 + static_cast<uint32_t>(s * a.stage_bytes);
                const uint32_t av = st + static_cast<uint32_t>(t) * (kTileM * 128u);
                const uint32_t xb = st + static_cast<uint32_t>(a.off_x);
                for (int kk = kk0; kk < kk0 + nkk; ++kk) {
                    // A: 16 values (32 bytes) of each row from value 16 kk of
                    // the slab; x: 32 positions, box kk / 2, 64-byte step kk % 2
                    const uint32_t aoff = static_cast<uint32_t>(kk) * 32u;
                    const uint32_t boff = (kk >> 1) * (a.x_bytes / 2) + (kk & 1) * 64;
                    const uint32_t meta =
                        tmem + sp_meta_col(a.meta_base, a.ntile, d, t, a.meta_sel ? 0 : kk);
                    const uint32_t idesc = a.meta_sel ? (a.idesc | static_cast<uint32_t>(kk)) : a.idesc;
                    // slab k adds into set k % nacc: the first slab of each set
                    // starts it
                    mma_sp_ss(dcol0 + static_cast<uint32_t>(ka * a.Np),
                              a.desc_hi | ((av + aoff) >> 4), a.desc_hi | ((xb + boff) >> 4),
                              meta, idesc, (k >= a.nacc || kk > kk0) ? 1u : 0u);
                }
                commit_to(&done[qd]);
                if (++s == S) {
                    s = 0;
                    ps ^= 1u;
                }
                if (++d == NB) {
                    d = 0;
                    pd ^= 1u;
                }
                if (++qd == Q) qd = 0;
                if (++ka == a.nacc) ka = 0;
            }
            commit_to(acc);
        }
    } else if (warp < nconv) {
        // ------------------------------------------------ metadata (warps 0-7)
        const int t = warp >> 2, q = warp & 3;
        const int rr = t * kTileM + 32 * q + lane;     // row of this lane in the CTA
        const int rs = rr < r_count ? rr : 0;          // lanes past the rows read row 0
        const uint32_t tlanes = tmem + (static_cast<uint32_t>(32 * q) << 16);
        int s = 0, d = 0, qn = 0;
        uint32_t ps = 0, pn = 0;
        for (int k = 0; k < nslab; ++k) {
            int ok = 0;
            if (lane == 0)
                ok = !*failed && sp_wait(&fullm[s], ps, a.spin) &&
                     (k < NB || sp_wait(&done[qn], pn, a.spin));
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0 && !*failed) {
                    *failed = 1;
                    atomicOr(a.err, kDevErrPipeTimeout);
                }
                break;
            }
            if (k >= NB && ++qn == Q) {
                qn = 0;
                pn ^= 1u;
            }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint4 m4 =
                *reinterpret_cast<const uint4 *>(smem + s * a.stage_bytes + a.off_m + rs * 16);
            const uint32_t mw[4] = {m4.x, m4.y, m4.z, m4.w};
            uint32_t lw[4];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                // this row's metadata word for MMA kk, interleaved with that of
                // the row 8 apart (sp_meta_lane_word)
                const uint32_t own = sp_meta_word(mw[kk], a.meta_mode);
                const uint32_t partner = __shfl_xor_sync(0xffffffffu, own, 8);
                lw[kk] = sp_meta_lane_word(own, partner, (lane & 8) != 0);
            }
            // the four words at their 8-aligned columns (or, with the selector
            // layout, in four consecutive columns); one 32-column store of the
            // four measured no faster than four single-column ones
            if (a.meta_sel) {
                tmem_st4(tlanes + sp_meta_col(a.meta_base, a.ntile, d, t, 0), lw[0], lw[1], lw[2],
                         lw[3]);
            } else {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tmem_st1(tlanes + sp_meta_col(a.meta_base, a.ntile, d, t, kk), lw[kk]);
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&mfull[d]);
            if (++s == S) {
                s = 0;
                ps ^= 1u;
            }
            if (++d == NB) d = 0;
        }
    }

    // ---------------------------------------------------- epilogue
    __syncwarp();
    bool ok = true;
    if (warp < nconv) ok = __all_sync(0xffffffffu, mbar_wait(acc, 0)) != 0;
    if (!ok && lane == 0) atomicOr(a.err, kDevErrPipeTimeout);
    const bool go = __syncthreads_and(ok && *failed == 0) != 0;
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    pdl_wait();  // y may still be read by the previous kernel
    if (a.ksplit > 1) {
        // K split (split_cols = 8, 16 or 32 columns matter, at least the
        // batch): ranks 1.. send their sums to rank 0's region with
        // st.async, which counts them on rank 0's `part` barrier; rank 0 adds
        // them in rank order.  Every rank sends (zeros after a failure) so
        // that rank 0's wait always ends; the cluster wait makes rank 0's
        // barrier initialisation visible first.
        cluster_wait();
        if (warp < nconv) {
            const int t = warp >> 2, q = warp & 3;
            const int row = t * kTileM + 32 * q + lane;  // row in the unit
            const int ncol = a.split_cols;
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0.f;
            if (go) {
                // the tile's sets that slabs started (issuer i, set j at
                // (i * nacc + j) * 16; issuers 2t, 2t + 1 with two tiles, else
                // all four), 8 columns at a time: up to 4 sets a batch, one
                // wait each
                const int i0 = ntile == 2 ? 2 * t : 0;
                const int ni = ntile == 2 ? 2 : kSpMmaWarps;
                const int nused = min(a.nacc, nslab);
                const uint32_t lanes = tmem + (static_cast<uint32_t>(32 * q) << 16);
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    if (8 * h >= ncol) break;
                    for (int i = i0; i < i0 + ni; ++i)
                        for (int j0 = 0; j0 < nused; j0 += 4) {
                            uint32_t r[4][8];
#pragma unroll
                            for (int jj = 0; jj < 4; ++jj)
                                if (j0 + jj < nused)
                                    tmem_ld8_nowait(lanes + (i * a.nacc + j0 + jj) * a.Np + 8 * h,
                                                    r[jj]);
                            tmem_wait_ld();
#pragma unroll
                            for (int jj = 0; jj < 4; ++jj)
                                if (j0 + jj < nused)
#pragma unroll
                                    for (int c = 0; c < 8; ++c)
                                        v[8 * h + c] += __uint_as_float(r[jj][c]);
                        }
                }
            }
            // rank r's sums at [r - 1][row] in rows of ncol floats, kTileM *
            // a.ntile rows a rank
            const int rank_rows = kTileM * a.ntile;
            const uint32_t my_part = smem_addr(smem + a.off_part);
            if (rank > 0) {
                const uint32_t dst = cluster_map(
                    my_part + static_cast<uint32_t>(((rank - 1) * rank_rows + row) * ncol * 4), 0);
                const uint32_t bar = cluster_map(smem_addr(part), 0);
#pragma unroll
                for (int c = 0; c < 32; c += 4)
                    if (c < ncol) st_async_v4(dst + 4 * c, v[c], v[c + 1], v[c + 2], v[c + 3], bar);
            } else {
                // ranks 1.. reach this point within their own bounded waits
                bool landed = true;
                if (lane == 0) landed = mbar_wait(part, 0, 8 * kWaitLimitNs);
                landed = __shfl_sync(0xffffffffu, landed ? 1 : 0, 0) != 0;
                if (!landed && lane == 0) atomicOr(a.err, kDevErrPipeTimeout);
                const float *pp = reinterpret_cast<const float *>(smem + a.off_part);
                for (int r = 1; r < a.ksplit; ++r) {
                    const float *src = pp + ((r - 1) * rank_rows + row) * ncol;
#pragma unroll
                    for (int c = 0; c < 32; c += 4)
                        if (c < ncol) {
                            const float4 pv = *reinterpret_cast<const float4 *>(src + c);
                            v[c] += pv.x;
                            v[c + 1] += pv.y;
                            v[c + 2] += pv.z;
                            v[c + 3] += pv.w;
                        }
                }
                if (go && landed && row < r_count) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j < a.batch) store_y(mt.y, j * mt.ldy + r_begin + row, v[j], a.y_f32 != 0);
                }
            }
        }
    } else if (go && warp < nconv) {
        const int t = warp >> 2, q = warp & 3;
        const int row = t * kTileM + 32 * q + lane;
        // the tile's partial sums: every accumulator set of issuers 2t, 2t + 1
        // (two tiles) or 0-3 (sets used: min(nacc, nslab))
        const int p0 = (ntile == 2 ? 2 * t : 0) * a.nacc;
        const int np = (ntile == 2 ? 2 : 4) * a.nacc;
        const int nused = min(a.nacc, nslab);
        const uint32_t lanes = static_cast<uint32_t>(32 * q) << 16;
        for (int b0 = 0; b0 < a.Np; b0 += 16) {
            float v[16];
            tmem_ld16(tmem + lanes + p0 * a.Np + b0, v);
            for (int pi = 1; pi < np; ++pi) {
                if (pi % a.nacc >= nused) continue;  // a set no slab started
                float w[16];
                tmem_ld16(tmem + lanes + (p0 + pi) * a.Np + b0, w);
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] += w[j];
            }
            if (row < r_count) {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (b0 + j < a.batch)
                        store_y(mt.y, (b0 + j) * mt.ldy + r_begin + row, v[j], a.y_f32 != 0);
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(a.tmem_cols)
                     : "memory");
    }
}

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                 const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                 const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_tiled_tc()
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

// x [batch][ldx] fp16 viewed as {64 positions, batch rows, K/64 blocks}: a
// {64, Np, 2} box lands as two [Np][64] boxes (the slab's positions 0-63,
// then 64-127), 128-byte swizzled.
bool encode_x3d(EncodeTiled enc, CUtensorMap *m, const void *x, uint64_t K, uint64_t batch,
                uint64_t ldx_bytes, uint32_t Np)
{
    const cuuint64_t dims[3] = {64, batch, K / 64};
    const cuuint64_t strides[2] = {ldx_bytes, 128};
    const cuuint32_t box[3] = {64, Np, 2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(x), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode2d(EncodeTiled enc, CUtensorMap *m, CUtensorMapDataType dt, const void *base,
              uint64_t inner, uint64_t outer, uint64_t stride_bytes, uint32_t box_inner,
              uint32_t box_outer, CUtensorMapSwizzle sw)
{
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// tcgen05 kind::f16 instruction descriptor: fp32 accumulator, fp16 A and B,
// both K-major, N / 8 at bit 17, M / 16 at bit 24.
uint32_t spmm_tc_idesc(int N) { return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (8u << 24); }

// K-major operand, 128-byte swizzle: 8-row groups 1024 bytes apart (SBO),
// LBO unused by this layout (encoded lbo), version 1, layout 2.
uint64_t spmm_tc_desc_hi(uint32_t lbo_enc)
{
    return (static_cast<uint64_t>(lbo_enc & 0x3FFFu) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

bool spmm_tc_applies(const SpmvProblem &p, int nsm)
{
    if (p.N != 2 || p.M != 4 || p.batch < 1 || p.batch > 32) return false;
    if (p.K % kSlabPos != 0 || p.K / 2 > (1ll << 31) || p.rows < 1) return false;
    if (p.ldx % 8 != 0) return false;
    // tensor-map bases must be 16-byte aligned
    if ((reinterpret_cast<uintptr_t>(p.values) | reinterpret_cast<uintptr_t>(p.masks) |
         reinterpret_cast<uintptr_t>(p.x)) & 15u)
        return false;
    const int64_t grid = std::min<int64_t>(p.rows, nsm);
    return (p.rows + grid - 1) / grid <= kMaxRows;
}

// The sparse kernel may take `bytes` of dynamic shared memory (set once per
// device, at the device's opt-in maximum, which every launch stays under).
bool sp_allow_smem(int bytes)
{
    static std::atomic<int> done[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (done[dev].load(std::memory_order_relaxed) >= bytes) return true;
    if (cudaFuncSetAttribute(nm_spmm_sp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             bytes) != cudaSuccess)
        return false;
    done[dev].store(bytes, std::memory_order_relaxed);
    return true;
}

// Clusters of k CTAs of the sparse kernel (one CTA an SM) that can be
// resident at once (cached per device and k; 0 if none or unknown).
int sp_resident_clusters(int k)
{
    static std::atomic<int> cache[64][9];
    int dev = 0;
    if (k < 2 || k > 8 || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int c = cache[dev][k].load(std::memory_order_relaxed);
    if (c != 0) return c > 0 ? c : 0;
    const int avail = max_dynamic_smem();
    const int nsm = sm_count();
    int n = 0;
    if (avail > 0 && nsm >= k && sp_allow_smem(avail)) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(nsm / k * k));
        cfg.blockDim = dim3(kSpThreads);
        cfg.dynamicSmemBytes = static_cast<size_t>(avail);
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = static_cast<unsigned>(k);
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, nm_spmm_sp_kernel, &cfg) != cudaSuccess) {
            cudaGetLastError();  // not a sticky error: clear it
            n = 0;
        }
    }
    cache[dev][k].store(n > 0 ? n : -1, std::memory_order_relaxed);
    return n;
}

// The plan for these products on this device (its resident cluster counts
// for k = 2, 4, 8).
SpGroupPlan sp_plan(const SpmvProblem *ps, int count, int nsm)
{
    int resident[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};
    for (int k = 2; k <= 8; k *= 2) resident[k] = sp_resident_clusters(k);
    int64_t rows[kSpMaxGroup];
    for (int i = 0; i < count; ++i) rows[i] = ps[i].rows;
    return sp_group_plan(rows, count, ps[0].K, ps[0].batch, nsm, resident);
}

// The sparse-operand variant (nm_spmm_sp_kernel) for `count` products with
// the same K, batch, x stride and y type in one launch (each as
// spmm_tc_applies allows); one product is a group of one.
cudaError_t launch_spmm_sp_group(const SpmvProblem *ps, int count, uint64_t desc_hi, int meta_mode,
                                 cudaStream_t s)
{
    if (count < 1 || count > kSpMaxGroup) return cudaErrorNotSupported;
    const SpmvProblem &p = ps[0];
    for (int i = 1; i < count; ++i)
        if (ps[i].K != p.K || ps[i].batch != p.batch || ps[i].ldx != p.ldx ||
            ps[i].y_f32 != p.y_f32)
            return cudaErrorNotSupported;
    EncodeTiled enc = encode_tiled_tc();
    if (!enc) return cudaErrorNotSupported;
    const int nsm = sm_count();
    if (nsm <= 0) return cudaErrorInvalidDevice;
    const int Np = p.batch <= 16 ? 16 : 32;
    const int64_t Lv = p.K / 2;
    const int64_t Lm = p.K / 32;
    const SpGroupPlan plan = sp_plan(ps, count, nsm);
    if (plan.max_box_rows > kMaxRows) return cudaErrorNotSupported;
    const int ksplit = plan.k;
    const int grid = static_cast<int>(plan.total_units) * ksplit;
    const int box_rows = plan.max_box_rows;  // the stages' layout
    // x: only the batch's rows, rounded up to 8 (one 128-byte-swizzle atom);
    // the MMA reads Np rows, and the rows past Bx read whatever follows: they
    // only feed accumulator columns that are never stored
    const int Bx = (p.batch + 7) / 8 * 8;
    SpMaps maps;
    SpArgs a = {};
    int64_t unit = 0;
    for (int i = 0; i < count; ++i) {
        const SpmvProblem &q = ps[i];
        const int br = plan.box_rows[i];
        if (!encode2d(enc, &maps.v[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, q.values, Lv, q.rows,
                      Lv * 2, 64, br, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode2d(enc, &maps.m[i], CU_TENSOR_MAP_DATA_TYPE_UINT32, q.masks, Lm, q.rows,
                      Lm * 4, 4, br, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorNotSupported;
        SpMat &m = a.mat[i];
        m.x3d = 1;
        if (!encode_x3d(enc, &maps.x[i], q.x, q.K, q.batch, q.ldx * 2, Bx)) {
            m.x3d = 0;
            if (!encode2d(enc, &maps.x[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, q.x, q.K, q.batch,
                          q.ldx * 2, 64, Bx, CU_TENSOR_MAP_SWIZZLE_128B))
                return cudaErrorNotSupported;
        }
        m.y = q.y;
        m.ldy = q.ldy;
        // rows spread evenly over the matrix's units (CTAs, or clusters with
        // the K split); a box carries row_base (+1) rows
        m.row_base = static_cast<int>(q.rows / plan.units[i]);
        m.row_extra = static_cast<int>(q.rows % plan.units[i]);
        m.unit_begin = static_cast<int>(unit);
        m.box_rows = br;
        unit += plan.units[i];
    }
    a.nmat = count;
    a.total_units = static_cast<int>(plan.total_units);
    a.K = static_cast<int>(p.K);
    a.batch = p.batch;
    a.Np = Np;
    a.y_f32 = p.y_f32 ? 1 : 0;
    a.idesc = spmm_tc_idesc(Np) | (1u << 2);  // sparse A
    a.desc_hi = desc_hi;
    a.meta_mode = meta_mode;
    a.meta_sel = bulk_tuning().sp_sel;
    a.ksplit = ksplit;
    a.spin = bulk_tuning().sp_spin;
    a.ntile = (box_rows + kTileM - 1) / kTileM;
    // accumulator sets and metadata buffers: the tuning keys sp_acc and
    // sp_mbufs, else as many as tensor memory holds
    a.tmem_cols = static_cast<uint32_t>(bulk_tuning().sp_tmem);
    a.nacc = std::max(1, std::min(kSpMaxAccSets, bulk_tuning().sp_acc));
    while (a.nacc > 1 && 4 * a.nacc * Np + a.ntile * 32 > static_cast<int>(a.tmem_cols)) --a.nacc;
    a.meta_base = static_cast<uint32_t>(4 * a.nacc * Np);
    const int fit = (static_cast<int>(a.tmem_cols) - static_cast<int>(a.meta_base)) / (a.ntile * 32);
    a.nmbuf = std::min(kSpMaxMetaBufs, fit);
    if (bulk_tuning().sp_mbufs > 0) a.nmbuf = std::min(a.nmbuf, bulk_tuning().sp_mbufs);
    if (a.nmbuf < 1) return cudaErrorNotSupported;
    // a stage: the loaded rows' values, their mask words, x.  The MMA reads
    // all 128 rows of a tile; rows past the box read the bytes after it
    // (their sums are never stored), and `slack` after the last stage keeps
    // those reads inside the allocation.  Small stages make a deep ring: a
    // stage is refilled only a full round trip (copy, metadata, MMA) after
    // it was issued, so the bytes in flight per SM are the ring's.
    a.x_bytes = 2 * Bx * 128;  // two 64-position planes of Bx rows
    a.off_m = (box_rows * 128 + 1023) / 1024 * 1024;
    a.off_x = a.off_m + (box_rows * 16 + 1023) / 1024 * 1024;
    a.stage_bytes = a.off_x + a.x_bytes;
    const int slack = std::max({0, a.ntile * kTileM * 128 - a.stage_bytes, (Np - Bx) * 128});
    const int tail = 1024 + 512;
    const int avail = max_dynamic_smem();
    if (avail <= 0) return cudaErrorInvalidDevice;
    // K split: rank 0 receives ranks 1..'s sums (4 KB each) in a region of
    // its own, which the ring never uses
    a.split_cols = p.batch <= 8 ? 8 : p.batch <= 16 ? 16 : 32;
    const int part_bytes = ksplit > 1 ? (ksplit - 1) * kTileM * a.ntile * a.split_cols * 4 : 0;
    a.S = std::min(kSpMaxStages, (avail - tail - slack - part_bytes) / a.stage_bytes);
    if (bulk_tuning().sp_stages > 0) a.S = std::min(a.S, bulk_tuning().sp_stages);
    if (a.S < 2) return cudaErrorNotSupported;
    a.off_part = a.S * a.stage_bytes + slack;  // 16-byte aligned (stages 1 KB, slack 128 B units)
    a.off_bar = a.off_part + part_bytes;
    a.err = p.err;
    const int smem = a.off_bar + tail;
    if (!sp_allow_smem(avail)) return cudaErrorNotSupported;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kSpThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int nattr = 0;
    if (bulk_tuning().pdl) {
        attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[nattr].val.programmaticStreamSerializationAllowed = 1;
        ++nattr;
    }
    if (ksplit > 1) {
        attr[nattr].id = cudaLaunchAttributeClusterDimension;
        attr[nattr].val.clusterDim.x = static_cast<unsigned>(ksplit);
        attr[nattr].val.clusterDim.y = 1;
        attr[nattr].val.clusterDim.z = 1;
        ++nattr;
    }
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    return cudaLaunchKernelEx(&cfg, nm_spmm_sp_kernel, maps, a);
}

cudaError_t launch_spmm_sp(const SpmvProblem &p, uint64_t desc_hi, int meta_mode, cudaStream_t s)
{
    return launch_spmm_sp_group(&p, 1, desc_hi, meta_mode, s);
}

cudaError_t launch_spmm_tc_group(const SpmvGroup &g, uint64_t desc_hi, cudaStream_t s)
{
    if (!bulk_tuning().tc_sp || !bulk_tuning().sp_group) return cudaErrorNotSupported;
    return launch_spmm_sp_group(g.p, g.count, desc_hi, bulk_tuning().sp_meta, s);
}

cudaError_t launch_spmm_tc(const SpmvProblem &p, uint64_t desc_hi, cudaStream_t s)
{
    if (bulk_tuning().tc_sp) return launch_spmm_sp(p, desc_hi, bulk_tuning().sp_meta, s);
    EncodeTiled enc = encode_tiled_tc();
    if (!enc) return cudaErrorNotSupported;
    const int nsm = sm_count();
    if (nsm <= 0) return cudaErrorInvalidDevice;
    const int Np = p.batch <= 16 ? 16 : 32;
    const int64_t Lv = p.K / 2;          // fp16 values a row
    const int64_t Lm = p.K / 32;         // mask words a row
    const int grid = static_cast<int>(std::min<int64_t>(p.rows, nsm));
    const int box_rows = static_cast<int>(p.rows / grid + (p.rows % grid ? 1 : 0));
    if (box_rows > kMaxRows) return cudaErrorNotSupported;
    CUtensorMap tv, tm, tx;
    if (!encode2d(enc, &tv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, p.values, Lv, p.rows, Lv * 2, 64,
                  box_rows, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode2d(enc, &tm, CU_TENSOR_MAP_DATA_TYPE_UINT32, p.masks, Lm, p.rows, Lm * 4, 4,
                  box_rows, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorNotSupported;  // the caller takes another kernel
    // the 3-D view of x has a stride (128 bytes) below the row pitch; a
    // driver that refuses it gets the 2-D map and two copies a slab
    int x3d = 1;
    if (!encode_x3d(enc, &tx, p.x, p.K, p.batch, p.ldx * 2, Np)) {
        x3d = 0;
        if (!encode2d(enc, &tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, p.x, p.K, p.batch, p.ldx * 2, 64,
                      Np, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorNotSupported;  // the caller takes another kernel
    }
    TcArgs a = {};
    a.x3d = x3d;
    a.box_rows = box_rows;
    a.y = p.y;
    a.ldy = p.ldy;
    a.rows = static_cast<int>(p.rows);
    a.K = static_cast<int>(p.K);
    a.batch = p.batch;
    a.Np = Np;
    a.row_base = static_cast<int>(p.rows / grid);
    a.row_extra = static_cast<int>(p.rows % grid);
    a.y_f32 = p.y_f32 ? 1 : 0;
    a.idesc = spmm_tc_idesc(Np);
    a.desc_hi = desc_hi;
    a.x_bytes = 2 * Np * 128;  // two 64-position boxes of Np rows
    a.off_m = (box_rows * 128 + 1023) / 1024 * 1024;
    a.off_x = a.off_m + (box_rows * 16 + 1023) / 1024 * 1024;
    a.stage_bytes = a.off_x + a.x_bytes;
    const int tail = 1024 + 512;  // alignment slack, barriers and table
    const int avail = max_dynamic_smem();
    if (avail <= 0) return cudaErrorInvalidDevice;
    a.S = std::min(kMaxStages, (avail - tail) / a.stage_bytes);
    if (a.S < 2) return cudaErrorNotSupported;
    a.off_bar = a.S * a.stage_bytes;
    a.err = p.err;
    const int smem = a.off_bar + tail;
    static std::atomic<int> smem_set{0};
    if (smem > smem_set.load(std::memory_order_relaxed)) {
        cudaError_t e =
            cudaFuncSetAttribute(nm_spmm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        smem_set.store(smem, std::memory_order_relaxed);
    }
    nm_spmm_tc_kernel<<<grid, kThreads, smem, s>>>(tv, tm, tx, a);
    return cudaGetLastError();
}

}  // namespace nm

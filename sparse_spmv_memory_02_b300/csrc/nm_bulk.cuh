// N:M SpMV with the weight stream staged through shared memory by bulk
// (TMA) copies -- the main kernel of libnm on sm_103a.
//
// The operation is the N:M sparse matrix-vector product with bitmask
// indexing and fixed-step traversal of "SparseDecoding: Decoding-Aware
// Pruning for Accurate and Efficient LLM Inference" (Abstract).  Every kept
// value (2 bytes) and every mask bit is read from HBM exactly once per call,
// so the kernel is built to keep enough bytes in flight to saturate HBM3e
// while spending as few issue slots as possible per byte.
//
// Roles inside a CTA (one CTA per SM, rows split evenly over the CTAs):
//   * warp 0, lane 0 -- the producer.  It walks the CTA's work as a
//     sequence of stages (R rows x one K tile each) and, for every stage,
//     issues one bulk copy of each row's value segment and one of its mask
//     segment into a ring of S shared-memory slots, completing on the slot's
//     "full" mbarrier.  Values and masks of consecutive rows are contiguous
//     in HBM (fixed step: a row is exactly K/M*N values and K/32 mask words),
//     so each copy is one contiguous byte range.
//   * warps 1..W -- the consumers.  Consumer thread t owns the chunk columns
//     t + j*32W (j < CPL) of every row of a K tile and holds the matching
//     slice of x in registers for the whole tile.  Per slot it reads each
//     16-byte value chunk and its CK mask bits from shared memory, decodes
//     the mask with byte permutes (Pattern<N, M>), accumulates in fp32, then
//     releases the slot ("empty" mbarrier) before reducing: a warp
//     reduce-scatter, partial sums across warps through shared memory and
//     one named barrier, one rounding into y (or a carry to the next K tile).
// The producer runs up to S stages ahead of the consumers, so the memory
// system always has about S-1 stages per SM in flight.
//
// Programmatic dependent launch: the kernel signals at once that the next
// kernel in the stream may start launching, and its own consumers wait for
// the previous kernel (griddepcontrol.wait) before they read x or write y.
// The producer does not wait: the packed weights are read-only input that
// no kernel of this library writes, so the weight stream of call i+1
// overlaps the tail of call i.
#pragma once

#include <cuda_runtime.h>

#include <atomic>

#include "nm_fast.cuh"
#include "nm_pipe.cuh"

namespace nm {

struct BulkArgs {
    const uint8_t *values;  // [rows][vrow_bytes]
    const uint8_t *masks;   // [rows][mrow_bytes]
    const __half *x;        // [B][ldx]
    void *y;                // [B][ldy]
    unsigned int *err;      // device error word
    int64_t ldx, ldy, vrow_bytes, mrow_bytes;
    int rows, chunks;       // 16-byte value chunks per row
    int tile_chunks;        // chunks per K tile = CPL * 32 * W
    int ktiles;
    int R;                  // rows per stage, <= bulk_rmax(B)
    int S;                  // ring slots
    int seg_v, seg_m;       // shared bytes of one row's value / mask segment
    int stage_bytes;        // R * (seg_v + seg_m)
    int off_bar, off_part, off_carry;  // byte offsets in dynamic shared memory
    int row_base, row_extra;  // CTA c owns row_base rows (+1 if c < row_extra)
    int y_f32;
};

// Rows per stage at most: R*B partial sums per consumer thread, at most 8.
__host__ __device__ constexpr int bulk_rmax(int B) { return B >= 8 ? 1 : (B >= 5 ? 1 : 8 / B); }

constexpr int kBulkMaxConsumerWarps = 12;
constexpr int kBulkMaxThreads = 32 * (kBulkMaxConsumerWarps + 1);

template <int N, int M, int B, int CPL>
__global__ void __launch_bounds__(kBulkMaxThreads, 1)
nm_spmv_bulk_kernel(const BulkArgs a)
{
    using P = Pattern<N, M>;
    using mask_t = typename P::mask_t;
    constexpr int CK = P::CK;
    constexpr int XR = CK / 2;  // x words per chunk and vector
    constexpr int XV = CK / 8;  // 16-byte x loads per chunk and vector
    constexpr int MB = CK / 8;  // mask bytes per chunk
    constexpr int RMAX = bulk_rmax(B);
    constexpr int V = pow2_ceil(RMAX * B);

    extern __shared__ __align__(128) uint8_t bulk_smem[];
    uint8_t *smem = bulk_smem;
    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + a.off_bar);
    uint64_t *empty = full + a.S;
    float *part = reinterpret_cast<float *>(smem + a.off_part);    // [2][W][V]
    float *carry = reinterpret_cast<float *>(smem + a.off_carry);  // [rows of CTA][B]

    const int W = (blockDim.x >> 5) - 1;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], W);
        }
        mbar_fence_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    const int cta = blockIdx.x;
    const int r_begin = cta * a.row_base + min(cta, a.row_extra);
    const int r_count = a.row_base + (cta < a.row_extra ? 1 : 0);
    const int nrt = (r_count + a.R - 1) / a.R;  // row tiles
    const int Q = nrt * a.ktiles;               // stages of this CTA

    if (warp == 0) {
        // ------------------------------------------------------ producer
        if (lane != 0) return;
        const uint64_t pol = l2_evict_first_policy();
        int q = 0;
        for (; q < Q; ++q) {
            const int slot = q % a.S;
            if (q >= a.S && !mbar_wait(&empty[slot], ((q / a.S) - 1) & 1)) {
                atomicOr(a.err, kDevErrPipeTimeout);
                break;
            }
            const int kt = q / nrt;
            const int i0 = (q - kt * nrt) * a.R;
            const int nr = min(a.R, r_count - i0);
            const int c0 = kt * a.tile_chunks;
            const int nc = min(a.tile_chunks, a.chunks - c0);
            const uint32_t vb = static_cast<uint32_t>(nc) * 16u;
            const uint32_t mb = static_cast<uint32_t>(nc) * MB;
            mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(nr) * (vb + mb));
            uint8_t *st = ring + static_cast<size_t>(slot) * a.stage_bytes;
            if (a.ktiles == 1) {
                // whole rows (seg_v == vrow_bytes, seg_m == mrow_bytes): the
                // stage's rows are one contiguous range of each array
                const int64_t row0 = r_begin + i0;
                bulk_g2s(st, a.values + row0 * a.vrow_bytes, static_cast<uint32_t>(nr) * vb,
                         &full[slot], pol);
                bulk_g2s(st + a.R * a.seg_v, a.masks + row0 * a.mrow_bytes,
                         static_cast<uint32_t>(nr) * mb, &full[slot], pol);
            } else {
                for (int i = 0; i < nr; ++i) {
                    const int64_t row = r_begin + i0 + i;
                    bulk_g2s(st + i * a.seg_v, a.values + row * a.vrow_bytes + c0 * 16LL, vb,
                             &full[slot], pol);
                    bulk_g2s(st + a.R * a.seg_v + i * a.seg_m,
                             a.masks + row * a.mrow_bytes + static_cast<int64_t>(c0) * MB, mb,
                             &full[slot], pol);
                }
            }
        }
        // Do not leave while copies into this CTA's shared memory may still
        // be in flight (normally they have long landed).
        for (int p = max(0, q - a.S); p < q; ++p)
            if (!mbar_wait(&full[p % a.S], (p / a.S) & 1)) {
                atomicOr(a.err, kDevErrPipeTimeout);
                break;
            }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int T = W * 32;
    const int ct = threadIdx.x - 32;
    const int cw = warp - 1;
    constexpr int SH = 5 - log2i<V>();
    bool failed = false;

    pdl_wait();  // x may be the previous kernel's output; y may still be read by it

    uint32_t xr[CPL][B][XR];
    bool okj[CPL];
    int buf = 0;
    for (int q = 0; q < Q; ++q) {
        const int slot = q % a.S;
        const int kt = q / nrt;
        const int rt = q - kt * nrt;
        const int i0 = rt * a.R;
        const int nr = min(a.R, r_count - i0);
        if (rt == 0) {  // new K tile: this thread's slice of x into registers
            const int c0 = kt * a.tile_chunks;
            const int nc = min(a.tile_chunks, a.chunks - c0);
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                const int cl = j * T + ct;
                okj[j] = cl < nc;
#pragma unroll
                for (int b = 0; b < B; ++b) {
                    const __half *xp = a.x + b * a.ldx + static_cast<int64_t>(c0 + cl) * CK;
#pragma unroll
                    for (int u = 0; u < XV; ++u) {
                        const uint4 t = okj[j] ? ld_cg_v4(xp + 8 * u) : make_uint4(0, 0, 0, 0);
                        xr[j][b][4 * u + 0] = t.x;
                        xr[j][b][4 * u + 1] = t.y;
                        xr[j][b][4 * u + 2] = t.z;
                        xr[j][b][4 * u + 3] = t.w;
                    }
                }
            }
        }

        if (!failed && !mbar_wait(&full[slot], (q / a.S) & 1)) {
            failed = true;  // keep taking part in the barriers; y is garbage
            atomicOr(a.err, kDevErrPipeTimeout);
        }
        const uint8_t *sv = ring + static_cast<size_t>(slot) * a.stage_bytes;
        const uint8_t *sm = sv + a.R * a.seg_v;

        float acc[V];
#pragma unroll
        for (int t = 0; t < V; ++t) acc[t] = 0.f;
#pragma unroll
        for (int i = 0; i < RMAX; ++i) {
            if (i < nr) {
#pragma unroll
                for (int j = 0; j < CPL; ++j) {
                    if (okj[j]) {
                        const int cl = j * T + ct;
                        const uint4 v = *reinterpret_cast<const uint4 *>(sv + i * a.seg_v + cl * 16);
                        const mask_t m = *reinterpret_cast<const mask_t *>(sm + i * a.seg_m + cl * MB);
                        const typename P::Sel sel = P::decode(m);
#pragma unroll
                        for (int b = 0; b < B; ++b)
                            acc[i * B + b] = P::dot(v, sel, xr[j][b], acc[i * B + b]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);

        warp_reduce_scatter<V>(acc, lane);
        if ((lane & ((1 << SH) - 1)) == 0) part[(buf * W + cw) * V + (lane >> SH)] = acc[0];
        named_barrier_sync(1, T);
        if (ct < nr * B) {
            const int i = ct / B, b = ct - (ct / B) * B;
            float tot = 0.f;
            for (int w = 0; w < W; ++w) tot += part[(buf * W + w) * V + ct];
            if (a.ktiles > 1) {
                float *c = carry + (i0 + i) * B + b;
                if (kt > 0) tot += *c;
                *c = tot;
            }
            if (kt == a.ktiles - 1) store_y(a.y, b * a.ldy + r_begin + i0 + i, tot, a.y_f32 != 0);
        }
        buf ^= 1;
        // The carry slot of (row, vector) is only ever touched by consumer
        // thread (row in tile) * B + vector, so K tiles need no extra barrier.
    }
}

// ---------------------------------------------------------------- host side

struct BulkTuning {
    int warps = 0;           // consumer warps (0: chosen per shape)
    int cpl = 0;             // chunk columns per consumer thread (0: chosen)
    int R = 0;               // rows per stage (0: chosen)
    int stage_bytes = 16384; // target bytes per stage
    int ring_bytes = 98304;  // shared memory for the ring
    int ctas_per_sm = 1;
    int pdl = 1;             // programmatic dependent launch
    // row kernel (batch 1 to 8)
    int rows_kernel = 1;           // 0: never take it
    int rows_warps = 0;            // warps per CTA (0: 16)
    int rows_R = 0;                // rows per task (0: chosen)
    int rows_task_bytes = 6144;    // largest task (rows x K tile) in bytes
    int rows_ring_bytes = 200000;  // shared memory for the slots
    int rows_xtile_bytes = 49152;  // largest x tile (B vectors) before K is tiled
    int rows_pair = 0;             // size each CTA to half an SM (see nm_rows.cuh)
    int rows_pre = 1;              // tasks per warp copied before the dependence wait (<= SW)
    int rows_prew = 16;            // warps of a CTA that copy them (the first ones)
    int rows_two = -1;             // 1: two rows a task (segments too) at batch <= 2 for
                                   // patterns whose chunk spans 32 positions; 0: never; -1: auto
    int rows_l2pre_bytes = 0;      // weight bytes per CTA warmed in L2 before that wait
    // tensor-core product (2:4, batch 8 and up; nm_spmm_tc.cu)
    int tc = -1;                   // 1: wherever it applies, 0: never, -1: by batch and
                                   // rows per SM (takes_tensor_cores in nm_api.cu)
    int tc_lbo = 1;                // encoded leading-byte-offset field of its descriptors
    // Test of the device-side failure path only: the row kernel issues no
    // copies and waits 2 ms (not 2 s) on its slot barriers, so every wait
    // runs out, the error word is set and the kernel returns.
    int wait_fault_test = 0;
    int tc_sp = 1;                 // 1: the tensor-core product takes the packed values as the
                                   // sparse A operand (tcgen05.mma.sp); 0: it expands them into
                                   // tensor memory (the earlier, slower kernel)
    int sp_meta = 0;               // metadata nibble order of that path (0: i0 | i1 << 2)
    int sp_acc = 2;                // accumulator sets each MMA issuer of that path rotates over
    int sp_mbufs = 0;              // its metadata buffers (0: as many as tensor memory holds)
    int sp_spin = 1;               // 1: its metadata warps and MMA issuers spin; 0: suspend
    int sp_split = 1;              // 1: one-tile layers split K over clusters of 2-8 CTAs
    int sp_sel = 0;                // 1: its four metadata words of a slab in consecutive columns,
                                   // the MMA picking one with the descriptor's sparsity selector
    int sp_stages = 0;             // its ring's stages at most (0: as many as shared memory holds)
    int sp_tmem = 512;             // tensor-memory columns a CTA of it allocates (256 or 512)
    int sp_k = 0;                  // its K split's cluster size (0: chosen by shape)
    int sp_units = 0;              // its K split's row units at least (0: one a tile or tile pair)
    int sp_group = 1;              // 1: a group's products in one launch of it; 0: one a product
};

// Tuning defaults, overridable by NM_BULK_TUNE="key=value,..." with keys
// warps, cpl, R, stage, ring (bulk kernel), rows_warps, rows_R, rows_task,
// rows_ring, rows_xtile, rows_pair, rows_pre, rows_prew, rows_l2pre, rows_two, rows (row-per-warp kernel),
// ctas, pdl, wait_fault_test, tc_sp, sp_meta, sp_acc, sp_mbufs, sp_sel, sp_spin, sp_split,
// sp_stages, sp_tmem, sp_k, sp_units, sp_group
// (both), tc, tc_lbo (tensor-core product); read once per process.
const BulkTuning &bulk_tuning();

// How the sparse-operand tensor-core product (nm_spmm_tc.cu) lays a 2:4
// product over the SMs: without the split (k = 1) the rows are spread over
// `units` CTAs; with it, `units` units of one or two 128-row tiles are each
// shared by a cluster of k = 2, 4 or 8 CTAs, each streaming 1/k of K's
// 128-position slabs.  box_rows: rows of the largest unit.
struct SpSplit {
    int k;
    int64_t units;
    int box_rows;
};

// The plan with the least estimated time (sp_split_plan in nm_bulk_plan.cu,
// where the cost model is described).  resident[k] (k = 2, 4, 8): clusters
// of k CTAs resident at once on the device (0: none).
SpSplit sp_split_plan(int64_t rows, int64_t K, int batch, int nsm, const int *resident);

// The same for `count` (<= 8) products with the same K and batch in one
// launch: units[i] row units of matrix i (consecutive, matrix 0 first), its
// rows spread evenly over them (box_rows[i] rows at most).  With one matrix
// it is sp_split_plan's plan.
struct SpGroupPlan {
    int k;
    int count;
    int64_t units[8];
    int box_rows[8];
    int64_t total_units;
    int max_box_rows;
};
SpGroupPlan sp_group_plan(const int64_t *rows, int count, int64_t K, int batch, int nsm,
                          const int *resident);

struct BulkPlan {
    int W, cpl, ktiles, tile_chunks, R, S, grid;
    int seg_v, seg_m, stage_bytes, off_bar, off_part, off_carry;
    size_t smem;
};

// Chooses consumer warps W and chunk columns per thread so that the K tile
// 32*W*CPL covers the row's chunks with few idle lanes and few K tiles;
// then R and S so that a stage is about `stage_bytes` and the ring fits.
// Returns false if no plan fits in shared memory.
bool bulk_plan(int64_t rows, int chunks, int CK, int B, int nsm, int max_smem, BulkPlan *out);

template <int N, int M, int B, int CPL>
cudaError_t launch_bulk_instance(const SpmvProblem &p, const BulkPlan &pl, cudaStream_t s)
{
    auto kernel = nm_spmv_bulk_kernel<N, M, B, CPL>;
    // Largest dynamic shared size configured so far, per device.
    static std::atomic<int> smem_set[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int need = static_cast<int>(pl.smem);
    if (dev < 0 || dev >= 64 || need > smem_set[dev].load(std::memory_order_relaxed)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, need);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) {
            int cur = smem_set[dev].load(std::memory_order_relaxed);
            while (need > cur && !smem_set[dev].compare_exchange_weak(cur, need)) {
            }
        }
    }
    using P = Pattern<N, M>;
    BulkArgs a;
    a.values = static_cast<const uint8_t *>(p.values);
    a.masks = reinterpret_cast<const uint8_t *>(p.masks);
    a.x = static_cast<const __half *>(p.x);
    a.y = p.y;
    a.err = p.err;
    a.ldx = p.ldx;
    a.ldy = p.ldy;
    a.vrow_bytes = p.K / P::CK * 16;
    a.mrow_bytes = ((p.K + 31) / 32) * 4;
    a.rows = static_cast<int>(p.rows);
    a.chunks = static_cast<int>(p.K / P::CK);
    a.tile_chunks = pl.tile_chunks;
    a.ktiles = pl.ktiles;
    a.R = pl.R;
    a.S = pl.S;
    a.seg_v = pl.seg_v;
    a.seg_m = pl.seg_m;
    a.stage_bytes = pl.stage_bytes;
    a.off_bar = pl.off_bar;
    a.off_part = pl.off_part;
    a.off_carry = pl.off_carry;
    a.row_base = a.rows / pl.grid;
    a.row_extra = a.rows % pl.grid;
    a.y_f32 = p.y_f32 ? 1 : 0;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl.grid);
    cfg.blockDim = dim3(32 * (pl.W + 1));
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = bulk_tuning().pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

// Chunk columns per consumer thread that have an instantiation: the x slice
// a thread holds (CPL * B * CK/2 words) stays at most 64 registers.
__host__ __device__ constexpr bool bulk_cpl_ok(int CK, int B, int cpl)
{
    return (cpl == 1 || cpl == 2 || cpl == 3 || cpl == 4 || cpl == 6 || cpl == 8) &&
           cpl * B * (CK / 2) <= 64;
}

template <int N, int M, int B, int CPL>
cudaError_t launch_bulk_cpl(const SpmvProblem &p, const BulkPlan &pl, cudaStream_t s)
{
    if constexpr (bulk_cpl_ok(Pattern<N, M>::CK, B, CPL))
        return launch_bulk_instance<N, M, B, CPL>(p, pl, s);
    return cudaErrorNotSupported;
}

template <int N, int M, int B>
cudaError_t launch_bulk_b(const SpmvProblem &p, const BulkPlan &pl, cudaStream_t s)
{
    switch (pl.cpl) {
    case 1: return launch_bulk_cpl<N, M, B, 1>(p, pl, s);
    case 2: return launch_bulk_cpl<N, M, B, 2>(p, pl, s);
    case 3: return launch_bulk_cpl<N, M, B, 3>(p, pl, s);
    case 4: return launch_bulk_cpl<N, M, B, 4>(p, pl, s);
    case 6: return launch_bulk_cpl<N, M, B, 6>(p, pl, s);
    case 8: return launch_bulk_cpl<N, M, B, 8>(p, pl, s);
    default: return cudaErrorNotSupported;
    }
}

// Returns cudaErrorNotSupported (nothing launched) when no plan fits; the
// caller then takes the direct-load kernel.
template <int N, int M>
cudaError_t launch_bulk_pattern(const SpmvProblem &p, cudaStream_t s)
{
    using P = Pattern<N, M>;
    const int nsm = sm_count();
    if (nsm <= 0) return cudaErrorInvalidDevice;
    const int max_smem = max_dynamic_smem();
    if (max_smem <= 0) return cudaErrorInvalidDevice;
    BulkPlan pl;
    if (!bulk_plan(p.rows, static_cast<int>(p.K / P::CK), P::CK, p.batch, nsm, max_smem, &pl))
        return cudaErrorNotSupported;
    switch (p.batch) {
    case 1: return launch_bulk_b<N, M, 1>(p, pl, s);
    case 2: return launch_bulk_b<N, M, 2>(p, pl, s);
    case 3: return launch_bulk_b<N, M, 3>(p, pl, s);
    case 4: return launch_bulk_b<N, M, 4>(p, pl, s);
    case 5: return launch_bulk_b<N, M, 5>(p, pl, s);
    case 6: return launch_bulk_b<N, M, 6>(p, pl, s);
    case 7: return launch_bulk_b<N, M, 7>(p, pl, s);
    case 8: return launch_bulk_b<N, M, 8>(p, pl, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace nm

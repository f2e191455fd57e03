// N:M SpMV for one to eight vectors: every warp owns whole rows and streams
// its own weights into shared memory with bulk (TMA) copies; x is held once
// per CTA in shared memory.  The main kernel of libnm.
//
// The operation is the N:M sparse matrix-vector product with bitmask
// indexing and fixed-step traversal of "SparseDecoding: Decoding-Aware
// Pruning for Accurate and Efficient LLM Inference" (Abstract); at batch 1
// it is the whole decode-step cost of an N:M-pruned linear layer.  Each kept
// value and mask bit is read from HBM once, so the kernel's job is to keep
// enough bytes in flight with as few instructions per byte as possible.
//
// Work split.  Rows are split evenly over one CTA per SM.  x is held in
// shared memory for all of K when B * K * 2 bytes fit the x budget (else K
// is cut into K tiles, each staged in turn).  A CTA's rows form row tiles of
// R rows; a task is one row tile x one segment of the K tile (a row longer
// than the task size is cut into even segments of a multiple of 32 chunks),
// and row tile rt belongs to warp rt % W, which takes its segments in order
// and keeps the row's sums in registers across them.
//
// Self-feeding warps.  Warp w owns SW shared-memory slots.  Its lane 0
// issues the bulk copies of w's own next tasks (the rows' value segments and
// mask segments; a segment of one row, or R whole rows, is one contiguous
// byte range of each array -- a packed row is exactly K/M*N values and K/32
// mask words -- so a task is two copies), each completing on the slot's
// mbarrier.  After the warp has read a slot it immediately issues its task
// SW ahead into it.  Every warp is thus its own pipeline with up to SW tasks
// in flight: bulk copies issued by one warp complete at a limited rate per
// warp on this GPU, and W independent issuers per SM are what reach HBM
// bandwidth.  There is no producer warp, no "empty" barrier and no
// synchronisation between warps other than one named barrier per K tile.
// A warp waits on every phase of its own slots in order, so a parity wait
// can never mistake an older phase for the one it wants.
//
// Per task, lane l walks the segment's chunk columns l, l+32, ...: it loads
// the column's x units from shared memory once and uses them for all R rows
// (from three vectors up, R = 2 and the vectors are taken a few at a time
// so that their x words fit in registers)
// (each a 16-byte value chunk plus its mask bits, decoded by byte permutes
// in Pattern<N, M>), accumulating in fp32; after a row tile's last segment
// the warp reduces its R*B sums with a reduce-scatter butterfly and one lane
// per sum rounds it into y (or adds it to the row's carry when the row spans
// several K tiles; a row's tiles always go to the same warp).
//
// Programmatic dependent launch: the packed weights are read-only input that
// no kernel of this library writes, so each warp issues its first `pre`
// tasks (one by default) before griddepcontrol.wait and one call's weight
// stream starts under the tail of the previous call; x is read and y written
// only after the wait.  The rest of the first SW tasks is issued once x is
// loaded: the x loads are L2 hits, and copies issued earlier by the same SM
// would be served ahead of them, so a deep prefetch before the wait delays
// the start of compute by more than it saves.  The prologue before the
// first copies is kept short (barriers initialised by one thread each, the
// CTA's rows looked up before the barrier setup) because a CTA of the next
// call only starts when the SM's CTA of the previous call exits.
//
// Two options measured slower on the Llama-3.1-8B-shaped block and are off
// by default: warming L2 with the CTA's next rows before the wait
// (rows_l2pre), and planning each launch for half an SM (rows_pair) so that
// CTAs of consecutive calls share SMs -- half the shared memory per CTA
// leaves too few bytes in flight once a call runs alone.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "nm_bulk.cuh"  // Pattern<N, M>, pipeline primitives, tuning

namespace nm {

// One matrix of a launch (a launch may fuse up to kRowsMaxGroup independent
// products with the same pattern, batch and K; each CTA works on exactly one
// of them).
constexpr int kRowsMaxGroup = NM_MAX_GROUP;
struct RowsMat {
    const uint8_t *values;  // [rows][vrow_bytes]
    const uint8_t *masks;   // [rows][mrow_bytes]
    const __half *x;        // [B][ldx]
    void *y;                // [B][ldy]
    int64_t ldy;
    int row_base, row_extra;  // its CTA c owns row_base rows (+1 if c < row_extra)
    const uint8_t *values2;   // gate/up pair: the up matrix (same shape as this one)
    const uint8_t *masks2;
};

// The scalars every CTA reads first come first (kernel parameters are read
// through the constant cache; keeping them on few lines keeps the prologue
// short), the per-matrix table last.
struct RowsArgs {
    int nmat;
    int SW;                 // slots per warp
    int pre;                // tasks per warp issued before the dependence wait (<= SW)
    int pre_warps;          // warps that issue them (the first pre_warps of the CTA)
    int chunks;             // 16-byte value chunks per row
    int tile_chunks;        // chunks per K tile (the x held in shared memory at once)
    int ktiles;
    int seg_chunks;         // chunks per row segment (one task) within a K tile
    int nseg, nseg_last;    // segments of a full K tile / of the last K tile
    int seg_v, seg_m;       // shared bytes of one row's value / mask segment
    int stage_bytes;        // R * (seg_v + seg_m)
    int xbuf_bytes;         // one x tile buffer: B * XV * tile_chunks * 16
    int off_x, off_bar, off_tab, off_carry;
    int y_f32;
    int pair;               // 1: gate/up pair, y = silu(gate x) * (up x) (R == 2)
    int l2pre_rows;         // rows per CTA warmed in L2 before the dependence wait
    int no_copy;            // test of the wait time-out: issue no copies (nothing ever
                            // completes a slot barrier, nothing is in flight at exit)
    uint64_t wait_limit_ns; // limit of every slot-barrier wait
    int cta_begin[kRowsMaxGroup + 1];  // first CTA of each matrix; [nmat] = grid
    int64_t ldx, vrow_bytes, mrow_bytes;
    unsigned int *err;      // device error word
    RowsMat mat[kRowsMaxGroup];
};

constexpr int kRowsMaxWarps = 16;

// Largest rows per task a batch size is built for (R * B partial sums per
// lane: at most 8 for one or two vectors, 16 from three up).
__host__ __device__ constexpr int rows_rmax(int B) { return B <= 2 ? 4 : 2; }

// Layout of the x tile in shared memory, in 16-byte units (XV = CK / 8 units
// per chunk column and vector).  One or two vectors: unit-major, unit u of
// vector b for column c at (b * XV + u) * tile + c, so that a warp reading
// one unit of 32 consecutive columns reads 512 contiguous bytes.  Three or
// more: column-major, column c's B * XV units contiguous and padded to an
// odd count (rows_x_col_units), so a lane reaches every unit of its column
// at a compile-time offset, and 8 lanes on consecutive columns (an odd
// number of units apart) hit 8 different 16-byte bank groups.
__host__ __device__ constexpr int rows_x_col_units(int B, int CK)
{
    return B <= 2 ? 0 : ((B * (CK / 8)) % 2 == 0 ? B * (CK / 8) + 1 : B * (CK / 8));
}
__host__ __device__ constexpr int rows_x_tile_bytes(int B, int CK, int tile_chunks)
{
    return B <= 2 ? B * (CK / 8) * tile_chunks * 16 : rows_x_col_units(B, CK) * tile_chunks * 16;
}

// Copies task (K tile kt, segment sg, rows i0 .. i0+nr-1 of the CTA) into a
// slot: the rows' value segments at st + i * seg_v, their mask segments at
// st + R * seg_v + i * seg_m, completing on bar.
template <int R, int MB>
__device__ __forceinline__ void rows_issue(const RowsArgs &a, const uint8_t *values,
                                           const uint8_t *masks, uint8_t *st, uint64_t *bar,
                                           int kt, int sg, int i0, int nr, int r_begin,
                                           uint64_t pol)
{
    const int t0 = kt * a.tile_chunks;
    const int c0 = t0 + sg * a.seg_chunks;
    const int nc = min(a.seg_chunks, min(a.tile_chunks, a.chunks - t0) - sg * a.seg_chunks);
    const uint32_t vb = static_cast<uint32_t>(nc) * 16u;
    const uint32_t mb = static_cast<uint32_t>(nc) * MB;
    const int64_t row0 = r_begin + i0;
    if (R == 2 && a.pair) {
        // gate/up pair: output row row0 is slot row 0 of the gate matrix
        // and slot row 1 of the up matrix
        const RowsMat &m = a.mat[0];
        mbar_arrive_expect_tx(bar, 2u * (vb + mb));
        bulk_g2s(st, values + row0 * a.vrow_bytes + c0 * 16LL, vb, bar, pol);
        bulk_g2s(st + a.seg_v, m.values2 + row0 * a.vrow_bytes + c0 * 16LL, vb, bar, pol);
        bulk_g2s(st + R * a.seg_v, masks + row0 * a.mrow_bytes + static_cast<int64_t>(c0) * MB,
                 mb, bar, pol);
        bulk_g2s(st + R * a.seg_v + a.seg_m,
                 m.masks2 + row0 * a.mrow_bytes + static_cast<int64_t>(c0) * MB, mb, bar, pol);
        return;
    }
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nr) * (vb + mb));
    if (R == 1 || a.seg_chunks == a.chunks) {
        // one row, or whole rows (then seg_v == vrow_bytes and seg_m ==
        // mrow_bytes): one contiguous range of each array, in the slot's layout
        bulk_g2s(st, values + row0 * a.vrow_bytes + c0 * 16LL, static_cast<uint32_t>(nr) * vb,
                 bar, pol);
        bulk_g2s(st + R * a.seg_v, masks + row0 * a.mrow_bytes + static_cast<int64_t>(c0) * MB,
                 static_cast<uint32_t>(nr) * mb, bar, pol);
    } else {
        for (int i = 0; i < nr; ++i) {
            const int64_t row = row0 + i;
            bulk_g2s(st + i * a.seg_v, values + row * a.vrow_bytes + c0 * 16LL, vb, bar, pol);
            bulk_g2s(st + R * a.seg_v + i * a.seg_m,
                     masks + row * a.mrow_bytes + static_cast<int64_t>(c0) * MB, mb, bar, pol);
        }
    }
}

template <int N, int M, int B, int R>
__global__ void __launch_bounds__(32 * kRowsMaxWarps, 1)
nm_spmv_rows_kernel(const __grid_constant__ RowsArgs a)
{
    using P = Pattern<N, M>;
    using mask_t = typename P::mask_t;
    constexpr int CK = P::CK;
    constexpr int XR = CK / 2;  // x words per chunk and vector
    constexpr int XV = CK / 8;  // 16-byte x units per chunk and vector
    constexpr int MB = CK / 8;  // mask bytes per chunk
    constexpr int V = pow2_ceil(R * B);
    constexpr int SH = 5 - log2i<V>();
    constexpr int XCU = rows_x_col_units(B, CK);  // x units a column (0: unit-major)

    extern __shared__ __align__(128) uint8_t rows_smem[];
    const int W = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint8_t *ring = rows_smem;                                             // [W][SW] slots
    uint8_t *xbuf = rows_smem + a.off_x;                                   // [<=2][B][XV][tile]
    uint64_t *full = reinterpret_cast<uint64_t *>(rows_smem + a.off_bar);  // [W][SW]
    float *carry = reinterpret_cast<float *>(rows_smem + a.off_carry);     // [rows of CTA][B]
    uint32_t *tab = reinterpret_cast<uint32_t *>(rows_smem + a.off_tab);   // [P::kTabWords]

    pdl_launch_dependents();

    // The matrix this CTA works on, and its rows of it.
    int mi = 0;
    while (mi + 1 < a.nmat && static_cast<int>(blockIdx.x) >= a.cta_begin[mi + 1]) ++mi;
    const RowsMat &mt = a.mat[mi];
    const int cta = static_cast<int>(blockIdx.x) - a.cta_begin[mi];
    const int r_begin = cta * mt.row_base + min(cta, mt.row_extra);
    const int r_count = mt.row_base + (cta < mt.row_extra ? 1 : 0);
    const int RT = a.pair ? 1 : R;  // output rows per row tile (a pair tile is one row of each)
    const int nrt = (r_count + RT - 1) / RT;                       // row tiles of the CTA
    const int per_kt = nrt > warp ? (nrt - warp + W - 1) / W : 0;  // this warp's tiles per K tile
    const int ntask = per_kt * ((a.ktiles - 1) * a.nseg + a.nseg_last);
    const int ncopy = a.no_copy ? 0 : ntask;  // tasks whose copies are issued
    uint8_t *my_ring = ring + static_cast<size_t>(warp) * a.SW * a.stage_bytes;
    uint64_t *my_full = full + warp * a.SW;
    const uint64_t pol = l2_evict_first_policy();

    // Thread s initialises slot barrier s (all at once, not one thread
    // looping over W * SW of them).
    if (threadIdx.x < W * a.SW) {
        mbar_init(&full[threadIdx.x], 1);
        mbar_fence_init();
    }
    __syncthreads();

    // Issue cursor over this warp's tasks in consumption order: K tile, then
    // row tile, then segment.  It advances by one task at a time.
    int issued = 0;
    int iss_kt = 0, iss_n = 0, iss_s = 0;
    auto issue_next = [&](uint8_t *st, uint64_t *bar) {
        const int rt = warp + iss_n * W;
        rows_issue<R, MB>(a, mt.values, mt.masks, st, bar, iss_kt, iss_s, rt * RT,
                          min(RT, r_count - rt * RT), r_begin, pol);
        ++issued;
        if (++iss_s == (iss_kt == a.ktiles - 1 ? a.nseg_last : a.nseg)) {
            iss_s = 0;
            if (++iss_n == per_kt) {
                iss_n = 0;
                ++iss_kt;
            }
        }
    };

    // This warp's first `pre` tasks (weights only: no dependence on the
    // previous kernel); the rest of its first SW after x is staged.
    if (lane == 0 && warp < a.pre_warps)
        while (issued < a.pre && issued < ncopy)
            issue_next(my_ring + static_cast<size_t>(issued) * a.stage_bytes, &my_full[issued]);

    // The mask-decode table (8-wide patterns), published to all warps by the
    // barrier after the x tile below.
    if constexpr (P::kTabWords > 0)
        for (int i = threadIdx.x; i < P::kTabWords; i += blockDim.x) tab[i] = P::tab_entry(i);

    // Warm L2 with the CTA's next rows (values and masks of consecutive rows
    // are contiguous) in pieces of up to 32 KB, one piece per lane of the
    // last warp: HBM streams them while the previous kernel drains, and no
    // data comes back to the SM to queue ahead of the x loads below.  The
    // rows the `pre` tasks copy are skipped.
    if (a.l2pre_rows > 0 && warp == W - 1) {
        const int skip = min(r_count, (a.pre + a.nseg - 1) / a.nseg * W * R);
        const int n = min(r_count - skip, a.l2pre_rows);
        const int64_t r0 = r_begin + skip;
        const uint8_t *vsrc = mt.values + r0 * a.vrow_bytes;
        const uint8_t *msrc = mt.masks + r0 * a.mrow_bytes;
        const int64_t vlen = n * a.vrow_bytes, mlen = n * a.mrow_bytes;
        constexpr int64_t kPiece = 32768;
        for (int64_t off = lane * kPiece; off < vlen; off += 32 * kPiece)
            prefetch_l2(vsrc + off, static_cast<uint32_t>(min(kPiece, vlen - off)));
        for (int64_t off = lane * kPiece; off < mlen; off += 32 * kPiece)
            prefetch_l2(msrc + off, static_cast<uint32_t>(min(kPiece, mlen - off)));
    }

    pdl_wait();  // x may be the previous kernel's output; y may still be read by it

    // loop-invariant strides, read from the parameter block once
    const int seg_chunks = a.seg_chunks;
    const int seg_v = a.seg_v, seg_m = a.seg_m;
    const int xstride = a.tile_chunks * 16;  // bytes between x units (unit-major layout)

    bool failed = false;
    int j = 0;          // next task of this warp
    int slot = 0;       // its slot (j % SW)
    uint32_t phase = 0; // parity of its slot's phase ((j / SW) & 1)
    for (int kt = 0; kt < a.ktiles; ++kt) {
        const int c0 = kt * a.tile_chunks;
        const int nc = min(a.tile_chunks, a.chunks - c0);
        const int nseg = kt == a.ktiles - 1 ? a.nseg_last : a.nseg;
        uint8_t *xs = xbuf + (kt & 1) * a.xbuf_bytes;
        // x tile -> shared memory in the layout of rows_x_col_units.  The
        // buffer written here was last read in K tile kt-2, and every warp
        // has passed the barrier of tile kt-1 since.
        // Each thread issues up to XU loads before its first store, so a
        // tile costs one memory round trip per XU * blockDim units.
        constexpr int XU = 4;
        const int xunits = B * XV * nc;
        for (int e0 = threadIdx.x; e0 < xunits; e0 += XU * blockDim.x) {
            uint4 t[XU];
            int dst[XU];
#pragma unroll
            for (int q = 0; q < XU; ++q) {
                const int e = e0 + q * static_cast<int>(blockDim.x);
                if (e < xunits) {
                    const int b = B == 1 ? 0 : e / (XV * nc);
                    const int r = e - b * (XV * nc);
                    const int c = r / XV, u = r - (r / XV) * XV;
                    t[q] = ld_cg_v4(mt.x + b * a.ldx + static_cast<int64_t>(c0 + c) * CK + 8 * u);
                    dst[q] = XCU == 0 ? ((b * XV + u) * a.tile_chunks + c) * 16
                                      : (c * XCU + b * XV + u) * 16;
                }
            }
#pragma unroll
            for (int q = 0; q < XU; ++q)
                if (e0 + q * static_cast<int>(blockDim.x) < xunits)
                    *reinterpret_cast<uint4 *>(xs + dst[q]) = t[q];
        }
        if (kt == 0 && lane == 0)
            while (issued < a.SW && issued < ncopy)
                issue_next(my_ring + static_cast<size_t>(issued) * a.stage_bytes,
                           &my_full[issued]);
        named_barrier_sync(1, blockDim.x);

        for (int n = 0; n < per_kt; ++n) {
            const int rt = warp + n * W;
            const int i0 = rt * RT;
            const int nr = min(RT, r_count - i0);
            float acc[V];
#pragma unroll
            for (int t = 0; t < V; ++t) acc[t] = 0.f;
            for (int sg = 0; sg < nseg; ++sg, ++j) {
                if (!failed && !mbar_wait(&my_full[slot], phase, a.wait_limit_ns)) {
                    failed = true;  // give up waiting; y is garbage, the error word says so
                    atomicOr(a.err, kDevErrPipeTimeout);
                }
                uint8_t *sv = my_ring + static_cast<size_t>(slot) * a.stage_bytes;
                const uint8_t *sm = sv + R * seg_v;
                // columns [cs, ce) of the K tile; the slot holds them from 0.
                // All R rows are computed even when the task has nr < R (the
                // CTA's last row tile): the rows past nr read stale slot
                // bytes -- the mask only feeds byte permutes, never an
                // address -- and their sums are never stored.  This keeps
                // the loop free of per-row branches.
                const int cs = sg * a.seg_chunks;
                const int ncol = min(nc, cs + seg_chunks) - cs;
                // per-lane pointers to column `lane` of the segment, advanced
                // by 32 columns an iteration; the other rows (and x units)
                // sit at fixed strides from them
                const uint8_t *vp = sv + lane * 16;
                const uint8_t *mp = sm + lane * MB;
                const uint8_t *xp = xs + (cs + lane) * 16;
                if constexpr (B <= 2) {
#pragma unroll 2
                    for (int c = lane; c < ncol; c += 32, vp += 512, mp += 32 * MB, xp += 512) {
                        uint32_t xw[B][XR];
#pragma unroll
                        for (int b = 0; b < B; ++b)
#pragma unroll
                            for (int u = 0; u < XV; ++u) {
                                const uint4 t = *reinterpret_cast<const uint4 *>(
                                    xp + (b * XV + u) * xstride);
                                xw[b][4 * u + 0] = t.x;
                                xw[b][4 * u + 1] = t.y;
                                xw[b][4 * u + 2] = t.z;
                                xw[b][4 * u + 3] = t.w;
                            }
#pragma unroll
                        for (int i = 0; i < R; ++i) {
                            const uint4 v = *reinterpret_cast<const uint4 *>(vp + i * seg_v);
                            const mask_t m = *reinterpret_cast<const mask_t *>(mp + i * seg_m);
                            const typename P::Sel sel = P::decode_tab(m, tab);
#pragma unroll
                            for (int b = 0; b < B; ++b)
                                acc[i * B + b] = P::dot(v, sel, xw[b], acc[i * B + b]);
                        }
                    }
                } else {
                    // Three or more vectors: decode the R rows' chunks once,
                    // then take the vectors BG at a time (x of BG vectors,
                    // at most 32 words, in registers at once), each x unit
                    // read once for R rows.
                    constexpr int BG = B < 32 / XR ? B : (32 / XR > 0 ? 32 / XR : 1);
                    const uint8_t *xq = xs + (cs + lane) * (XCU * 16);  // column-major x
                    for (int c = lane; c < ncol;
                         c += 32, vp += 512, mp += 32 * MB, xq += 32 * XCU * 16) {
                        uint4 v[R];
                        typename P::Sel sel[R];
#pragma unroll
                        for (int i = 0; i < R; ++i) {
                            v[i] = *reinterpret_cast<const uint4 *>(vp + i * seg_v);
                            sel[i] = P::decode_tab(*reinterpret_cast<const mask_t *>(mp + i * seg_m),
                                                   tab);
                        }
#pragma unroll
                        for (int b0 = 0; b0 < B; b0 += BG) {
                            uint32_t xw[BG][XR];
#pragma unroll
                            for (int bb = 0; bb < BG; ++bb)
#pragma unroll
                                for (int u = 0; u < XV; ++u) {
                                    if (b0 + bb < B) {
                                        const uint4 t = *reinterpret_cast<const uint4 *>(
                                            xq + ((b0 + bb) * XV + u) * 16);
                                        xw[bb][4 * u + 0] = t.x;
                                        xw[bb][4 * u + 1] = t.y;
                                        xw[bb][4 * u + 2] = t.z;
                                        xw[bb][4 * u + 3] = t.w;
                                    }
                                }
#pragma unroll
                            for (int i = 0; i < R; ++i)
#pragma unroll
                                for (int bb = 0; bb < BG; ++bb)
                                    if (b0 + bb < B)
                                        acc[i * B + b0 + bb] =
                                            P::dot(v[i], sel[i], xw[bb], acc[i * B + b0 + bb]);
                        }
                    }
                }
                // Every lane has read the slot: refill it with this warp's
                // task SW ahead (generic-proxy reads, then async-proxy
                // writes of the same bytes: fence between them).
                __syncwarp();
                if (lane == 0 && issued < ncopy && !failed) {
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    issue_next(sv, &my_full[slot]);
                }
                if (++slot == a.SW) {
                    slot = 0;
                    phase ^= 1u;
                }
            }

            warp_reduce_scatter<V>(acc, lane);
            const int idx = lane >> SH;
            const bool lead = (lane & ((1 << SH) - 1)) == 0;
            // sums held: nr rows x B vectors, or for a pair the gate and the
            // up sum of one row (index i = 0, 1) per vector
            const int nsum = (a.pair ? 2 : nr) * B;
            const int i = idx / B, b = idx - (idx / B) * B;
            float tot = acc[0];
            if (a.ktiles > 1 && lead && idx < nsum) {
                float *cp = carry + ((a.pair ? 2 * i0 : i0) + i) * B + b;
                if (kt > 0) tot += *cp;
                *cp = tot;
            }
            if (R == 2 && a.pair) {
                // the up sum of vector b sits B places further on
                const float up = __shfl_sync(0xffffffffu, tot, ((idx + B) << SH) & 31);
                if (kt == a.ktiles - 1 && lead && idx < B)
                    store_y(mt.y, b * mt.ldy + r_begin + i0, tot / (1.0f + expf(-tot)) * up,
                            a.y_f32 != 0);
            } else if (kt == a.ktiles - 1 && lead && idx < nsum) {
                store_y(mt.y, b * mt.ldy + r_begin + i0 + i, tot, a.y_f32 != 0);
            }
        }
    }
    // After a timeout, copies this warp issued may still be landing in its
    // slots: wait for them (again with a limit) before the CTA can exit.
    if (failed && lane == 0)
        for (int p = j; p < issued; ++p)
            if (!mbar_wait(&my_full[p % a.SW], (p / a.SW) & 1)) break;
}

// ---------------------------------------------------------------- host side

struct RowsPlan {
    int W, R, ktiles, tile_chunks, seg_chunks, nseg, nseg_last, SW, grid;
    int seg_v, seg_m, stage_bytes, xbuf_bytes, off_x, off_bar, off_tab, off_carry;
    size_t smem;
};

// Chooses rows per task, K tile, warps and slots per warp for a shape;
// false if nothing fits in shared memory (the caller then takes another
// kernel).  rows_plan_group does the same for `count` matrices with the same
// K in one launch and writes each matrix's first CTA to cta_begin[0..count].
// max_warps caps the warps per CTA; tab_bytes is the pattern's shared decode
// table (Pattern<N, M>::kTabWords words).
bool rows_plan(int64_t rows, int chunks, int CK, int B, int nsm, int max_smem, int max_warps,
               RowsPlan *out, bool pair = false, int tab_bytes = 0);
bool rows_plan_group(const int64_t *rows, int count, int chunks, int CK, int B, int nsm,
                     int max_smem, int max_warps, RowsPlan *out, int *cta_begin,
                     int tab_bytes = 0);

// Shared memory and registers one CTA may take so that two fit on an SM
// (cached per device); false if the device cannot say.
bool rows_pair_limits(int *smem_per_cta, int *regs_per_cta);

template <int N, int M, int B, int R>
cudaError_t launch_rows_instance(const SpmvGroup &g, const RowsPlan &pl, const int *cta_begin,
                                 cudaStream_t s)
{
    auto kernel = nm_spmv_rows_kernel<N, M, B, R>;
    static std::atomic<int> smem_set[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int need = static_cast<int>(pl.smem);
    if (dev < 0 || dev >= 64 || need > smem_set[dev].load(std::memory_order_relaxed)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, need);
        if (e != cudaSuccess) return e;
        // Every instance asks for the same (largest) shared-memory carve-out,
        // so CTAs of consecutive calls never wait for an SM to be
        // reconfigured before they can share it.
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) {
            int cur = smem_set[dev].load(std::memory_order_relaxed);
            while (need > cur && !smem_set[dev].compare_exchange_weak(cur, need)) {
            }
        }
    }
    using P = Pattern<N, M>;
    const SpmvProblem &p0 = g.p[0];
    RowsArgs a = {};
    const int nmat = g.pair ? 1 : g.count;  // a pair is one matrix entry (gate) plus up's arrays
    for (int i = 0; i < nmat; ++i) {
        const SpmvProblem &p = g.p[i];
        RowsMat &m = a.mat[i];
        m.values = static_cast<const uint8_t *>(p.values);
        m.masks = reinterpret_cast<const uint8_t *>(p.masks);
        m.x = static_cast<const __half *>(p.x);
        m.y = p.y;
        m.ldy = p.ldy;
        a.cta_begin[i] = cta_begin[i];
        const int ctas = cta_begin[i + 1] - cta_begin[i];
        m.row_base = static_cast<int>(p.rows / ctas);
        m.row_extra = static_cast<int>(p.rows % ctas);
    }
    if (g.pair) {
        a.mat[0].values2 = static_cast<const uint8_t *>(g.p[1].values);
        a.mat[0].masks2 = reinterpret_cast<const uint8_t *>(g.p[1].masks);
    }
    a.pair = g.pair ? 1 : 0;
    a.nmat = nmat;
    a.cta_begin[nmat] = cta_begin[nmat];
    a.err = p0.err;
    a.ldx = p0.ldx;
    a.vrow_bytes = p0.K / P::CK * 16;
    a.mrow_bytes = ((p0.K + 31) / 32) * 4;
    a.chunks = static_cast<int>(p0.K / P::CK);
    a.tile_chunks = pl.tile_chunks;
    a.ktiles = pl.ktiles;
    a.seg_chunks = pl.seg_chunks;
    a.nseg = pl.nseg;
    a.nseg_last = pl.nseg_last;
    a.SW = pl.SW;
    a.pre = std::min(bulk_tuning().rows_pre, pl.SW);
    a.pre_warps = bulk_tuning().rows_prew;
    // L2 warm-up only where the CTA consumes its rows in address order (one K tile)
    a.l2pre_rows = pl.ktiles == 1 ? static_cast<int>(bulk_tuning().rows_l2pre_bytes /
                                                     (a.vrow_bytes + a.mrow_bytes))
                                  : 0;
    a.seg_v = pl.seg_v;
    a.seg_m = pl.seg_m;
    a.stage_bytes = pl.stage_bytes;
    a.xbuf_bytes = pl.xbuf_bytes;
    a.off_x = pl.off_x;
    a.off_bar = pl.off_bar;
    a.off_tab = pl.off_tab;
    a.off_carry = pl.off_carry;
    a.y_f32 = p0.y_f32 ? 1 : 0;
    // the time-out test: no copies, and a 2 ms limit on the waits that then
    // cannot complete
    a.no_copy = bulk_tuning().wait_fault_test ? 1 : 0;
    a.wait_limit_ns = bulk_tuning().wait_fault_test ? 2000000ull : kWaitLimitNs;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cta_begin[nmat]);
    cfg.blockDim = dim3(32 * pl.W);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = bulk_tuning().pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

// Registers per thread of one kernel instance (0 if unknown).
template <int N, int M, int B, int R>
int rows_instance_regs()
{
    static std::atomic<int> regs{-1};
    int r = regs.load(std::memory_order_relaxed);
    if (r < 0) {
        cudaFuncAttributes fa;
        r = cudaFuncGetAttributes(&fa, nm_spmv_rows_kernel<N, M, B, R>) == cudaSuccess
                ? fa.numRegs : 0;
        regs.store(r, std::memory_order_relaxed);
    }
    return r;
}

template <int N, int M, int B>
int rows_regs(int R)
{
    switch (R) {
    case 1: return rows_instance_regs<N, M, B, 1>();
    case 2: return rows_instance_regs<N, M, B, 2>();
    case 4:
        if constexpr (rows_rmax(B) >= 4) return rows_instance_regs<N, M, B, 4>();
        return 0;
    default: return 0;
    }
}

template <int N, int M>
int rows_regs_any(int B, int R)
{
    switch (B) {
    case 1: return rows_regs<N, M, 1>(R);
    case 2: return rows_regs<N, M, 2>(R);
    case 3: return rows_regs<N, M, 3>(R);
    case 4: return rows_regs<N, M, 4>(R);
    case 5: return rows_regs<N, M, 5>(R);
    case 6: return rows_regs<N, M, 6>(R);
    case 7: return rows_regs<N, M, 7>(R);
    case 8: return rows_regs<N, M, 8>(R);
    default: return 0;
    }
}

template <int N, int M, int B>
cudaError_t launch_rows_b(const SpmvGroup &g, const RowsPlan &pl, const int *cta_begin,
                          cudaStream_t s)
{
    switch (pl.R) {
    case 1: return launch_rows_instance<N, M, B, 1>(g, pl, cta_begin, s);
    case 2: return launch_rows_instance<N, M, B, 2>(g, pl, cta_begin, s);
    case 4:
        if constexpr (rows_rmax(B) >= 4) return launch_rows_instance<N, M, B, 4>(g, pl, cta_begin, s);
        return cudaErrorNotSupported;
    default: return cudaErrorNotSupported;
    }
}

// Batch 1 to 8; cudaErrorNotSupported (nothing launched) otherwise or
// when no plan fits.  All problems of the group share N, M, K, batch, ldx
// and the y type.
template <int N, int M>
cudaError_t launch_rows_pattern(const SpmvGroup &g, cudaStream_t s)
{
    using P = Pattern<N, M>;
    const SpmvProblem &p0 = g.p[0];
    if (p0.batch < 1 || p0.batch > NM_MAX_BATCH || g.count < 1 || g.count > kRowsMaxGroup)
        return cudaErrorNotSupported;
    const int nsm = sm_count();
    if (nsm <= 0) return cudaErrorInvalidDevice;
    const int max_smem = max_dynamic_smem();
    if (max_smem <= 0) return cudaErrorInvalidDevice;
    RowsPlan pl;
    int cta_begin[kRowsMaxGroup + 1];
    const int chunks = static_cast<int>(p0.K / P::CK);
    int64_t rows[kRowsMaxGroup];
    for (int i = 0; i < g.count; ++i) rows[i] = g.p[i].rows;
    if (g.pair && (g.count != 2 || g.p[1].rows != p0.rows)) return cudaErrorNotSupported;
    auto plan = [&](int smem_cap, int max_warps) {
        if (g.count == 1 || g.pair) {
            if (!rows_plan(p0.rows, chunks, P::CK, p0.batch, nsm, smem_cap, max_warps, &pl,
                           g.pair, 4 * P::kTabWords))
                return false;
            cta_begin[0] = 0;
            cta_begin[1] = pl.grid;
            return true;
        }
        return rows_plan_group(rows, g.count, chunks, P::CK, p0.batch, nsm, smem_cap, max_warps,
                               &pl, cta_begin, 4 * P::kTabWords);
    };
    // Half an SM per CTA when the plan allows it (the warp cap follows from
    // the chosen instance's registers, allocated 8 a thread at a time);
    // otherwise the whole SM.
    bool planned = false;
    int pair_smem = 0, pair_regs = 0;
    if (bulk_tuning().rows_pair && bulk_tuning().ctas_per_sm == 1 &&
        rows_pair_limits(&pair_smem, &pair_regs)) {
        int max_warps = kRowsMaxWarps;
        for (int attempt = 0; attempt < 3 && !planned; ++attempt) {
            if (!plan(std::min(pair_smem, max_smem), max_warps)) break;
            const int regs = rows_regs_any<N, M>(p0.batch, pl.R);
            if (regs <= 0) break;
            const int fit = pair_regs / (32 * ((regs + 7) / 8 * 8));
            if (pl.W <= fit) planned = true;
            else if (fit < 4) break;
            else max_warps = fit;
        }
    }
    if (!planned && !plan(max_smem, kRowsMaxWarps)) return cudaErrorNotSupported;
    switch (p0.batch) {
    case 1: return launch_rows_b<N, M, 1>(g, pl, cta_begin, s);
    case 2: return launch_rows_b<N, M, 2>(g, pl, cta_begin, s);
    case 3: return launch_rows_b<N, M, 3>(g, pl, cta_begin, s);
    case 4: return launch_rows_b<N, M, 4>(g, pl, cta_begin, s);
    case 5: return launch_rows_b<N, M, 5>(g, pl, cta_begin, s);
    case 6: return launch_rows_b<N, M, 6>(g, pl, cta_begin, s);
    case 7: return launch_rows_b<N, M, 7>(g, pl, cta_begin, s);
    case 8: return launch_rows_b<N, M, 8>(g, pl, cta_begin, s);
    default: return cudaErrorNotSupported;
    }
}

}  // namespace nm

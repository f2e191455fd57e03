// Vectorised N:M SpMV kernel (direct loads) and the mask-decode patterns
// shared by every vectorised kernel, for sm_103a.
//
// The operation is the N:M sparse matrix-vector product with bitmask
// indexing and fixed-step traversal of "SparseDecoding: Decoding-Aware
// Pruning for Accurate and Efficient LLM Inference" (Abstract).  It is a
// pure HBM stream: every kept value (2 bytes) and mask bit is read exactly
// once per call, so the kernel is designed around bytes in flight and
// issue slots, not around arithmetic.
//
// Work decomposition.
//   * A 16-byte "chunk" of a row's values holds 8 kept fp16 weights, i.e.
//     8/N groups spanning CK = 8*M/N positions along K; its mask bits are
//     the CK consecutive bits at bit offset c*CK of the row's mask words.
//   * A block of KW warps owns a contiguous range of rows.  Thread t of the
//     block owns chunks c = kt*T + j*blockDim.x + t (j < CPL, T = CPL *
//     blockDim.x) of every row, for each K tile kt.  It keeps the matching
//     slice of x (CK fp16 per chunk and vector) in registers for the whole
//     tile, so x is read from memory once per block and tile, not per row.
//   * Rows are processed R at a time: all R*CPL chunk loads (16 B values +
//     CK/8 B of mask) are issued before any is used, giving each thread
//     R*CPL independent 16-byte loads in flight.
//   * Mask decode in registers (Pattern<N, M> below: byte-permute lookup
//     tables for 2:4 and 1:4, one find-leading-one per kept position for the
//     8-wide patterns), and a byte permute gathers the matching fp16 x lanes
//     into a half2 next to the value pair.  Products use fp16 x fp16 -> fp32
//     FMA.
// This kernel loads with plain 128-bit loads and is the path for K not a
// multiple of 128; the bulk-staged kernels (nm_rows.cuh, nm_bulk.cuh) take
// the other shapes.
//   * Each warp reduces its R*B partial sums with a reduce-scatter butterfly
//     (V-1 shuffles for V sums), warps combine through shared memory, and
//     the totals are rounded once into y (or carried to the next K tile in
//     shared memory when the row needs more than one tile).
#pragma once

#include <cuda_runtime.h>

#include <atomic>

#include "nm_device.cuh"
#include "nm_internal.h"

namespace nm {

// ---------------------------------------------------------------- patterns
// Pattern<N, M> consumes one 16-byte chunk of kept values (8 fp16 = 8/N
// groups spanning CK = 8*M/N positions along K) and its CK mask bits.
//   decode(m) -> Sel: everything that depends on the mask alone (the byte
//                permute selectors that gather the x lanes of the kept
//                positions); done once per chunk and shared by all vectors.
//   dot(v, sel, x, acc): acc + the products of the 8 values with the
//                matching x lanes, x = the chunk's CK fp16 activations
//                packed two per word (XR = CK/2 words).
// Results for groups without exactly N set bits are unspecified; the mask
// only ever feeds byte permutes and selects, never an address.
//
//   decode_tab(m, tab): the same Sel, for kernels that hold a per-CTA decode
//                table in shared memory: kTabWords 32-bit words, word i =
//                tab_entry(i).  The 8-wide patterns look each group's byte
//                up in a 256-word table (one shared load replaces a chain of
//                bit scans and selector arithmetic); the others ignore tab.
//                An invalid group byte reads a defined word of the table.

template <int N, int M> struct Pattern;

// For patterns decoded from registers alone.
struct NoTable {
    static constexpr int kTabWords = 0;
    __host__ __device__ static constexpr uint32_t tab_entry(uint32_t) { return 0; }
};

// 2:4 -- four groups per chunk, one value pair per group.  A valid nibble
// has exactly two set bits, so its low three bits already identify it; two
// 8-entry byte tables (held in immediates, indexed by byte permutes) map
// those bits to the selector bytes of the first and second kept lane.
template <> struct Pattern<2, 4> : NoTable {
    static constexpr int CK = 16;
    using mask_t = uint16_t;
    struct Sel { uint32_t s[4]; };
    __host__ __device__ static __forceinline__ Sel decode(uint32_t m)
    {
        const uint32_t idx = m & 0x7777u;
        const uint32_t first = prmt(0x10321010u, 0x10321054u, idx);   // lane of the lower kept k
        const uint32_t second = prmt(0x32767676u, 0x76545476u, idx);  // lane of the upper kept k
        const uint32_t s01 = prmt(first, second, 0x5140u);
        const uint32_t s23 = prmt(first, second, 0x7362u);
        return Sel{{s01, s01 >> 16, s23, s23 >> 16}};
    }
    __host__ __device__ static __forceinline__ Sel decode_tab(uint32_t m, const uint32_t *)
    {
        return decode(m);
    }
    __host__ __device__ static __forceinline__ float dot(const uint4 &v, const Sel &sel, const uint32_t *x,
                                                float acc)
    {
        acc = fma_h2(v.x, prmt(x[0], x[1], sel.s[0]), acc);
        acc = fma_h2(v.y, prmt(x[2], x[3], sel.s[1]), acc);
        acc = fma_h2(v.z, prmt(x[4], x[5], sel.s[2]), acc);
        return fma_h2(v.w, prmt(x[6], x[7], sel.s[3]), acc);
    }
};

// 1:4 -- eight groups per chunk; a value pair spans two groups.  A valid
// nibble has one set bit and its low three bits identify it (8 -> 0).
template <> struct Pattern<1, 4> : NoTable {
    static constexpr int CK = 32;
    using mask_t = uint32_t;
    struct Sel { uint32_t s[4]; };
    __host__ __device__ static __forceinline__ Sel decode(uint32_t m)
    {
        const uint32_t lo = prmt(0x10321076u, 0x10101054u, m & 0x7777u);
        const uint32_t hi = prmt(0x10321076u, 0x10101054u, (m >> 16) & 0x7777u);
        return Sel{{lo, lo >> 16, hi, hi >> 16}};
    }
    __host__ __device__ static __forceinline__ Sel decode_tab(uint32_t m, const uint32_t *)
    {
        return decode(m);
    }
    __host__ __device__ static __forceinline__ float dot(const uint4 &v, const Sel &sel, const uint32_t *x,
                                                float acc)
    {
        const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            // low half: lane of group 2q; high half: lane of group 2q+1
            const uint32_t a = prmt(x[4 * q], x[4 * q + 1], sel.s[q]);
            const uint32_t b = prmt(x[4 * q + 2], x[4 * q + 3], sel.s[q]);
            acc = fma_h2(vw[q], prmt(a, b, 0x7610u), acc);
        }
        return acc;
    }
};

// Selector pair that gathers fp16 lanes pa and pb (0..7) of four words with
// gather8(): a permute of words 0-1 and one of words 2-3 by the lanes'
// positions within a half, then a permute picking the half each lives in.
struct Pair8 { uint32_t s, pick; };
__host__ __device__ __forceinline__ Pair8 pair8(uint32_t pa, uint32_t pb)
{
    // Both selectors at once from q = pa | pb << 8: the within-half lane of
    // each (bits 0-1 of each byte) scales the sel_pair step 0x22, the half
    // (bit 2) scales the step 0x44 that moves a pick from lo's bytes to hi's.
    const uint32_t q = pa | (pb << 8);
    return Pair8{0x1010u + 0x22u * (q & 0x0303u), 0x3210u + 0x44u * ((q >> 2) & 0x0101u)};
}
__host__ __device__ __forceinline__ uint32_t gather8(const uint32_t *xg, const Pair8 &p)
{
    return prmt(prmt(xg[0], xg[1], p.s), prmt(xg[2], xg[3], p.s), p.pick);
}
// Position of the lowest / highest set bit of a nonzero byte (one
// find-leading-one each; the lowest set bit is isolated with b & -b).
__host__ __device__ __forceinline__ uint32_t lowest(uint32_t b) { return msb(b & (0u - b)); }

// 2:8 -- four groups of 8 per chunk, one value pair per group.  Table word
// g(b) = b ^ (b >> 1): the gather selectors of the lowest and the highest
// set bit of b, s in bits 0-15 and pick in bits 16-31.  Indexed by b itself
// the 28 valid bytes would crowd into six of the 32 shared-memory banks (3
// to a bank); their Gray codes g(b) fall at most 2 to a bank, and one shift
// and one logic op give g of all four group bytes of a chunk at once.
template <> struct Pattern<2, 8> {
    static constexpr int CK = 32;
    using mask_t = uint32_t;
    struct Sel { Pair8 p[4]; };
    static constexpr int kTabWords = 256;
    __host__ __device__ static __forceinline__ Sel decode(uint32_t m)
    {
        Sel s;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const uint32_t b = (m >> (8 * g)) & 0xFFu;
            s.p[g] = pair8(lowest(b), msb(b));
        }
        return s;
    }
    // word i of the table: the entry of the byte whose Gray code is i
    __host__ __device__ static uint32_t tab_entry(uint32_t i)
    {
        uint32_t b = i;  // inverse Gray code of an 8-bit value
        b ^= b >> 1;
        b ^= b >> 2;
        b ^= b >> 4;
        const Pair8 p = b ? pair8(lowest(b), msb(b)) : pair8(0, 0);
        return p.s | (p.pick << 16);
    }
    __host__ __device__ static __forceinline__ Sel decode_tab(uint32_t m, const uint32_t *tab)
    {
        // Gray code of each byte: the bit shifted in from the next byte is
        // masked off
        const uint32_t gm = m ^ ((m >> 1) & 0x7F7F7F7Fu);
        Sel s;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const uint32_t e = tab[(gm >> (8 * g)) & 0xFFu];
            s.p[g] = Pair8{e, e >> 16};
        }
        return s;
    }
    __host__ __device__ static __forceinline__ float dot(const uint4 &v, const Sel &sel, const uint32_t *x,
                                                float acc)
    {
        const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int g = 0; g < 4; ++g) acc = fma_h2(vw[g], gather8(x + 4 * g, sel.p[g]), acc);
        return acc;
    }
};

// 4:8 -- two groups of 8 per chunk, two value pairs per group: the two
// lowest and the two highest kept positions.  Table word b: the positions
// of the (up to) four lowest set bits of b, one a byte in increasing order
// (0 for missing ones); the selectors of both pairs follow from it with two
// masked multiplies, since selector byte j of a gather is 0x10 + 0x22 *
// (p_j & 3) and pick byte j is its base + 0x44 * (p_j >> 2).
template <> struct Pattern<4, 8> {
    static constexpr int CK = 16;
    using mask_t = uint16_t;
    struct Sel { Pair8 p[4]; };
    static constexpr int kTabWords = 256;
    __host__ __device__ static __forceinline__ Sel decode(uint32_t m)
    {
        Sel s;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            const uint32_t b = (m >> (8 * g)) & 0xFFu;
            const uint32_t p0 = lowest(b);
            const uint32_t p1 = lowest(b & (b - 1u));
            const uint32_t p3 = msb(b);
            const uint32_t p2 = msb(b & ~(1u << p3));
            s.p[2 * g] = pair8(p0, p1);
            s.p[2 * g + 1] = pair8(p2, p3);
        }
        return s;
    }
    __host__ __device__ static uint32_t tab_entry(uint32_t b)
    {
        uint32_t q = 0;
        for (int n = 0; n < 4 && b != 0; ++n) {
            q |= lowest(b) << (8 * n);
            b &= b - 1u;
        }
        return q;
    }
    __host__ __device__ static __forceinline__ Sel decode_tab(uint32_t m, const uint32_t *tab)
    {
        Sel s;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            const uint32_t q = tab[(m >> (8 * g)) & 0xFFu];
            const uint32_t sel = (q & 0x03030303u) * 0x22u + 0x10101010u;
            const uint32_t pick = (q & 0x04040404u) * 0x11u + 0x32103210u;
            s.p[2 * g] = Pair8{sel, pick};
            s.p[2 * g + 1] = Pair8{sel >> 16, pick >> 16};
        }
        return s;
    }
    __host__ __device__ static __forceinline__ float dot(const uint4 &v, const Sel &sel, const uint32_t *x,
                                                float acc)
    {
        acc = fma_h2(v.x, gather8(x, sel.p[0]), acc);
        acc = fma_h2(v.y, gather8(x, sel.p[1]), acc);
        acc = fma_h2(v.z, gather8(x + 4, sel.p[2]), acc);
        return fma_h2(v.w, gather8(x + 4, sel.p[3]), acc);
    }
};

// 1:8 -- eight groups of 8 per chunk; a value pair spans two groups.  The
// single set bit of a group is its highest.
template <> struct Pattern<1, 8> : NoTable {
    static constexpr int CK = 64;
    using mask_t = uint64_t;
    struct Sel { uint32_t pa[4], pb[4]; };
    __host__ __device__ static __forceinline__ Sel decode(uint64_t m)
    {
        Sel s;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t bits = static_cast<uint32_t>(m >> (16 * q));
            s.pa[q] = msb(bits & 0xFFu);
            s.pb[q] = msb((bits >> 8) & 0xFFu);
        }
        return s;
    }
    __host__ __device__ static __forceinline__ Sel decode_tab(uint64_t m, const uint32_t *)
    {
        return decode(m);
    }
    __host__ __device__ static __forceinline__ float dot(const uint4 &v, const Sel &sel, const uint32_t *x,
                                                float acc)
    {
        const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t pa = sel.pa[q], pb = sel.pb[q];
            const uint32_t *xa = x + 8 * q;      // group 2q: 8 fp16 in 4 words
            const uint32_t *xb = x + 8 * q + 4;  // group 2q+1
            const uint32_t ia = (pa >> 1) & 3u, ib = (pb >> 1) & 3u;
            const uint32_t ra = (ia & 2u) ? ((ia & 1u) ? xa[3] : xa[2]) : ((ia & 1u) ? xa[1] : xa[0]);
            const uint32_t rb = (ib & 2u) ? ((ib & 1u) ? xb[3] : xb[2]) : ((ib & 1u) ? xb[1] : xb[0]);
            const uint32_t sl = 0x5410u + 0x22u * (pa & 1u) + 0x2200u * (pb & 1u);
            acc = fma_h2(vw[q], prmt(ra, rb, sl), acc);
        }
        return acc;
    }
};

template <int M> struct DensePattern : NoTable {  // N == M: every position kept, mask not consulted
    static constexpr int CK = 8;
    using mask_t = uint8_t;
    struct Sel {};
    __host__ __device__ static __forceinline__ Sel decode(uint32_t) { return Sel{}; }
    __host__ __device__ static __forceinline__ Sel decode_tab(uint32_t, const uint32_t *) { return Sel{}; }
    __host__ __device__ static __forceinline__ float dot(const uint4 &v, const Sel &, const uint32_t *x,
                                                float acc)
    {
        acc = fma_h2(v.x, x[0], acc);
        acc = fma_h2(v.y, x[1], acc);
        acc = fma_h2(v.z, x[2], acc);
        return fma_h2(v.w, x[3], acc);
    }
};
template <> struct Pattern<4, 4> : DensePattern<4> {};
template <> struct Pattern<8, 8> : DensePattern<8> {};

template <typename T> __device__ __forceinline__ T ld_mask(const uint8_t *p);
template <> __device__ __forceinline__ uint8_t ld_mask<uint8_t>(const uint8_t *p)
{
    return static_cast<uint8_t>(ld_stream_u8(p));
}
template <> __device__ __forceinline__ uint16_t ld_mask<uint16_t>(const uint8_t *p)
{
    return static_cast<uint16_t>(ld_stream_u16(reinterpret_cast<const uint16_t *>(p)));
}
template <> __device__ __forceinline__ uint32_t ld_mask<uint32_t>(const uint8_t *p)
{
    return ld_stream_u32(reinterpret_cast<const uint32_t *>(p));
}
template <> __device__ __forceinline__ uint64_t ld_mask<uint64_t>(const uint8_t *p)
{
    return ld_stream_u64(reinterpret_cast<const uint64_t *>(p));
}

// ---------------------------------------------------------------- kernel

struct FastArgs {
    const uint4 *values;   // [rows][chunks] 16-byte chunks
    const uint8_t *masks;  // row stride mrow_bytes
    const __half *x;       // [B][ldx]
    void *y;               // [B][ldy]
    int64_t ldx, ldy, mrow_bytes;
    int rows, chunks, ktiles;
    int row_base, row_extra;  // block b owns row_base (+1 if b < row_extra) rows
    int y_f32;
};

// Rows per tile: keep about 8 (B <= 2) or 4 (B > 2) chunk loads per thread
// in flight and at most 32 partial sums per lane.
__host__ __device__ constexpr int rows_per_tile(int B, int CPL)
{
    int r = ((B <= 2) ? 8 : 4) / CPL;
    r = r < 1 ? 1 : r;
    while (r > 1 && r * B > 32) r /= 2;
    return r;
}

constexpr int kMaxWarps = 16;

template <int N, int M, int B, int CPL>
__global__ void __launch_bounds__(kMaxWarps * 32)
nm_spmv_fast_kernel(const FastArgs a)
{
    using P = Pattern<N, M>;
    using mask_t = typename P::mask_t;
    constexpr int CK = P::CK;
    constexpr int XR = CK / 2;   // x words per chunk and vector
    constexpr int XV = CK / 8;   // 16-byte x loads per chunk and vector
    constexpr int R = rows_per_tile(B, CPL);
    constexpr int V = pow2_ceil(R * B);
    constexpr int MB = CK / 8;   // mask bytes per chunk

    extern __shared__ float smem[];
    const int KW = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    float *part = smem;               // [2][KW][V]
    float *carry = smem + 2 * KW * V;  // [rows of block][B], only with ktiles > 1

    const int bid = blockIdx.x;
    const int r_begin = bid * a.row_base + min(bid, a.row_extra);
    const int r_count = a.row_base + (bid < a.row_extra ? 1 : 0);
    const int tile_w = CPL * blockDim.x;
    int buf = 0;

    for (int kt = 0; kt < a.ktiles; ++kt) {
        int cj[CPL];
        bool okj[CPL];
        uint32_t xr[CPL][B][XR];
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            cj[j] = kt * tile_w + j * blockDim.x + threadIdx.x;
            okj[j] = cj[j] < a.chunks;
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const uint4 *xp = reinterpret_cast<const uint4 *>(
                    a.x + b * a.ldx + static_cast<int64_t>(cj[j]) * CK);
#pragma unroll
                for (int u = 0; u < XV; ++u) {
                    const uint4 t = okj[j] ? ld_keep_v4(xp + u) : make_uint4(0, 0, 0, 0);
                    xr[j][b][4 * u + 0] = t.x;
                    xr[j][b][4 * u + 1] = t.y;
                    xr[j][b][4 * u + 2] = t.z;
                    xr[j][b][4 * u + 3] = t.w;
                }
            }
        }

        for (int rt = 0; rt < r_count; rt += R) {
            uint4 v[R][CPL];
            mask_t m[R][CPL];
#pragma unroll
            for (int i = 0; i < R; ++i) {
                const bool rok = rt + i < r_count;
                const int64_t row = r_begin + rt + i;
#pragma unroll
                for (int j = 0; j < CPL; ++j) {
                    if (rok && okj[j]) {
                        v[i][j] = ld_stream_v4(a.values + row * a.chunks + cj[j]);
                        m[i][j] = ld_mask<mask_t>(a.masks + row * a.mrow_bytes +
                                                  static_cast<int64_t>(cj[j]) * MB);
                    } else {
                        v[i][j] = make_uint4(0, 0, 0, 0);
                        m[i][j] = static_cast<mask_t>(~static_cast<mask_t>(0));
                    }
                }
            }

            float acc[V];
#pragma unroll
            for (int t = 0; t < V; ++t) acc[t] = 0.f;
#pragma unroll
            for (int i = 0; i < R; ++i)
#pragma unroll
                for (int j = 0; j < CPL; ++j) {
                    const typename P::Sel sel = P::decode(m[i][j]);
#pragma unroll
                    for (int b = 0; b < B; ++b)
                        acc[i * B + b] = P::dot(v[i][j], sel, xr[j][b], acc[i * B + b]);
                }

            warp_reduce_scatter<V>(acc, lane);
            constexpr int SH = 5 - log2i<V>();
            if ((lane & ((1 << SH) - 1)) == 0)
                part[(buf * KW + warp) * V + (lane >> SH)] = acc[0];
            __syncthreads();

            if (threadIdx.x < R * B) {
                const int t = threadIdx.x;
                const int i = t / B, b = t - (t / B) * B;
                if (rt + i < r_count) {
                    float tot = 0.f;
                    for (int w = 0; w < KW; ++w) tot += part[(buf * KW + w) * V + t];
                    if (a.ktiles > 1) {
                        float *c = carry + (rt + i) * B + b;
                        if (kt > 0) tot += *c;
                        *c = tot;
                    }
                    if (kt == a.ktiles - 1)
                        store_y(a.y, b * a.ldy + r_begin + rt + i, tot, a.y_f32 != 0);
                }
            }
            buf ^= 1;
        }
        // The carry slot of (row, vector) is read and written only by thread
        // row_in_tile * B + vector, so K tiles need no extra barrier.
    }
}

// ---------------------------------------------------------------- host side

struct FastTiling {
    int cpl, kw, ktiles;
};

// Choose chunks-per-thread and warps-per-block so that one K tile covers a
// row where possible, with few idle lanes and at most kMaxWarps warps.
inline FastTiling choose_tiling(int chunks, int batch)
{
    // Larger batches hold B copies of the x slice in registers: keep one
    // chunk per thread from B = 5 on so that nothing spills.
    static const int cpl_b1[] = {1, 2, 4};
    static const int cpl_bn[] = {1, 2};
    const int *cpls = batch == 1 ? cpl_b1 : cpl_bn;
    const int ncpl = batch == 1 ? 3 : (batch <= 4 ? 2 : 1);
    FastTiling best = {1, 1, 1};
    double best_cost = 1e30;
    for (int ci = 0; ci < ncpl; ++ci) {
        const int cpl = cpls[ci];
        for (int kw = 1; kw <= kMaxWarps; ++kw) {
            const long tile = 32L * kw * cpl;
            const long nt = (chunks + tile - 1) / tile;
            const double idle = double(nt * tile - chunks) / double(nt * tile);
            double cost = 4.0 * idle + 0.05 * double(nt - 1) + 0.01 * cpl;
            if (kw < 4 && chunks > 32L * kw * cpl) cost += 0.1;  // prefer >= 4 warps
            if (cost < best_cost - 1e-12) {
                best_cost = cost;
                best = {cpl, kw, static_cast<int>(nt)};
            }
        }
    }
    return best;
}

template <int N, int M, int B, int CPL>
cudaError_t launch_fast_instance(const SpmvProblem &p, const FastTiling &t, cudaStream_t s)
{
    constexpr int R = rows_per_tile(B, CPL);
    constexpr int V = pow2_ceil(R * B);
    auto kernel = nm_spmv_fast_kernel<N, M, B, CPL>;
    const int threads = 32 * t.kw;
    const int nsm = sm_count();
    if (nsm <= 0) return cudaErrorInvalidDevice;

    static std::atomic<int> occ_cache[kMaxWarps + 1];
    const size_t part_bytes = sizeof(float) * 2 * t.kw * V;
    int occ = occ_cache[t.kw].load(std::memory_order_relaxed);
    if (occ <= 0) {
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, threads,
                                                                      part_bytes);
        if (e != cudaSuccess) return e;
        if (occ <= 0) return cudaErrorInvalidConfiguration;
        occ_cache[t.kw].store(occ, std::memory_order_relaxed);
    }
    const int rows = static_cast<int>(p.rows);
    int grid = occ * nsm;
    if (grid > rows) grid = rows;
    size_t smem = part_bytes;
    if (t.ktiles > 1) {
        // Partial sums carried across K tiles live in shared memory; keep them
        // under 96 KB by giving each block fewer rows (more blocks) if needed.
        const long max_rows = (96L * 1024) / (sizeof(float) * B);
        const long need = (rows + max_rows - 1) / max_rows;
        if (grid < need) grid = static_cast<int>(need);
        const long rpb = (rows + grid - 1) / grid;
        smem += sizeof(float) * B * rpb;
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem));
            if (e != cudaSuccess) return e;
        }
    }
    using P = Pattern<N, M>;
    FastArgs a;
    a.values = static_cast<const uint4 *>(p.values);
    a.masks = reinterpret_cast<const uint8_t *>(p.masks);
    a.x = static_cast<const __half *>(p.x);
    a.y = p.y;
    a.ldx = p.ldx;
    a.ldy = p.ldy;
    a.mrow_bytes = ((p.K + 31) / 32) * 4;
    a.rows = rows;
    a.chunks = static_cast<int>(p.K / P::CK);
    a.ktiles = t.ktiles;
    a.row_base = rows / grid;
    a.row_extra = rows % grid;
    a.y_f32 = p.y_f32 ? 1 : 0;
    kernel<<<grid, threads, smem, s>>>(a);
    return cudaGetLastError();
}

template <int N, int M, int B>
cudaError_t launch_fast_b(const SpmvProblem &p, const FastTiling &t, cudaStream_t s)
{
    switch (t.cpl) {
    case 1: return launch_fast_instance<N, M, B, 1>(p, t, s);
    case 2:
        if constexpr (B <= 4) return launch_fast_instance<N, M, B, 2>(p, t, s);
        return cudaErrorInvalidConfiguration;
    case 4:
        if constexpr (B == 1) return launch_fast_instance<N, M, B, 4>(p, t, s);
        [[fallthrough]];
    default: return cudaErrorInvalidConfiguration;
    }
}

template <int N, int M>
cudaError_t launch_fast_pattern(const SpmvProblem &p, cudaStream_t s)
{
    const int chunks = static_cast<int>(p.K / Pattern<N, M>::CK);
    const FastTiling t = choose_tiling(chunks, p.batch);
    switch (p.batch) {
    case 1: return launch_fast_b<N, M, 1>(p, t, s);
    case 2: return launch_fast_b<N, M, 2>(p, t, s);
    case 3: return launch_fast_b<N, M, 3>(p, t, s);
    case 4: return launch_fast_b<N, M, 4>(p, t, s);
    case 5: return launch_fast_b<N, M, 5>(p, t, s);
    case 6: return launch_fast_b<N, M, 6>(p, t, s);
    case 7: return launch_fast_b<N, M, 7>(p, t, s);
    case 8: return launch_fast_b<N, M, 8>(p, t, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace nm

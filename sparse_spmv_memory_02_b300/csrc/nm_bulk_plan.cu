// Host-side planning of the bulk-staged SpMV kernels (nm_bulk.cuh and
// nm_rows.cuh): consumer warps, chunk columns per thread or rows per task,
// K tiles, ring depth, and where each piece lives in shared memory.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>

#include "nm_bulk.cuh"
#include "nm_rows.cuh"

namespace nm {

namespace {

BulkTuning parse_tuning()
{
    BulkTuning t;
    const char *env = std::getenv("NM_BULK_TUNE");
    if (!env) return t;
    char buf[256];
    std::strncpy(buf, env, sizeof(buf) - 1);
    buf[sizeof(buf) - 1] = 0;
    char *save = nullptr;
    for (char *tok = strtok_r(buf, ",", &save); tok; tok = strtok_r(nullptr, ",", &save)) {
        char *eq = std::strchr(tok, '=');
        if (!eq) continue;
        *eq = 0;
        const int v = std::atoi(eq + 1);
        if (!std::strcmp(tok, "warps") && v >= 1 && v <= kBulkMaxConsumerWarps) t.warps = v;
        else if (!std::strcmp(tok, "cpl") && v >= 1 && v <= 8) t.cpl = v;
        else if (!std::strcmp(tok, "R") && v >= 1 && v <= 8) t.R = v;
        else if (!std::strcmp(tok, "stage") && v >= 1024) t.stage_bytes = v;
        else if (!std::strcmp(tok, "ring") && v >= 4096) t.ring_bytes = v;
        else if (!std::strcmp(tok, "ctas") && v >= 1 && v <= 4) t.ctas_per_sm = v;
        else if (!std::strcmp(tok, "pdl") && (v == 0 || v == 1)) t.pdl = v;
        else if (!std::strcmp(tok, "rows_warps") && v >= 1 && v <= kRowsMaxWarps) t.rows_warps = v;
        else if (!std::strcmp(tok, "rows_R") && (v == 1 || v == 2 || v == 4)) t.rows_R = v;
        else if (!std::strcmp(tok, "rows_task") && v >= 512) t.rows_task_bytes = v;
        else if (!std::strcmp(tok, "rows_ring") && v >= 4096) t.rows_ring_bytes = v;
        else if (!std::strcmp(tok, "rows_xtile") && v >= 1024) t.rows_xtile_bytes = v;
        else if (!std::strcmp(tok, "rows") && (v == 0 || v == 1)) t.rows_kernel = v;
        else if (!std::strcmp(tok, "rows_pair") && (v == 0 || v == 1)) t.rows_pair = v;
        else if (!std::strcmp(tok, "rows_pre") && v >= 0 && v <= 8) t.rows_pre = v;
        else if (!std::strcmp(tok, "rows_prew") && v >= 0 && v <= 16) t.rows_prew = v;
        else if (!std::strcmp(tok, "rows_two") && v >= -1 && v <= 1) t.rows_two = v;
        else if (!std::strcmp(tok, "wait_fault_test") && (v == 0 || v == 1)) t.wait_fault_test = v;
        else if (!std::strcmp(tok, "tc_sp") && (v == 0 || v == 1)) t.tc_sp = v;
        else if (!std::strcmp(tok, "sp_meta") && (v == 0 || v == 1)) t.sp_meta = v;
        else if (!std::strcmp(tok, "sp_acc") && v >= 1 && v <= 4) t.sp_acc = v;
        else if (!std::strcmp(tok, "sp_mbufs") && v >= 1 && v <= 12) t.sp_mbufs = v;
        else if (!std::strcmp(tok, "sp_sel") && (v == 0 || v == 1)) t.sp_sel = v;
        else if (!std::strcmp(tok, "sp_spin") && (v == 0 || v == 1)) t.sp_spin = v;
        else if (!std::strcmp(tok, "sp_split") && (v == 0 || v == 1)) t.sp_split = v;
        else if (!std::strcmp(tok, "sp_stages") && v >= 0 && v <= 32 && v != 1) t.sp_stages = v;
        else if (!std::strcmp(tok, "sp_tmem") && (v == 256 || v == 512)) t.sp_tmem = v;
        else if (!std::strcmp(tok, "sp_k") && v >= 0 && v <= 8 && v != 1) t.sp_k = v;
        else if (!std::strcmp(tok, "sp_units") && v >= 0) t.sp_units = v;
        else if (!std::strcmp(tok, "sp_group") && (v == 0 || v == 1)) t.sp_group = v;
        else if (!std::strcmp(tok, "rows_l2pre") && v >= 0) t.rows_l2pre_bytes = v;
        else if (!std::strcmp(tok, "tc") && (v == -1 || v == 0 || v == 1)) t.tc = v;
        else if (!std::strcmp(tok, "tc_lbo") && v >= 0 && v < 16384) t.tc_lbo = v;
    }
    return t;
}

int round_up(int v, int a) { return (v + a - 1) / a * a; }

}  // namespace

const BulkTuning &bulk_tuning()
{
    static const BulkTuning t = parse_tuning();
    return t;
}

int spmm_tc_mode(uint32_t *lbo_enc)
{
    const BulkTuning &t = bulk_tuning();
    *lbo_enc = static_cast<uint32_t>(t.tc_lbo);
    return t.tc;
}

int max_dynamic_smem()
{
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (dev >= 0 && dev < 64) {
        const int v = cache[dev].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return -1;
    if (dev >= 0 && dev < 64) cache[dev].store(v, std::memory_order_relaxed);
    return v;
}

bool rows_pair_limits(int *smem_per_cta, int *regs_per_cta)
{
    static std::atomic<int> smem_cache[64], regs_cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return false;
    if (dev < 64 && smem_cache[dev].load(std::memory_order_acquire) > 0) {
        *smem_per_cta = smem_cache[dev].load(std::memory_order_relaxed);
        *regs_per_cta = regs_cache[dev].load(std::memory_order_relaxed);
        return true;
    }
    int per_sm = 0, reserved = 0, regs = 0;
    if (cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&regs, cudaDevAttrMaxRegistersPerMultiprocessor, dev) !=
            cudaSuccess)
        return false;
    const int smem = per_sm / 2 - reserved;
    if (smem <= 0 || regs <= 0) return false;
    if (dev < 64) {
        regs_cache[dev].store(regs / 2, std::memory_order_relaxed);
        smem_cache[dev].store(smem, std::memory_order_release);
    }
    *smem_per_cta = smem;
    *regs_per_cta = regs / 2;
    return true;
}

bool bulk_plan(int64_t rows, int chunks, int CK, int B, int nsm, int max_smem, BulkPlan *out)
{
    const int MB = CK / 8;  // mask bytes per chunk
    if (rows <= 0 || chunks <= 0 || B < 1 || B > 8) return false;
    const BulkTuning &t = bulk_tuning();

    // 1. K tile: consumer warps W and chunk columns per thread.
    double best_cost = 1e30;
    int bw = 0, bc = 0;
    static const int cpls[] = {1, 2, 3, 4, 6, 8};
    for (int cpl : cpls) {
        if (!bulk_cpl_ok(CK, B, cpl) || (t.cpl && cpl != t.cpl)) continue;
        for (int w = 2; w <= kBulkMaxConsumerWarps; ++w) {
            if (t.warps && w != t.warps) continue;
            const long tile = 32L * w * cpl;
            const long nt = (chunks + tile - 1) / tile;
            const double idle = double(nt * tile - chunks) / double(nt * tile);
            // idle lanes cost issue slots, extra K tiles cost x reloads and
            // carries; among equal fits prefer more warps (latency hiding)
            const double cost = 2.0 * idle + 0.03 * double(nt - 1) +
                                0.002 * (kBulkMaxConsumerWarps - w) + 0.001 * cpl;
            if (cost < best_cost - 1e-12) {
                best_cost = cost;
                bw = w;
                bc = cpl;
            }
        }
    }
    if (bw == 0) return false;
    BulkPlan p;
    p.W = bw;
    p.cpl = bc;
    p.tile_chunks = 32 * bw * bc;
    p.ktiles = (chunks + p.tile_chunks - 1) / p.tile_chunks;
    // With one K tile a stage's rows are copied as one contiguous range, so
    // the shared row stride must be exactly the packed row.
    const int seg_chunks = p.ktiles == 1 ? chunks : p.tile_chunks;
    p.seg_v = seg_chunks * 16;
    p.seg_m = round_up(seg_chunks * MB, 16);
    const int seg = p.seg_v + p.seg_m;

    // 2. Rows per stage and ring depth.
    const int rmax = bulk_rmax(B);
    p.R = t.R ? std::min(t.R, rmax) : std::max(1, std::min(rmax, t.stage_bytes / seg));
    p.stage_bytes = p.R * seg;

    // 3. Grid: one wave of CTAs; more CTAs only if the carried partial sums
    //    of a CTA's rows would not fit in 64 KB.
    const int64_t want = static_cast<int64_t>(nsm) * t.ctas_per_sm;
    int64_t grid = std::min<int64_t>(rows, want);
    if (p.ktiles > 1) {
        const int64_t max_rows = (64 * 1024) / (4 * B);
        grid = std::max<int64_t>(grid, (rows + max_rows - 1) / max_rows);
    }
    if (grid > 0x7fffffff) return false;
    p.grid = static_cast<int>(grid);
    const int64_t rows_per_cta = (rows + grid - 1) / grid;
    const int carry = p.ktiles > 1 ? static_cast<int>(rows_per_cta * B * 4) : 0;

    const int part = 2 * p.W * 8 * 4;
    int S = std::max(2, std::min(16, t.ring_bytes / p.stage_bytes));
    auto total = [&](int s) {
        return static_cast<size_t>(s) * p.stage_bytes + 16 * s + part + carry;
    };
    while (S > 2 && total(S) > static_cast<size_t>(max_smem)) --S;
    if (total(S) > static_cast<size_t>(max_smem)) return false;
    p.S = S;
    p.off_bar = S * p.stage_bytes;
    p.off_part = p.off_bar + 16 * S;
    p.off_carry = p.off_part + part;
    p.smem = total(S);
    *out = p;
    return true;
}

namespace {

// The row kernel's plan for a K (in chunks), batch, warp count and a grid
// whose busiest CTA has rows_per_cta rows.
bool rows_plan_w(int64_t rows_per_cta, int grid, int chunks, int CK, int B, int max_smem, int W,
                 RowsPlan *out, bool pair, int tab_bytes)
{
    const BulkTuning &t = bulk_tuning();
    const int MB = CK / 8;  // mask bytes per chunk
    if (W < 1) return false;

    // 1. K tile: the x all warps share, B * tile * CK * 2 bytes; all of K
    //    unless that exceeds rows_xtile bytes, else even tiles of a multiple
    //    of 32 chunks (two buffers, and the rows' partial sums carried).
    RowsPlan p;
    p.W = W;
    p.grid = grid;
    const int64_t x_bytes = static_cast<int64_t>(rows_x_tile_bytes(B, CK, 1)) * chunks;
    int64_t kt = std::max<int64_t>(1, (x_bytes + t.rows_xtile_bytes - 1) / t.rows_xtile_bytes);
    int64_t tile = (chunks + kt - 1) / kt;
    if (kt > 1) tile = (tile + 31) / 32 * 32;
    if (tile >= chunks) tile = chunks;
    p.tile_chunks = static_cast<int>(tile);
    p.ktiles = static_cast<int>((chunks + tile - 1) / tile);
    const int last_chunks = chunks - (p.ktiles - 1) * p.tile_chunks;
    p.xbuf_bytes = rows_x_tile_bytes(B, CK, p.tile_chunks);
    const int nxb = p.ktiles > 1 ? 2 : 1;
    const int64_t carry64 = p.ktiles > 1 ? rows_per_cta * B * 4 * (pair ? 2 : 1) : 0;
    if (carry64 > 64 * 1024) return false;
    const int carry = static_cast<int>(carry64);

    // 2. Tasks: R rows x one segment of a K tile, at most `target` bytes; a
    //    tile row longer than that is cut into even segments of a multiple
    //    of 32 chunks.  Smaller tasks are tried until everything fits with
    //    at least two slots per warp.
    // Three or more vectors: two rows per task (R * B partial sums per lane
    // stay <= 16), so each x unit read from shared memory serves two rows;
    // the task size then bounds the two rows' segments together.  Patterns
    // whose chunk spans 32 or more positions (x read per chunk is then at
    // least four times the value bytes) also take two rows a task when a
    // whole row fits the task size (measured: two-row tasks of short
    // segments lose more to copy count than they save on x reads).
    // (A gate/up pair always takes two rows a task: one of each matrix.)
    const bool two_rows = B >= 3 || pair;
    const int R_many = t.rows_R ? std::min(t.rows_R, rows_rmax(B)) : 2;
    for (int target = t.rows_task_bytes; target >= 512; target /= 2) {
        const int per_row = two_rows ? std::max(512, target / R_many) : target;
        const int64_t tile_bytes = static_cast<int64_t>(p.tile_chunks) * (16 + MB);
        int64_t nseg = std::max<int64_t>(1, (tile_bytes + per_row - 1) / per_row);
        int64_t seg = (p.tile_chunks + nseg - 1) / nseg;
        if (nseg > 1) seg = (seg + 31) / 32 * 32;
        if (seg >= p.tile_chunks) seg = p.tile_chunks;
        p.seg_chunks = static_cast<int>(seg);
        p.nseg = static_cast<int>((p.tile_chunks + seg - 1) / seg);
        p.nseg_last = static_cast<int>((last_chunks + seg - 1) / seg);
        p.seg_v = p.seg_chunks * 16;
        p.seg_m = round_up(p.seg_chunks * MB, 16);
        const int segb = p.seg_v + p.seg_m;

        // One or two vectors: the largest of 1, 2, 4 rows with R * segb <=
        // target (R * B partial sums per lane stay <= 8), whole tile rows
        // only.
        int R = 1;
        if (pair) R = 2;
        else if (two_rows) R = R_many;
        else if (t.rows_R) R = p.nseg == 1 ? t.rows_R : 1;
        else if (CK >= 32 && p.nseg == 1) R = 2;  // whole rows: two copies a task
        else if (CK >= 32 && t.rows_two == 1) R = 2;  // two rows' segments: four copies
        else
            while (p.nseg == 1 && R < 4 && 2 * R * segb <= target && 2 * R * B <= 8) R *= 2;
        if (R > rows_rmax(B)) return false;
        p.R = R;
        p.stage_bytes = R * segb;

        // 3. Shared memory: slots [W][SW] | x buffers | barriers | decode
        //    table | carry; SW from 2 to 4, as many as the ring budget and
        //    max_smem allow.
        const int tab = round_up(tab_bytes, 16);
        auto total = [&](int sw) {
            const size_t S = static_cast<size_t>(sw) * W;
            return S * p.stage_bytes + static_cast<size_t>(nxb) * p.xbuf_bytes +
                   round_up(static_cast<int>(8 * S), 16) + tab + carry;
        };
        int SW = std::max(2, std::min(4, t.rows_ring_bytes / (W * p.stage_bytes)));
        // no more slots than a warp has tasks (a small layer's CTA then
        // leaves room on its SM for the next call's CTA to start beside it)
        {
            const int64_t tiles = pair ? rows_per_cta : (rows_per_cta + R - 1) / R;
            const int64_t tasks = (tiles + W - 1) / W *
                                  (static_cast<int64_t>(p.ktiles - 1) * p.nseg + p.nseg_last);
            SW = static_cast<int>(std::max<int64_t>(2, std::min<int64_t>(SW, tasks)));
        }
        while (SW > 2 && total(SW) > static_cast<size_t>(max_smem)) --SW;
        if (total(SW) > static_cast<size_t>(max_smem)) continue;
        const int S = SW * W;
        p.SW = SW;
        p.off_x = S * p.stage_bytes;
        p.off_bar = p.off_x + nxb * p.xbuf_bytes;
        p.off_tab = p.off_bar + round_up(8 * S, 16);
        p.off_carry = p.off_tab + tab;
        p.smem = total(SW);
        *out = p;
        return true;
    }
    return false;
}

// Row tiles are dealt to the warps round robin, so the busiest warp has
// ceil(tiles / W) of them; the share of warp-time doing work is
// tiles / (W * ceil(tiles / W)).
double warp_balance(int64_t rows_per_cta, const RowsPlan &p, bool pair)
{
    const int64_t tiles = (rows_per_cta + (pair ? 1 : p.R) - 1) / (pair ? 1 : p.R);
    if (tiles <= p.W) return 1.0;  // one round: every tile runs at once
    const int64_t per = (tiles + p.W - 1) / p.W;
    return static_cast<double>(tiles) / static_cast<double>(per * p.W);
}

// The plan with the most warps up to max_warps, unless 12 to 15 warps
// share the CTA's row tiles much more evenly (the CTA ends with its busiest
// warp): e.g. 35 rows take 3 tiles on each of 12 warps instead of 3 on
// three of 16 and 2 on the rest.  Fewer warps also keep fewer bytes in
// flight, so the switch needs a large gain: measured, 35 rows (balance 0.73
// -> 0.97) gained, 56 and 97 rows (0.88 -> 1.0, 0.87 -> 0.99) lost.  The
// tuning key rows_warps fixes W.
bool rows_plan_impl(int64_t rows_per_cta, int grid, int chunks, int CK, int B, int max_smem,
                    int max_warps, RowsPlan *out, bool pair, int tab_bytes)
{
    const BulkTuning &t = bulk_tuning();
    const int wmax = std::min(t.rows_warps ? t.rows_warps : kRowsMaxWarps, max_warps);
    RowsPlan best;
    if (!rows_plan_w(rows_per_cta, grid, chunks, CK, B, max_smem, wmax, &best, pair, tab_bytes))
        return false;
    double best_bal = warp_balance(rows_per_cta, best, pair);
    // fewer row tiles than warps, one or two vectors: one warp a tile (the
    // rest would idle and only hold shared memory, which the next call's
    // CTA can then use beside this one: 1024 x 1024 2.00 -> 1.71 us), but
    // enough warps to stage the x tile in one round of loads (each thread
    // four 16-byte loads: 2 KB a warp; with 4 of 16 warps the 32 KB tile of
    // 1024 x 8192 at batch 4 took 8.0 -> 11.2 us).  From three vectors the
    // fewer warps measured ~4 % slower.
    if (!t.rows_warps && B <= 2) {
        const int64_t tiles = pair ? rows_per_cta : (rows_per_cta + best.R - 1) / best.R;
        const int64_t wcap = std::max<int64_t>(tiles, (best.xbuf_bytes + 2047) / 2048);
        if (wcap < best.W) {
            RowsPlan p;
            if (rows_plan_w(rows_per_cta, grid, chunks, CK, B, max_smem,
                            static_cast<int>(std::max<int64_t>(1, wcap)), &p, pair, tab_bytes) &&
                p.R == best.R) {
                *out = p;
                return true;
            }
        }
    }
    if (!t.rows_warps)
        for (int w = wmax - 1; w >= 12; --w) {
            RowsPlan p;
            if (!rows_plan_w(rows_per_cta, grid, chunks, CK, B, max_smem, w, &p, pair, tab_bytes))
                continue;
            const double bal = warp_balance(rows_per_cta, p, pair);
            if (bal > best_bal + 0.2) {
                best = p;
                best_bal = bal;
            }
        }
    *out = best;
    return true;
}

}  // namespace

bool rows_plan(int64_t rows, int chunks, int CK, int B, int nsm, int max_smem, int max_warps,
               RowsPlan *out, bool pair, int tab_bytes)
{
    if (rows <= 0 || chunks <= 0 || B < 1 || B > NM_MAX_BATCH) return false;
    const BulkTuning &t = bulk_tuning();
    if (!t.rows_kernel) return false;
    // One wave of CTAs; more only if the carried partial sums of a CTA's rows
    // would not fit (they are bounded by 32 KB here).
    int64_t grid = std::min<int64_t>(rows, static_cast<int64_t>(nsm) * t.ctas_per_sm);
    const int64_t max_rows = (32 * 1024) / (4 * B);
    grid = std::max<int64_t>(grid, (rows + max_rows - 1) / max_rows);
    if (grid > 0x7fffffff) return false;
    return rows_plan_impl((rows + grid - 1) / grid, static_cast<int>(grid), chunks, CK, B,
                          max_smem, max_warps, out, pair, tab_bytes);
}

bool rows_plan_group(const int64_t *rows, int count, int chunks, int CK, int B, int nsm,
                     int max_smem, int max_warps, RowsPlan *out, int *cta_begin, int tab_bytes)
{
    if (count < 1 || count > kRowsMaxGroup || chunks <= 0 || B < 1 || B > NM_MAX_BATCH)
        return false;
    const BulkTuning &t = bulk_tuning();
    if (!t.rows_kernel) return false;
    int64_t total = 0;
    for (int i = 0; i < count; ++i) {
        if (rows[i] <= 0) return false;
        total += rows[i];
    }
    const int G = static_cast<int>(std::min<int64_t>(total, static_cast<int64_t>(nsm) * t.ctas_per_sm));
    if (G < count) return false;
    // CTAs in proportion to rows (largest remainder), at least one and at
    // most rows[i] each.
    int g[kRowsMaxGroup];
    double frac[kRowsMaxGroup];
    int used = 0;
    for (int i = 0; i < count; ++i) {
        const double share = static_cast<double>(G) * rows[i] / total;
        g[i] = static_cast<int>(std::min<int64_t>(rows[i], std::max<int64_t>(1, static_cast<int64_t>(share))));
        frac[i] = share - g[i];
        used += g[i];
    }
    while (used < G) {  // hand out the rest by largest remainder
        int best = -1;
        for (int i = 0; i < count; ++i)
            if (g[i] < rows[i] && (best < 0 || frac[i] > frac[best])) best = i;
        if (best < 0) break;
        ++g[best];
        frac[best] -= 1.0;
        ++used;
    }
    while (used > G) {  // the at-least-one rule overshot: take from the largest
        int best = 0;
        for (int i = 1; i < count; ++i)
            if (g[i] > g[best]) best = i;
        if (g[best] <= 1) return false;
        --g[best];
        --used;
    }
    int64_t rpc = 0;
    cta_begin[0] = 0;
    for (int i = 0; i < count; ++i) {
        rpc = std::max<int64_t>(rpc, (rows[i] + g[i] - 1) / g[i]);
        cta_begin[i + 1] = cta_begin[i] + g[i];
    }
    return rows_plan_impl(rpc, used, chunks, CK, B, max_smem, max_warps, out, false, tab_bytes);
}

// The sparse-operand tensor-core product's plan, for one matrix or a group
// launched together.  Without the split the rows are spread over min(rows,
// nsm) CTAs (a group's CTAs split over its matrices in proportion to their
// rows); with it, units of one or two 128-row tiles are each shared by a
// cluster of k = 2, 4 or 8 CTAs (rank 0 receives
// the other ranks' sums, 8, 16 or 32 floats a row by the batch, in at most
// 64 KB of shared memory).
// Measured on B300: a CTA's 128-position slab costs ~0.43 us with one tile
// and ~0.61 us with two whatever rows they hold (below the HBM rate for
// small tiles), a CTA streams at most ~55 GB/s and all of them ~6.2 TB/s;
// the estimate of a plan is the largest of those bounds (weights at 1.125
// bytes each), and the least estimate is taken, the smaller cluster within
// 3 %.  Clusters of 3, 5, 6 or 7 are not used: the GPU held only ~40
// clusters of 3 at once where the occupancy query promised 48, so part of
// the grid ran in a second wave; a plan never has more units than clusters
// of its size are resident.  Tuning keys: sp_split=0 (never split), sp_k
// (only that cluster size, taken wherever it fits), sp_units (at least that
// many units).
SpGroupPlan sp_group_plan(const int64_t *rows, int count, int64_t K, int batch, int nsm,
                          const int *resident)
{
    constexpr int kTile = 128;  // rows of an MMA tile
    constexpr int kSlab = 128;  // K positions of a slab
    const int64_t nslab = K / kSlab;
    int64_t total_rows = 0;
    for (int i = 0; i < count; ++i) total_rows += rows[i];
    const double bytes = static_cast<double>(total_rows) * static_cast<double>(K) * 1.125;
    auto finish = [&](SpGroupPlan &g) {
        g.total_units = 0;
        g.max_box_rows = 0;
        for (int i = 0; i < g.count; ++i) {
            g.box_rows[i] = static_cast<int>((rows[i] + g.units[i] - 1) / g.units[i]);
            g.total_units += g.units[i];
            g.max_box_rows = std::max(g.max_box_rows, g.box_rows[i]);
        }
    };
    auto estimate = [&](const SpGroupPlan &g) {
        const int nt = (g.max_box_rows + kTile - 1) / kTile;
        const double t_slab = static_cast<double>((nslab + g.k - 1) / g.k) * (nt == 1 ? 0.43 : 0.61);
        const double ctas = static_cast<double>(g.total_units * g.k);
        const double t_bw = std::max(bytes / 6.2e6, bytes / (ctas * 55e3));
        return std::max(t_slab, t_bw);
    };
    // no split: min(total rows, nsm) CTAs, each matrix at least one and a
    // share in proportion to its rows (never more CTAs than rows)
    SpGroupPlan best = {};
    best.k = 1;
    best.count = count;
    const int64_t ctas = std::max<int64_t>(count, std::min<int64_t>(total_rows, nsm));
    int64_t used = 0;
    for (int i = 0; i < count; ++i) {
        const int64_t share = total_rows > 0 ? ctas * rows[i] / total_rows : 1;
        best.units[i] = std::max<int64_t>(1, std::min<int64_t>(rows[i], share));
        used += best.units[i];
    }
    while (used < ctas) {  // the rest to the matrices with the most rows a CTA
        int at = -1;
        for (int i = 0; i < count; ++i)
            if (best.units[i] < rows[i] &&
                (at < 0 || rows[i] * best.units[at] > rows[at] * best.units[i]))
                at = i;
        if (at < 0) break;
        ++best.units[at];
        ++used;
    }
    finish(best);
    double t_best = estimate(best);
    const BulkTuning &tu = bulk_tuning();
    if (!tu.sp_split || batch > 32 || total_rows < 1) return best;
    const int row_bytes = batch <= 8 ? 32 : batch <= 16 ? 64 : 128;  // a rank's sums of a row
    for (int k = 2; k <= 8; k *= 2) {
        if (tu.sp_k > 0 && k != tu.sp_k) continue;
        if (k > nslab) break;
        for (int nt = 1; nt <= 2; ++nt) {
            SpGroupPlan g = {};
            g.k = k;
            g.count = count;
            for (int i = 0; i < count; ++i) {
                g.units[i] = (rows[i] + kTile * nt - 1) / (kTile * nt);
                if (tu.sp_units > 0 && count == 1)
                    g.units[i] = std::max<int64_t>(g.units[i], std::min<int64_t>(tu.sp_units, rows[i]));
            }
            finish(g);
            if (g.total_units * k > nsm || g.total_units > resident[k]) continue;
            if (g.max_box_rows > kTile * nt) continue;
            // rank 0's region for the other ranks' sums stays within 64 KB
            if ((k - 1) * kTile * nt * row_bytes > 65536) continue;
            const double t = estimate(g);
            if (t < 0.97 * t_best || (tu.sp_k > 0 && best.k == 1)) {
                best = g;
                t_best = t;
            }
        }
    }
    return best;
}

SpSplit sp_split_plan(int64_t rows, int64_t K, int batch, int nsm, const int *resident)
{
    const SpGroupPlan g = sp_group_plan(&rows, 1, K, batch, nsm, resident);
    SpSplit p;
    p.k = g.k;
    p.units = g.units[0];
    p.box_rows = g.box_rows[0];
    return p;
}

}  // namespace nm

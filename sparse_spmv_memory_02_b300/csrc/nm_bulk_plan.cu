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
        else if (!std::strcmp(tok, "rows_task") && v >= 1024) t.rows_task_bytes = v;
        else if (!std::strcmp(tok, "rows_ring") && v >= 4096) t.rows_ring_bytes = v;
        else if (!std::strcmp(tok, "rows_seg") && v >= 1024) t.rows_max_seg = v;
        else if (!std::strcmp(tok, "rows") && (v == 0 || v == 1)) t.rows_kernel = v;
        else if (!std::strcmp(tok, "l2pf") && v >= 0) t.l2_prefetch_bytes = v / 16 * 16;
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

// The row kernel's plan for a K (in chunks), batch and a grid whose busiest
// CTA has rows_per_cta rows.
bool rows_plan_impl(int64_t rows_per_cta, int grid, int chunks, int CK, int B, int max_smem,
                    RowsPlan *out)
{
    const BulkTuning &t = bulk_tuning();
    const int MB = CK / 8;  // mask bytes per chunk
    const int W = t.rows_warps ? t.rows_warps : 16;
    const int64_t row_bytes = static_cast<int64_t>(chunks) * (16 + MB);
    const int64_t x_bytes = static_cast<int64_t>(B) * chunks * CK * 2;

    // Every warp owns SW >= 2 slots of one task each; a task is R rows x one
    // K tile of at most `target` bytes, rows longer than that are split into
    // K tiles.  Smaller tasks are tried until everything fits.
    for (int target = t.rows_task_bytes; target >= 1024; target /= 2) {
        RowsPlan p;
        p.W = W;
        p.grid = grid;
        // 1. K tile: whole rows if a row fits the task and the x tile 48 KB;
        //    tiles are multiples of 32 chunks and split the row evenly.
        const int64_t seg_cap = std::min<int64_t>(target, t.rows_max_seg);
        int64_t kt = std::max<int64_t>((row_bytes + seg_cap - 1) / seg_cap,
                                       (x_bytes + 48 * 1024 - 1) / (48 * 1024));
        kt = std::max<int64_t>(1, kt);
        int64_t tile = (chunks + kt - 1) / kt;
        tile = (tile + 31) / 32 * 32;
        if (tile > chunks) tile = chunks;  // one tile: exactly the row
        p.tile_chunks = static_cast<int>(tile);
        p.ktiles = static_cast<int>((chunks + tile - 1) / tile);
        p.seg_v = p.tile_chunks * 16;
        p.seg_m = round_up(p.tile_chunks * MB, 16);
        const int seg = p.seg_v + p.seg_m;

        // 2. Rows per task: the largest of 1, 2, 4 with R * seg <= target
        //    (R * B partial sums per lane stay <= 8).
        int R = 1;
        if (t.rows_R) R = t.rows_R;
        else
            while (R < 4 && 2 * R * seg <= target && 2 * R * B <= 8) R *= 2;
        if (R * B > 8) return false;
        p.R = R;
        p.stage_bytes = R * seg;

        // 3. Shared memory: slots [W][SW] | x buffers | barriers | carry.
        const int64_t carry64 = p.ktiles > 1 ? rows_per_cta * B * 4 : 0;
        if (carry64 > 64 * 1024) return false;
        const int carry = static_cast<int>(carry64);
        p.xbuf_bytes = B * (CK / 8) * p.tile_chunks * 16;
        const int nxb = p.ktiles > 1 ? 2 : 1;
        int SW = std::max(2, std::min(4, t.rows_ring_bytes / (W * p.stage_bytes)));
        auto total = [&](int sw) {
            const size_t S = static_cast<size_t>(sw) * W;
            return S * p.stage_bytes + static_cast<size_t>(nxb) * p.xbuf_bytes +
                   round_up(static_cast<int>(8 * S), 16) + carry;
        };
        while (SW > 2 && total(SW) > static_cast<size_t>(max_smem)) --SW;
        if (total(SW) > static_cast<size_t>(max_smem)) continue;
        const int S = SW * W;
        p.SW = SW;
        p.off_x = S * p.stage_bytes;
        p.off_bar = p.off_x + nxb * p.xbuf_bytes;
        p.off_carry = p.off_bar + round_up(8 * S, 16);
        p.smem = total(SW);
        *out = p;
        return true;
    }
    return false;
}

}  // namespace

bool rows_plan(int64_t rows, int chunks, int CK, int B, int nsm, int max_smem, RowsPlan *out)
{
    if (rows <= 0 || chunks <= 0 || B < 1 || B > 2) return false;
    const BulkTuning &t = bulk_tuning();
    if (!t.rows_kernel) return false;
    // One wave of CTAs; more only if the carried partial sums of a CTA's rows
    // would not fit (they are bounded by 32 KB here).
    int64_t grid = std::min<int64_t>(rows, static_cast<int64_t>(nsm) * t.ctas_per_sm);
    const int64_t max_rows = (32 * 1024) / (4 * B);
    grid = std::max<int64_t>(grid, (rows + max_rows - 1) / max_rows);
    if (grid > 0x7fffffff) return false;
    return rows_plan_impl((rows + grid - 1) / grid, static_cast<int>(grid), chunks, CK, B,
                          max_smem, out);
}

bool rows_plan_group(const int64_t *rows, int count, int chunks, int CK, int B, int nsm,
                     int max_smem, RowsPlan *out, int *cta_begin)
{
    if (count < 1 || count > kRowsMaxGroup || chunks <= 0 || B < 1 || B > 2) return false;
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
    return rows_plan_impl(rpc, used, chunks, CK, B, max_smem, out);
}

}  // namespace nm

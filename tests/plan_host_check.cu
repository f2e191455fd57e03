// Host-side check of the streaming kernels' launch planning (rows_plan,
// rows_plan_group and bulk_plan from csrc/nm_bulk_plan.cu, compiled for and
// run on the CPU).  Built and run by tests/test_plan_host.py; no GPU is used.
//
// Over the decode-layer shapes of the workloads, ragged shapes, every vector
// count 1-8 and every chunk span (CK = 8, 16, 32, 64), each plan must:
//   * fit the shared-memory limit, with every region 16-byte aligned;
//   * cover K exactly: K tiles and their segments tile the row's chunks with
//     no gap and no chunk twice (tiles and segments of a multiple of 32
//     chunks when cut);
//   * cover the rows: grid CTAs of ceil(rows / grid) rows, at most one CTA
//     per row; a group's CTAs split in order, at least one per matrix and
//     at most one per row;
//   * keep the per-lane partial sums (R rows x B vectors) within the
//     kernel's register budget, and the carried partial sums within 64 KB.
// The tensor-core product's K-split plans (sp_split_plan) are checked for
// their limits too, and for the plans measured best on B300.
#include <cstdint>
#include <cstdio>
#include <vector>

#include "nm_bulk.cuh"
#include "nm_rows.cuh"

namespace {

constexpr int kNsm = 148;
constexpr int kMaxSmem = 232448;  // opt-in shared memory per CTA on sm_103a
long g_fail = 0, g_plans = 0, g_none = 0;

#define EXPECT(cond, ...)                                                   \
    do {                                                                    \
        if (!(cond)) {                                                      \
            if (g_fail < 20) {                                              \
                std::printf("FAIL %s: ", #cond);                            \
                std::printf(__VA_ARGS__);                                   \
                std::printf("\n");                                          \
            }                                                               \
            ++g_fail;                                                       \
        }                                                                   \
    } while (0)

void check_rows_plan(const nm::RowsPlan &p, int64_t rows_per_cta, int chunks, int CK, int B,
                     const char *what, int tab_bytes)
{
    const int MB = CK / 8;
    EXPECT(p.smem <= static_cast<size_t>(kMaxSmem), "%s smem %zu", what, p.smem);
    EXPECT(p.W >= 1 && p.W <= nm::kRowsMaxWarps, "%s W %d", what, p.W);
    EXPECT(p.SW >= 2 && p.SW <= 4, "%s SW %d", what, p.SW);
    // K tiles
    EXPECT(p.ktiles >= 1 && static_cast<int64_t>(p.ktiles) * p.tile_chunks >= chunks &&
               static_cast<int64_t>(p.ktiles - 1) * p.tile_chunks < chunks,
           "%s ktiles %d tile %d chunks %d", what, p.ktiles, p.tile_chunks, chunks);
    EXPECT(p.ktiles == 1 || p.tile_chunks % 32 == 0, "%s tile %d", what, p.tile_chunks);
    const int last = chunks - (p.ktiles - 1) * p.tile_chunks;
    // segments of a tile and of the last tile
    EXPECT(p.nseg >= 1 && static_cast<int64_t>(p.nseg) * p.seg_chunks >= p.tile_chunks &&
               static_cast<int64_t>(p.nseg - 1) * p.seg_chunks < p.tile_chunks,
           "%s nseg %d seg %d tile %d", what, p.nseg, p.seg_chunks, p.tile_chunks);
    EXPECT(p.nseg_last >= 1 && static_cast<int64_t>(p.nseg_last) * p.seg_chunks >= last &&
               static_cast<int64_t>(p.nseg_last - 1) * p.seg_chunks < last,
           "%s nseg_last %d seg %d last %d", what, p.nseg_last, p.seg_chunks, last);
    EXPECT(p.nseg == 1 || p.seg_chunks % 32 == 0, "%s seg %d", what, p.seg_chunks);
    // slot layout: one row's segment of values and of mask bytes
    EXPECT(p.seg_v == p.seg_chunks * 16, "%s seg_v", what);
    EXPECT(p.seg_m >= p.seg_chunks * MB && p.seg_m % 16 == 0 && p.seg_m < p.seg_chunks * MB + 16,
           "%s seg_m %d", what, p.seg_m);
    EXPECT(p.stage_bytes == p.R * (p.seg_v + p.seg_m), "%s stage", what);
    EXPECT(p.R >= 1 && p.R <= nm::rows_rmax(B) && p.R * B <= 16, "%s R %d B %d", what, p.R, B);
    // x buffer: B vectors of the tile's positions, fp16; from three vectors
    // each column's units padded to an odd count
    const int col_units = B <= 2 ? 0 : B * (CK / 8) + ((B * (CK / 8)) % 2 == 0 ? 1 : 0);
    EXPECT(p.xbuf_bytes == (B <= 2 ? B * p.tile_chunks * CK * 2 : col_units * p.tile_chunks * 16),
           "%s xbuf", what);
    EXPECT(col_units == nm::rows_x_col_units(B, CK) && (B <= 2 || col_units % 2 == 1),
           "%s column units", what);
    // regions in order, 16-byte aligned, inside smem
    const int S = p.SW * p.W;
    EXPECT(p.off_x == S * p.stage_bytes, "%s off_x", what);
    EXPECT(p.off_bar == p.off_x + (p.ktiles > 1 ? 2 : 1) * p.xbuf_bytes, "%s off_bar", what);
    EXPECT(p.off_tab >= p.off_bar + 8 * S, "%s off_tab", what);
    EXPECT(p.off_carry >= p.off_tab + tab_bytes, "%s off_carry", what);
    EXPECT(p.off_x % 16 == 0 && p.off_bar % 16 == 0 && p.off_tab % 16 == 0 &&
               p.off_carry % 16 == 0 &&
               p.stage_bytes % 16 == 0 && p.xbuf_bytes % 16 == 0,
           "%s alignment", what);
    const int64_t carry = p.ktiles > 1 ? rows_per_cta * B * 4 : 0;
    EXPECT(carry <= 64 * 1024, "%s carry %lld", what, static_cast<long long>(carry));
    EXPECT(static_cast<int64_t>(p.off_carry) + carry <= static_cast<int64_t>(p.smem),
           "%s carry region", what);
}

void one(int64_t rows, int64_t K, int N, int M, int B)
{
    const int CK = 8 * M / N;
    if (K % CK != 0) return;
    const int chunks = static_cast<int>(K / CK);
    char what[128];
    std::snprintf(what, sizeof(what), "rows %lld K %lld %d:%d B %d", static_cast<long long>(rows),
                  static_cast<long long>(K), N, M, B);
    // the 8-wide patterns with two or four kept carry a 1 KB decode table
    const int tab = (M == 8 && (N == 2 || N == 4)) ? 1024 : 0;
    nm::RowsPlan p;
    if (nm::rows_plan(rows, chunks, CK, B, kNsm, kMaxSmem, nm::kRowsMaxWarps, &p, false, tab)) {
        ++g_plans;
        EXPECT(p.grid >= 1 && p.grid <= rows, "%s grid %d", what, p.grid);
        const int64_t rpc = (rows + p.grid - 1) / p.grid;
        EXPECT(rpc * p.grid >= rows && (rpc - 1) * p.grid < rows, "%s rpc", what);
        check_rows_plan(p, rpc, chunks, CK, B, what, tab);
    } else {
        ++g_none;
        // the chunk-column kernel must then take it
        nm::BulkPlan b;
        const bool ok = nm::bulk_plan(rows, chunks, CK, B, kNsm, kMaxSmem, &b);
        EXPECT(ok, "%s: no plan at all", what);
        if (ok) EXPECT(b.smem <= static_cast<size_t>(kMaxSmem), "%s bulk smem", what);
    }
}

void group(const std::vector<int64_t> &rows, int64_t K, int N, int M, int B)
{
    const int CK = 8 * M / N;
    const int chunks = static_cast<int>(K / CK);
    char what[128];
    std::snprintf(what, sizeof(what), "group of %zu, K %lld %d:%d B %d", rows.size(),
                  static_cast<long long>(K), N, M, B);
    const int tab = (M == 8 && (N == 2 || N == 4)) ? 1024 : 0;
    nm::RowsPlan p;
    int cta_begin[nm::kRowsMaxGroup + 1];
    if (!nm::rows_plan_group(rows.data(), static_cast<int>(rows.size()), chunks, CK, B, kNsm,
                             kMaxSmem, nm::kRowsMaxWarps, &p, cta_begin, tab)) {
        ++g_none;
        return;
    }
    ++g_plans;
    int64_t total = 0;
    for (int64_t r : rows) total += r;
    EXPECT(cta_begin[0] == 0 && cta_begin[rows.size()] == p.grid, "%s grid %d", what, p.grid);
    const int64_t ctas = static_cast<int64_t>(kNsm) * nm::bulk_tuning().ctas_per_sm;
    EXPECT(p.grid == static_cast<int>(std::min<int64_t>(total, ctas)), "%s grid %d", what, p.grid);
    int64_t rpc = 0;
    for (size_t i = 0; i < rows.size(); ++i) {
        const int g = cta_begin[i + 1] - cta_begin[i];
        EXPECT(g >= 1 && g <= rows[i], "%s matrix %zu gets %d CTAs", what, i, g);
        if (g >= 1) rpc = std::max<int64_t>(rpc, (rows[i] + g - 1) / g);
    }
    check_rows_plan(p, rpc, chunks, CK, B, what, tab);
}

}  // namespace

// The tensor-core product's K-split plan for one shape: at most one CTA an
// SM and one row a unit, no more units than clusters of that size are
// resident, units of at most two 128-row tiles (one or two for a split),
// every rank at least one 128-position slab, clusters of 2, 4 or 8, at most
// 32 vectors and rank 0's region for the other ranks' sums within 64 KB.
void sp_one(int64_t rows, int64_t K, int B, const int *resident, const char *dev)
{
    const nm::SpSplit p = nm::sp_split_plan(rows, K, B, kNsm, resident);
    ++g_plans;
    EXPECT(p.k == 1 || p.k == 2 || p.k == 4 || p.k == 8, "%s %lldx%lld B%d k %d", dev,
           (long long)rows, (long long)K, B, p.k);
    EXPECT(p.units >= 1 && p.units <= rows && p.units * p.k <= kNsm,
           "%s %lldx%lld B%d units %lld k %d", dev, (long long)rows, (long long)K, B,
           (long long)p.units, p.k);
    EXPECT(p.box_rows == static_cast<int>((rows + p.units - 1) / p.units),
           "%s %lldx%lld box %d", dev, (long long)rows, (long long)K, p.box_rows);
    if (p.k > 1) {
        const int nt = (p.box_rows + 127) / 128;
        EXPECT(B <= 32 && p.units <= resident[p.k] && p.k <= K / 128 && p.box_rows <= 256 &&
                   (p.k - 1) * 128 * nt * (B <= 8 ? 32 : B <= 16 ? 64 : 128) <= 65536,
               "%s %lldx%lld B%d split k %d units %lld box %d", dev, (long long)rows,
               (long long)K, B, p.k, (long long)p.units, p.box_rows);
    }
}

// A group's plan: every matrix at least one unit and at most one a row, its
// rows spread over its units, at most one CTA an SM, the split's limits as
// for one matrix; a group of one has sp_split_plan's plan.
void sp_group_one(const std::vector<int64_t> &rows, int64_t K, int B, const int *resident,
                  const char *dev)
{
    const nm::SpGroupPlan g = nm::sp_group_plan(rows.data(), static_cast<int>(rows.size()), K, B,
                                                kNsm, resident);
    ++g_plans;
    int64_t total = 0, total_rows = 0;
    int maxb = 0;
    for (size_t i = 0; i < rows.size(); ++i) {
        EXPECT(g.units[i] >= 1 && g.units[i] <= std::max<int64_t>(1, rows[i]),
               "%s group %zu: units %lld rows %lld", dev, i, (long long)g.units[i],
               (long long)rows[i]);
        EXPECT(g.box_rows[i] == static_cast<int>((rows[i] + g.units[i] - 1) / g.units[i]),
               "%s group %zu: box %d", dev, i, g.box_rows[i]);
        total += g.units[i];
        total_rows += rows[i];
        maxb = std::max(maxb, g.box_rows[i]);
    }
    EXPECT(g.count == static_cast<int>(rows.size()) && g.total_units == total &&
               g.max_box_rows == maxb && total * g.k <= std::max<int64_t>(kNsm, total),
           "%s group totals: units %lld k %d", dev, (long long)total, g.k);
    if (g.k > 1) {
        const int nt = (maxb + 127) / 128;
        EXPECT(B <= 32 && total * g.k <= kNsm && total <= resident[g.k] && g.k <= K / 128 &&
                   maxb <= 256 && (g.k - 1) * 128 * nt * (B <= 8 ? 32 : B <= 16 ? 64 : 128) <= 65536,
               "%s group split k %d units %lld box %d", dev, g.k, (long long)total, maxb);
    }
    if (rows.size() == 1) {
        const nm::SpSplit p = nm::sp_split_plan(rows[0], K, B, kNsm, resident);
        EXPECT(p.k == g.k && p.units == g.units[0] && p.box_rows == g.box_rows[0],
               "%s group of one differs from the single plan", dev);
    }
}

// Plans the B300 measurements chose (resident clusters of 2, 4, 8: 74, 37,
// 18), at batch 8 with the default tuning.
void sp_expect(int64_t rows, int64_t K, int k, int64_t units)
{
    const int resident[9] = {0, 0, 74, 0, 37, 0, 0, 0, 18};
    const nm::SpSplit p = nm::sp_split_plan(rows, K, 8, kNsm, resident);
    EXPECT(p.k == k && p.units == units, "%lldx%lld: plan k %d units %lld, expected k %d units %lld",
           (long long)rows, (long long)K, p.k, (long long)p.units, k, (long long)units);
}

int main()
{
    const int pats[][2] = {{2, 4}, {4, 8}, {1, 4}, {2, 8}, {1, 8}, {4, 4}, {8, 8}};
    const int64_t rows_list[] = {1, 7, 77, 148, 149, 300, 1024, 4096, 5120, 8192, 14336,
                                 17408, 25600, 28672, 37000, 100000};
    const int64_t k_list[] = {128, 1024, 3072, 4096, 5120, 8192, 14336, 17408, 25600, 28672,
                              36864, 40960, 81920};
    for (auto &pm : pats)
        for (int64_t r : rows_list)
            for (int64_t K : k_list)
                for (int B = 1; B <= 8; ++B) one(r, K, pm[0], pm[1], B);
    const std::vector<std::vector<int64_t>> groups = {
        {4096, 1024, 1024}, {14336, 14336}, {28672, 28672}, {8192, 1024, 1024},
        {25600, 25600}, {333, 77, 250, 4, 5, 6, 7, 900}, {1, 1}, {100000, 1}, {700, 300, 1}};
    for (auto &g : groups)
        for (int64_t K : {1024L, 4096L, 5120L, 8192L})
            for (int B = 1; B <= 8; ++B) {
                group(g, K, 2, 4, B);
                group(g, K, 4, 8, B);
            }
    // the tensor-core product's split plans, with the resident cluster counts
    // measured on B300, fewer of them, and none (no split possible)
    const int res_b300[9] = {0, 0, 74, 0, 37, 0, 0, 0, 18};
    const int res_small[9] = {0, 0, 30, 0, 10, 0, 0, 0, 3};
    const int res_none[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};
    for (int64_t r : rows_list)
        for (int64_t K : {128L, 256L, 384L, 1024L, 4096L, 8192L, 25600L, 28672L})
            for (int B : {1, 2, 3, 5, 8, 9, 16, 32}) {
                sp_one(r, K, B, res_b300, "b300");
                sp_one(r, K, B, res_small, "small");
                sp_one(r, K, B, res_none, "none");
            }
    const std::vector<std::vector<int64_t>> sp_groups = {
        {8192, 1024, 1024}, {4096, 1024, 1024}, {28672, 28672}, {1}, {5, 7},
        {100000, 1}, {300, 77, 250, 4, 5, 6, 7, 900}, {8192}, {20000, 20000}};
    for (auto &g : sp_groups)
        for (int64_t K : {128L, 1024L, 8192L})
            for (int B : {3, 8, 16, 32}) {
                sp_group_one(g, K, B, res_b300, "b300");
                sp_group_one(g, K, B, res_small, "small");
                sp_group_one(g, K, B, res_none, "none");
            }
    if (nm::bulk_tuning().sp_split && nm::bulk_tuning().sp_k == 0 &&
        nm::bulk_tuning().sp_units == 0) {
        sp_expect(8192, 28672, 4, 32);   // 32 two-tile units, clusters of 4
        sp_expect(8192, 8192, 4, 32);
        sp_expect(5120, 25600, 4, 20);
        sp_expect(1024, 8192, 8, 8);     // 8 one-tile units, clusters of 8
        sp_expect(28672, 8192, 1, 148);  // 194 rows a CTA, no split
    }
    std::printf("%ld plans checked, %ld shapes without a row plan, %ld failures\n", g_plans,
                g_none, g_fail);
    std::printf(g_fail ? "FAIL\n" : "OK\n");
    return g_fail ? 1 : 0;
}

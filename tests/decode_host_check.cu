// Host-side check of the vectorised kernels' mask decode and lane gather
// (Pattern<N, M>::decode and ::dot from csrc/nm_fast.cuh, compiled for the
// CPU).  Built and run by tests/test_decode_host.py; no GPU is used.
//
// For every valid mask of one 16-byte value chunk (all of them for 2:4, 1:4,
// 2:8 and 4:8, a seeded sample for 1:8) and every value slot i of the chunk,
// dot() is called with a one-hot value vector (slot i = 1.0, the others 0)
// and x lane p = p + 1: the result must be 1 + the position of the chunk's
// i-th kept weight, the positions taken group by group in increasing k (the
// packed layout's fixed-step order).  The dense patterns (N = M) keep every
// position.  Every mask is decoded both from registers alone (decode) and
// through the shared-memory table of the 8-wide patterns (decode_tab).
//
// It also checks the tensor-core product's group expansion (expand_sel in
// csrc/nm_tc_expand.cuh, used as the two 16-bit selectors the kernel
// stores): for every 2:4 nibble, the group's value pair lands on its two
// kept positions, lower k first, and the other two positions are zero.
#include <cstdint>
#include <cstdio>
#include <vector>

#include "nm_fast.cuh"
#include "nm_tc_expand.cuh"

namespace {

uint16_t f16_of_int(int v)  // exact for 0 <= v <= 2048
{
    if (v == 0) return 0;
    int e = 0;
    while ((v >> e) > 1) ++e;
    const uint32_t frac = (static_cast<uint32_t>(v) << (10 - e)) & 0x3FFu;
    return static_cast<uint16_t>(((e + 15) << 10) | frac);
}

struct Result { long checks = 0, fails = 0; };

template <int N, int M>
void check_mask(uint64_t mask, Result &r)
{
    using P = nm::Pattern<N, M>;
    constexpr int CK = P::CK;
    // kept positions in order: groups in order, increasing k inside a group
    std::vector<int> kept;
    for (int p = 0; p < CK; ++p)
        if (N == M || ((mask >> p) & 1u)) kept.push_back(p);
    if (static_cast<int>(kept.size()) != 8) {
        std::printf("internal: %zu kept positions\n", kept.size());
        ++r.fails;
        return;
    }
    uint32_t x[CK / 2];
    for (int w = 0; w < CK / 2; ++w)
        x[w] = f16_of_int(2 * w + 1) | (static_cast<uint32_t>(f16_of_int(2 * w + 2)) << 16);
    // both decodes: from registers alone, and through the shared-memory
    // table the streaming kernel builds (word i = tab_entry(i))
    static uint32_t tab[256];
    static bool tab_ready = false;
    if (!tab_ready) {
        for (int i = 0; i < 256; ++i) tab[i] = P::tab_entry(static_cast<uint32_t>(i));
        tab_ready = true;
    }
    const auto sel = P::decode(static_cast<typename P::mask_t>(mask));
    const auto sel_tab = P::decode_tab(static_cast<typename P::mask_t>(mask), tab);
    for (int i = 0; i < 8; ++i) {
        uint32_t vw[4] = {0, 0, 0, 0};
        vw[i / 2] = static_cast<uint32_t>(0x3C00u) << (16 * (i % 2));
        const uint4 v = make_uint4(vw[0], vw[1], vw[2], vw[3]);
        for (int way = 0; way < 2; ++way) {
            const float got = P::dot(v, way ? sel_tab : sel, x, 0.0f);
            ++r.checks;
            if (got != static_cast<float>(kept[i] + 1)) {
                if (r.fails < 5)
                    std::printf("%d:%d mask %016llx slot %d (%s): got %g, want %d\n", N, M,
                                static_cast<unsigned long long>(mask), i,
                                way ? "table" : "registers", got, kept[i] + 1);
                ++r.fails;
            }
        }
    }
}

// Every group mask of width M with exactly N set bits.
std::vector<uint32_t> group_masks(int N, int M)
{
    std::vector<uint32_t> out;
    for (uint32_t g = 0; g < (1u << M); ++g)
        if (__builtin_popcount(g) == N) out.push_back(g);
    return out;
}

template <int N, int M>
Result check_all(long sample)
{
    Result r;
    constexpr int groups = nm::Pattern<N, M>::CK / M;
    const std::vector<uint32_t> gm = group_masks(N, M);
    long total = 1;
    for (int g = 0; g < groups; ++g) total *= static_cast<long>(gm.size());
    uint64_t state = 0x9E3779B97F4A7C15ull;
    const bool all = sample <= 0 || total <= sample;
    const long count = all ? total : sample;
    for (long t = 0; t < count; ++t) {
        long idx = t;
        if (!all) {  // xorshift64 sample of the combinations
            state ^= state << 13;
            state ^= state >> 7;
            state ^= state << 17;
            idx = static_cast<long>(state % static_cast<uint64_t>(total));
        }
        uint64_t mask = 0;
        for (int g = 0; g < groups; ++g) {
            mask |= static_cast<uint64_t>(gm[idx % gm.size()]) << (M * g);
            idx /= static_cast<long>(gm.size());
        }
        check_mask<N, M>(mask, r);
    }
    std::printf("%d:%d %ld masks%s, %ld checks, %ld failures\n", N, M, count,
                all ? " (all)" : " (sampled)", r.checks, r.fails);
    return r;
}

Result check_expand()
{
    Result r;
    const uint32_t lo = 0x1357u, hi = 0x2468u, v = lo | (hi << 16);
    for (uint32_t n : group_masks(2, 4)) {
        const uint32_t sel = nm::expand_sel(n);
        const uint32_t w[2] = {nm::prmt(v, 0u, sel & 0xFFFFu), nm::prmt(v, 0u, sel >> 16)};
        int j = 0;
        for (int p = 0; p < 4; ++p) {
            const uint32_t want = ((n >> p) & 1u) ? (j++ == 0 ? lo : hi) : 0u;
            const uint32_t got = (w[p / 2] >> (16 * (p % 2))) & 0xFFFFu;
            ++r.checks;
            if (got != want) {
                std::printf("expand nibble %x position %d: got %04x, want %04x\n", n, p, got, want);
                ++r.fails;
            }
        }
    }
    std::printf("2:4x expand %zu nibbles, %ld checks, %ld failures\n", group_masks(2, 4).size(),
                r.checks, r.fails);
    return r;
}

// The sparse tensor-core metadata: every combination of valid 2:4 groups in
// a mask word (sampled), each nibble's code = the positions of its two set
// bits, lower first (mode 0) or swapped (mode 1).
Result check_sp_meta()
{
    Result r;
    const std::vector<uint32_t> gm = group_masks(2, 4);
    uint64_t state = 0x2545F4914F6CDD1Dull;
    for (int t = 0; t < 200000; ++t) {
        state ^= state << 13;
        state ^= state >> 7;
        state ^= state << 17;
        uint32_t m = 0, want0 = 0, want1 = 0;
        uint64_t s = state;
        for (int g = 0; g < 8; ++g) {
            const uint32_t n = gm[s % gm.size()];
            s /= gm.size();
            m |= n << (4 * g);
            int i0 = -1, i1 = -1;
            for (int p = 0; p < 4; ++p)
                if ((n >> p) & 1u) (i0 < 0 ? i0 : i1) = p;
            want0 |= static_cast<uint32_t>(i0 | (i1 << 2)) << (4 * g);
            want1 |= static_cast<uint32_t>(i1 | (i0 << 2)) << (4 * g);
        }
        for (int mode = 0; mode < 2; ++mode) {
            ++r.checks;
            const uint32_t got = nm::sp_meta_word(m, mode), want = mode ? want1 : want0;
            if (got != want) {
                if (r.fails < 5)
                    std::printf("sp meta mode %d mask %08x: got %08x, want %08x\n", mode, m, got,
                                want);
                ++r.fails;
            }
        }
    }
    // lane interleave of rows r, r + 8: the word a lane stores gives, read
    // back as the tensor cores read it (low lane: own low half = row r groups
    // 0-3, partner's low half = row r groups 4-7; high lane: partner's high
    // half = row r+8 groups 0-3, own high half = groups 4-7), each row's own
    // metadata word
    for (int t = 0; t < 100000; ++t) {
        state ^= state << 13;
        state ^= state >> 7;
        state ^= state << 17;
        const uint32_t wr = static_cast<uint32_t>(state), wr8 = static_cast<uint32_t>(state >> 32);
        const uint32_t lane_lo = nm::sp_meta_lane_word(wr, wr8, false);   // stored in lane r
        const uint32_t lane_hi = nm::sp_meta_lane_word(wr8, wr, true);    // stored in lane r + 8
        const uint32_t read_r = (lane_lo & 0xFFFFu) | ((lane_hi & 0xFFFFu) << 16);
        const uint32_t read_r8 = (lane_lo >> 16) | (lane_hi & 0xFFFF0000u);
        ++r.checks;
        if (read_r != wr || read_r8 != wr8) {
            if (r.fails < 5)
                std::printf("sp lane words %08x %08x: read back %08x %08x\n", wr, wr8, read_r,
                            read_r8);
            ++r.fails;
        }
    }
    std::printf("2:4s metadata %ld checks, %ld failures\n", r.checks, r.fails);
    return r;
}

}  // namespace

int main()
{
    long fails = 0;
    fails += check_all<2, 4>(0).fails;
    fails += check_all<1, 4>(0).fails;
    fails += check_all<2, 8>(0).fails;
    fails += check_all<4, 8>(0).fails;
    fails += check_all<1, 8>(300000).fails;
    fails += check_all<4, 4>(0).fails;
    fails += check_all<8, 8>(0).fails;
    fails += check_expand().fails;
    fails += check_sp_meta().fails;
    std::printf(fails ? "FAIL\n" : "OK\n");
    return fails ? 1 : 0;
}

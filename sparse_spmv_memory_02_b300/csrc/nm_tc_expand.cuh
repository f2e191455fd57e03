// Expansion of a 2:4 group into dense fp16 positions, for the tensor-core
// product (nm_spmm_tc.cu): the byte-permute selectors that move a group's
// value pair to its two kept positions.  Host-callable, so the table can be
// checked on a machine without a GPU.
#pragma once

#include <cstdint>

#include "nm_device.cuh"

namespace nm {

// Byte-permute selectors that expand a 2:4 group: for nibble n (the group's
// mask bits), the two dense words (positions 0-1 and 2-3) of the group are
// prmt(v, 0, sel & 0xFFFF) and prmt(v, 0, sel >> 16), v = the group's value
// pair: each position takes v's low half (bytes 0-1), its high half (2-3)
// or zero (bytes 4-5 of the zero operand).  Nibbles with other than two set
// bits give zeros or unspecified picks (never an out-of-range byte).
__host__ __device__ constexpr uint32_t expand_sel(uint32_t n)
{
    uint32_t s[4] = {0x54u, 0x54u, 0x54u, 0x54u};
    int j = 0;
    for (int q = 0; q < 4; ++q)
        if ((n >> q) & 1u) {
            if (j == 0) s[q] = 0x10u;
            else if (j == 1) s[q] = 0x32u;
            ++j;
        }
    return s[0] | (s[1] << 8) | (s[2] << 16) | (s[3] << 24);
}

// Sparse-operand metadata of the 2:4 tensor-core product (tcgen05.mma.sp):
// for each group of four positions with two kept, the positions (0-3) of
// the two kept weights, the lower first, two bits each -- code = i0 | i1 << 2
// (0x4, 0x8, 0x9, 0xC, 0xD, 0xE for the six valid groups).  One mask word
// (32 positions, 8 groups) gives one metadata word, group g in bits
// 4g .. 4g+3, the order in which the packed layout stores the group's two
// values.  A valid nibble is identified by its low three bits, so two byte
// permutes look up four groups' codes each; `mode` 1 swaps the two 2-bit
// fields (i1 | i0 << 2).  Invalid groups get some valid code (never an
// out-of-range position).
__host__ __device__ __forceinline__ uint32_t sp_meta_word(uint32_t m, int mode = 0)
{
    // byte i: code of the valid nibble whose low three bits are i
    const uint32_t lo = mode == 1 ? 0x01070301u : 0x040D0C04u;
    const uint32_t hi = mode == 1 ? 0x0106020Bu : 0x0409080Eu;
    const uint32_t p = prmt(lo, hi, m & 0x7777u);          // groups 0-3, one code a byte
    const uint32_t q = prmt(lo, hi, (m >> 16) & 0x7777u);  // groups 4-7
    // byte 0 of p | p >> 4 holds codes 0 and 1, byte 2 codes 2 and 3
    return prmt(p | (p >> 4), q | (q >> 4), 0x6420u);
}

// Tensor-memory layout of that metadata for an M = 128 MMA (found on the
// GPU from a full placement map, see the kernel): rows r and r + 8 of each
// 16-row block share lanes r and r + 8.  Lane r (r % 16 < 8) holds, in its
// low 16 bits, row r's groups 0-3 of the MMA's 32 positions and, in its
// high 16 bits, row r + 8's groups 0-3; lane r + 8 holds the groups 4-7 of
// row r (low half) and of row r + 8 (high half).  Given a lane's own
// metadata word (sp_meta_word of its row) and that of lane ^ 8, the word the
// lane stores:
__host__ __device__ __forceinline__ uint32_t sp_meta_lane_word(uint32_t own, uint32_t partner,
                                                               bool high_lane)
{
    return high_lane ? prmt(own, partner, 0x3276u)   // partner's groups 4-7, then own 4-7
                     : prmt(own, partner, 0x5410u);  // own groups 0-3, then partner's 0-3
}

}  // namespace nm

// Expansion of a 2:4 group into dense fp16 positions, for the tensor-core
// product (nm_spmm_tc.cu): the byte-permute selectors that move a group's
// value pair to its two kept positions.  Host-callable, so the table can be
// checked on a machine without a GPU.
#pragma once

#include <cstdint>

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

}  // namespace nm

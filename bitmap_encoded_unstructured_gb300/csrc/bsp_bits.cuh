// Bit arithmetic on BitmapTile words shared by the decode and prefill
// kernels.
#pragma once

#include <cstdint>

namespace bspx {

// First value index of each of the 8 rows of a BT whose first value is
// `base`: row r starts after the set bits of rows 0..r-1.  Per-byte
// popcounts by the usual bit-slicing sums, their running sum by one
// multiply (bytes <= 32, no carry between them), then spread to u16 pairs
// (r0 | r1 << 16, ..., r6 | r7 << 16).  base + 64 must fit 16 bits.
__device__ __forceinline__ uint4 row_starts(uint64_t bits, uint32_t base)
{
    uint32_t pre[2];
#pragma unroll
    for (int hw = 0; hw < 2; ++hw) {
        uint32_t x = (uint32_t)(bits >> (32 * hw));
        x = x - ((x >> 1) & 0x55555555u);
        x = (x & 0x33333333u) + ((x >> 2) & 0x33333333u);
        x = (x + (x >> 4)) & 0x0F0F0F0Fu;          // popcount of each byte (row)
        const uint32_t incl = x * 0x01010101u;       // byte k: rows 0..k
        pre[hw] = incl << 8;                         // byte k: rows 0..k-1
    }
    const uint32_t lo_total = (uint32_t)__popc((uint32_t)bits);
    const uint32_t b0 = base * 0x10001u, b1 = (base + lo_total) * 0x10001u;
    return make_uint4(__byte_perm(pre[0], 0u, 0x5140) + b0, __byte_perm(pre[0], 0u, 0x5342) + b0,
                      __byte_perm(pre[1], 0u, 0x5140) + b1, __byte_perm(pre[1], 0u, 0x5342) + b1);
}

}  // namespace bspx

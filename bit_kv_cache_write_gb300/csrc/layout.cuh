// Device-side description of the paged INT2 / BF16 layout declared in include/oscar.h.
#pragma once

#include <cstdint>

namespace oscar {

// Bit offset of rotated channel c's 2-bit code inside a K row (d channels).
// One m16n8k16 k-step covers channels 16kk..16kk+15. Quad lane t holds channels
// 16kk+4t+{0,1} in one register and 16kk+4t+{2,3} in the other. So lane t's
// codes for all k-steps form one run of 8n bits, with the pair of k-step kk at
// positions 2(kk%4) and 2(kk%4)+1 of 32-bit word kk/4, low half-word first.
__host__ __device__ constexpr int k_bit_offset(int c, int d) {
    return 8 * (d / 16) * ((c % 16) / 4) + 32 * ((c / 16) / 4) + 16 * ((c % 4) % 2) +
           2 * (2 * ((c / 16) % 4) + (c % 4) / 2);
}

// Bit offset of rotated channel c's code inside a V row. One m-step covers
// channels 16m..16m+15 as fragment rows r = c%16. The lane that owns rows r and
// r+8 finds code m of row r at bit 2m of its (2n)-bit unit 2r, and of row r+8 in
// unit 2r+1.
__host__ __device__ constexpr int v_bit_offset(int c, int d) {
    return 4 * (d / 16) * ((c % 16) % 8) + 2 * (d / 16) * ((c % 16) / 8) + 2 * (c / 16);
}

template <int D, int G>
struct Geo {
    static constexpr int kCodeRow = D / 4;                 // bytes of codes per token
    static constexpr int kGroups = D / G;
    static constexpr int kCodeBytes = 16 * kCodeRow;      // per page segment
    static constexpr int kSzBytes = 16 * kGroups * 4;
    static constexpr int kSeg = kCodeBytes + kSzBytes;    // K or V segment of one (page, head)
    static constexpr int kBlock = 2 * kSeg;               // one (page, head)
};

__device__ __forceinline__ void record_error(int* kind_word, long long* index_word, int kind, long long idx) {
    if (atomicCAS(kind_word, 0, kind) == 0) *index_word = idx;
}

}  // namespace oscar

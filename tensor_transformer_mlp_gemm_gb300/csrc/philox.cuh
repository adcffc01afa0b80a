// philox.cuh -- Philox4x32-10, the counter-based generator of Salmon, Moraes,
// Dror and Shaw ("Parallel random numbers: as easy as 1, 2, 3", SC'11), for the
// dropout masks of the sequence-parallel sublayer.
//
// Ten rounds on a 4-word counter with a 2-word key; each round multiplies
// words 0 and 2 by the two round multipliers, crosses the high halves with the
// other two words and the key, and the key advances by the two Weyl constants
// between rounds.  Mask convention (shared with the host-side description in
// include/tpmlp.h): element e of a row-major [T, h] tensor reads word e % 4 of
// the output for counter (lo, hi, 0, 0) of offset + e / 4 and key (seed_lo,
// seed_hi), and is kept iff that word is below the keep threshold
// floor((1 - p) * 2^32).
#pragma once

#include <cstdint>

namespace tpmlp {

struct PhiloxOut {
    uint32_t w[4];
};

__device__ __forceinline__ PhiloxOut philox4x32_10(uint64_t counter, uint64_t seed) {
    constexpr uint32_t kMul0 = 0xD2511F53u, kMul1 = 0xCD9E8D57u;
    constexpr uint32_t kWeyl0 = 0x9E3779B9u, kWeyl1 = 0xBB67AE85u;
    uint32_t c0 = static_cast<uint32_t>(counter), c1 = static_cast<uint32_t>(counter >> 32);
    uint32_t c2 = 0u, c3 = 0u;
    uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t hi0 = __umulhi(kMul0, c0), lo0 = kMul0 * c0;
        const uint32_t hi1 = __umulhi(kMul1, c2), lo1 = kMul1 * c2;
        const uint32_t n0 = hi1 ^ c1 ^ k0;
        const uint32_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
        k0 += kWeyl0;
        k1 += kWeyl1;
    }
    return PhiloxOut{{c0, c1, c2, c3}};
}

// Dropout parameters as the kernels see them.  The forward pass draws the
// mask and, when `mask` is set, also stores it as bits: bit n % 32 of word
// row * mask_words + n / 32 is the keep decision of element (row, n), so the
// backward pass reads 1 bit per element instead of drawing the mask again.
struct DropoutParams {
    uint64_t seed;
    uint64_t offset;   // counter offset in 4-element blocks
    uint64_t thresh;   // keep iff word < thresh, thresh in [0, 2^32]
    float scale;       // 1 / (1 - p)
    uint32_t* mask;    // [rows][mask_words] keep bits (null: not stored)
    long long mask_words;
};

}  // namespace tpmlp

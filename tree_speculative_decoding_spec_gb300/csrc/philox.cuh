// Philox4x32-10 on the device.
//
// Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3"
// (SC'11): a keyed bijection of a 4 x 32-bit counter built from 10 rounds.  A
// round multiplies words 0 and 2 by two fixed odd constants, keeps the high and
// low halves of both 64-bit products, XORs the high halves with words 3/1 and
// the two key words, and permutes; the key gets a Weyl increment between rounds.
#pragma once

#include <cstdint>

namespace spec {

struct Philox4 {
    uint32_t w[4];
};

__host__ __device__ __forceinline__ uint32_t mulhi32(uint32_t a, uint32_t b) {
#ifdef __CUDA_ARCH__
    return __umulhi(a, b);
#else
    return static_cast<uint32_t>((static_cast<uint64_t>(a) * b) >> 32);
#endif
}

__host__ __device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                         uint32_t k0, uint32_t k1) {
    constexpr uint32_t kMul0 = 0xD2511F53u, kMul1 = 0xCD9E8D57u;
    constexpr uint32_t kWeyl0 = 0x9E3779B9u, kWeyl1 = 0xBB67AE85u;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t hi0 = mulhi32(kMul0, c0), lo0 = kMul0 * c0;
        const uint32_t hi1 = mulhi32(kMul1, c2), lo1 = kMul1 * c2;
        const uint32_t n0 = hi1 ^ c1 ^ k0;
        const uint32_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
        k0 += kWeyl0; k1 += kWeyl1;
    }
    return Philox4{{c0, c1, c2, c3}};
}

// Top 24 bits of a word as a uniform in [0, 1): exact in fp32.
__host__ __device__ __forceinline__ float uniform24(uint32_t x) {
    return static_cast<float>(x >> 8) * (1.0f / 16777216.0f);
}

// The library's draw for (node, seq) under (seed, offset): key = seed halves,
// counter = (node, seq, offset halves).
__host__ __device__ __forceinline__ Philox4 spec_draw(uint64_t seed, uint64_t offset, uint32_t node, uint32_t seq) {
    return philox4x32_10(node, seq, static_cast<uint32_t>(offset), static_cast<uint32_t>(offset >> 32),
                         static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
}

}  // namespace spec

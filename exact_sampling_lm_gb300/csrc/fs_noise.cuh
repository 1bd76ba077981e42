// fs_noise.cuh -- counter-based Gumbel noise of the sampling epilogue.
//
// FlashSampling's method section draws i.i.d. Gumbels g_i and perturbs the
// logits (s_i = l~_i + g_i).  For the fused kernel the draw must depend only
// on (seed, offset, row, vocabulary index) so that any tiling of the
// vocabulary sees the same noise.  Generator: Philox4x64-10 (Salmon, Moraes,
// Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11), key
// (seed, 0), counter (v >> 3, b, offset, 0).  One call yields four 64-bit
// words = eight 32-bit draws, one per vocabulary index v .. v+7 (v a multiple
// of 8): draw j is half (j & 1) (low half first) of word j >> 1.
#pragma once

#include <stdint.h>

namespace fs {

struct Philox4x64Out {
    uint64_t w[4];
};

// Ten rounds of the 4x64 Philox bijection.  Per round: the two 64x64->128
// products of words 0 and 2 with the round multipliers; the high halves are
// xored with words 1 / 3 and the round key; the low halves move to words 3 / 1.
// The key advances by the two Weyl increments between rounds.
__device__ __forceinline__ Philox4x64Out philox4x64_10(uint64_t c0, uint64_t c1, uint64_t c2,
                                                      uint64_t c3, uint64_t k0, uint64_t k1) {
    constexpr uint64_t kMul0 = 0xD2E7470EE14C6C93ull;
    constexpr uint64_t kMul1 = 0xCA5A826395121157ull;
    constexpr uint64_t kWeyl0 = 0x9E3779B97F4A7C15ull;
    constexpr uint64_t kWeyl1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint64_t lo0 = kMul0 * c0;
        const uint64_t hi0 = __umul64hi(kMul0, c0);
        const uint64_t lo1 = kMul1 * c2;
        const uint64_t hi1 = __umul64hi(kMul1, c2);
        const uint64_t n0 = hi1 ^ c1 ^ k0;
        const uint64_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
        k0 += kWeyl0;
        k1 += kWeyl1;
    }
    Philox4x64Out o;
    o.w[0] = c0;
    o.w[1] = c1;
    o.w[2] = c2;
    o.w[3] = c3;
    return o;
}

// The eight 32-bit draws of vocabulary indices v8*8 .. v8*8+7 of row b.
__device__ __forceinline__ void noise_words8(uint64_t seed, uint64_t offset, uint64_t b,
                                             uint64_t v8, uint32_t (&x)[8]) {
    const Philox4x64Out o = philox4x64_10(v8, b, offset, 0ull, seed, 0ull);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        x[2 * j] = static_cast<uint32_t>(o.w[j]);
        x[2 * j + 1] = static_cast<uint32_t>(o.w[j] >> 32);
    }
}

// u = ((x >> 8) | 1) * 2^-24: exact in f32, never 0 or 1, symmetric about 1/2.
__device__ __forceinline__ float uniform_from_word(uint32_t x) {
    return static_cast<float>((x >> 8) | 1u) * 0x1p-24f;
}

// g = -log(-log(u)) with CUDA's accurate single-precision logf (not the
// approximate __logf, whose absolute error is fatal near u = 1 where -log(u)
// is tiny).  The two roundings keep |g - g_exact| within a few ulp of g plus
// about 1e-7 absolute.
__device__ __forceinline__ float gumbel_from_word(uint32_t x) {
    const float u = uniform_from_word(x);
    const float e = -logf(u);
    return -logf(e);
}

}  // namespace fs

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

constexpr uint64_t kPhiloxMul0 = 0xD2E7470EE14C6C93ull;
constexpr uint64_t kPhiloxMul1 = 0xCA5A826395121157ull;
constexpr uint64_t kPhiloxWeyl0 = 0x9E3779B97F4A7C15ull;
constexpr uint64_t kPhiloxWeyl1 = 0xBB67AE8584CAA73Bull;

// One round of the 4x64 Philox bijection: the two 64x64->128 products of
// words 0 and 2 with the round multipliers; the high halves are xored with
// words 1 / 3 and the round key; the low halves move to words 3 / 1.
__device__ __forceinline__ void philox_round(uint64_t &c0, uint64_t &c1, uint64_t &c2,
                                             uint64_t &c3, uint64_t k0, uint64_t k1) {
    const uint64_t lo0 = kPhiloxMul0 * c0;
    const uint64_t hi0 = __umul64hi(kPhiloxMul0, c0);
    const uint64_t lo1 = kPhiloxMul1 * c2;
    const uint64_t hi1 = __umul64hi(kPhiloxMul1, c2);
    c0 = hi1 ^ c1 ^ k0;
    c1 = lo1;
    c2 = hi0 ^ c3 ^ k1;
    c3 = lo0;
}

// Per-row constants of the counter (v >> 3, b, offset, 0): the product of
// word 2 (= offset) in round 1 and, through it, the product of word 0 in
// round 2 do not depend on v.  Precomputing them saves 2 of the 20 products
// of every call; the result is bit-identical to the plain ten rounds.
struct PhiloxRow {
    uint64_t seed;
    uint64_t r1_c0_part;  // round 1: hi(M1*offset) ^ b ^ k0   (new word 0)
    uint64_t r1_c1;       // round 1: lo(M1*offset)            (new word 1)
    uint64_t r2_hi0;      // round 2: hi(M0 * new word 0)
    uint64_t r2_lo0;      // round 2: lo(M0 * new word 0)      (new word 3)
};

__device__ __forceinline__ PhiloxRow philox_row(uint64_t seed, uint64_t offset, uint64_t b) {
    PhiloxRow r;
    r.seed = seed;
    const uint64_t lo1 = kPhiloxMul1 * offset;
    const uint64_t hi1 = __umul64hi(kPhiloxMul1, offset);
    r.r1_c0_part = hi1 ^ b ^ seed;  // key word 0 of round 1 is the seed
    r.r1_c1 = lo1;
    r.r2_hi0 = __umul64hi(kPhiloxMul0, r.r1_c0_part);
    r.r2_lo0 = kPhiloxMul0 * r.r1_c0_part;
    return r;
}

// The eight 32-bit draws of vocabulary indices 8*v8 .. 8*v8+7 of the row.
__device__ __forceinline__ void noise_words8(const PhiloxRow &row, uint64_t v8,
                                             uint32_t (&x)[8]) {
    // round 1 (key seed, 0): word 0 = v8 varies, word 2 = offset is per row
    const uint64_t lo0 = kPhiloxMul0 * v8;
    const uint64_t hi0 = __umul64hi(kPhiloxMul0, v8);
    uint64_t c0 = row.r1_c0_part;
    uint64_t c1 = row.r1_c1;
    uint64_t c2 = hi0;  // ^ word 3 (0) ^ key word 1 (0)
    uint64_t c3 = lo0;
    // round 2 (key + Weyl): word 0's product is per row
    {
        const uint64_t k0 = row.seed + kPhiloxWeyl0;
        const uint64_t k1 = kPhiloxWeyl1;
        const uint64_t lo1 = kPhiloxMul1 * c2;
        const uint64_t hi1 = __umul64hi(kPhiloxMul1, c2);
        const uint64_t n0 = hi1 ^ c1 ^ k0;
        const uint64_t n2 = row.r2_hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = row.r2_lo0;
    }
#pragma unroll
    for (int r = 2; r < 10; ++r)
        philox_round(c0, c1, c2, c3, row.seed + kPhiloxWeyl0 * static_cast<uint64_t>(r),
                     kPhiloxWeyl1 * static_cast<uint64_t>(r));
    const uint64_t w[4] = {c0, c1, c2, c3};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        x[2 * j] = static_cast<uint32_t>(w[j]);
        x[2 * j + 1] = static_cast<uint32_t>(w[j] >> 32);
    }
}

// A whole Philox4x64-10 block for an arbitrary counter (used off the hot
// path: the grouped sampler's draws, counter word 3 = 1).
__device__ __forceinline__ void philox4x64_10_block(uint64_t c0, uint64_t c1, uint64_t c2,
                                                    uint64_t c3, uint64_t seed,
                                                    uint64_t (&w)[4]) {
#pragma unroll
    for (int r = 0; r < 10; ++r)
        philox_round(c0, c1, c2, c3, seed + kPhiloxWeyl0 * static_cast<uint64_t>(r),
                     kPhiloxWeyl1 * static_cast<uint64_t>(r));
    w[0] = c0;
    w[1] = c1;
    w[2] = c2;
    w[3] = c3;
}

// The uniform of a 32-bit word x is u = k * 2^-24 with k = (x >> 8) | 1: exact
// in f32, never 0 or 1, symmetric about 1/2.

// log2(x) from the hardware approximation (absolute error about 2^-22).
__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// w = -log(u) for u = k * 2^-24 (k odd, 0 < k < 2^24), within about 1 ulp.
// For u >= 15/16 -- the only u that can still win once a row's running best
// is established, since the screen only passes u above exp(-exp(-d)) -- the
// Mercator series -log(1 - e) = e + e^2/2 + e^3/3 + ... in e = 1 - u, which
// is exact in f32 here.  Six terms: the dropped tail (e^n/n for n >= 7) is
// below e^6/7 * 1/(1-e) <= 2^-24/6 relative to w for e <= 2^-4, well under
// half an ulp.
// Otherwise CUDA's accurate logf.  (The approximate __logf is not usable for
// this inner logarithm: its absolute error is fatal near u = 1, where w is
// tiny and the Gumbel large.)
constexpr uint32_t kSeriesMinK = 15u << 20;  // u >= 15/16
__device__ __forceinline__ float neglog_uniform(uint32_t k) {
    if (k >= kSeriesMinK) {
        const float e = static_cast<float>((1u << 24) - k) * 0x1p-24f;  // exact
        float p = fmaf(e, 1.0f / 6.0f, 0.2f);
        p = fmaf(p, e, 0.25f);
        p = fmaf(p, e, 1.0f / 3.0f);
        p = fmaf(p, e, 0.5f);
        p = fmaf(p, e, 1.0f);
        return p * e;
    }
    return -logf(static_cast<float>(k) * 0x1p-24f);
}

// g = -log(w), w = -log(u) in [6e-8, 16.7], from the hardware log2: its
// absolute error (about 2^-22 in log2) becomes about 1e-7 in g, below an
// ulp of any score s = l~ + g with |s| >= 1 and far below the screen's
// slack; w's own error (about 1 ulp, relative) adds another 1e-7.
__device__ __forceinline__ float gumbel_from_word(uint32_t x) {
    const float w = neglog_uniform((x >> 8) | 1u);
    return -0.69314718055994531f * lg2_approx(w);
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Screen of the argmax, one test per element.  An element with transformed
// logit lt can beat the running best only if its Gumbel g = -log(w), with
// w = -log(u), exceeds best - lt.  Because -log(u) >= 1 - u, w is at least
// the tail 1 - u = 2^-24 (2^24 - k) >= 2^-23 e2, where e2 = (~x) >> 9 is the
// top 23 bits of the complemented word (k = (x >> 8) | 1).  So the element
// can win only if 2^-23 e2 < exp(lt - best), i.e. if
//     lg2(e2) < (lt - best) log2(e) + 23.
// screen_lg2_tail gives lg2(e2) from the hardware log2 (e2 = 0 gives -inf,
// which always passes); screen_bound gives the right-hand side plus a margin
// of 2^-8 in log2 units (2.7e-3 in natural units).  The margin covers the
// computed Gumbel's error (a few 1e-6), the hardware log2's error (below 1e-5
// for results up to 23), and the roundings of lt - best and of the fma, which
// are tiny wherever |lt - best| is small enough for the test to be close.  A
// rejected element therefore has lt + g < best in exact arithmetic, so its
// rounded score cannot exceed best: the screened scan returns what the
// unscreened one does.  Non-finite cases: best = -inf makes the bound +inf
// (everything passes); a NaN lt - best fails the comparison, and such an
// element could not win either.
constexpr float kScreenBias = 23.0f + 0x1p-8f;

__device__ __forceinline__ float screen_lg2_tail(uint32_t x) {
    const uint32_t e2 = (~x) >> 9;                                   // below 2^23
    const float f = __uint_as_float(0x4B000000u | e2) - 8388608.0f;  // e2, exactly
    return lg2_approx(f);
}

__device__ __forceinline__ float screen_bound(float lt, float best) {
    return fmaf(lt - best, 1.4426950408889634f, kScreenBias);
}

}  // namespace fs

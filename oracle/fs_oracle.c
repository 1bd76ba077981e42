/*
 * fs_oracle.c -- CPU oracle for FlashSampling's fused LM-head + exact sampling.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the GPU path computes.  Only the tests, the smoke check
 * and the benchmark's CPU-baseline leg may load it.  It shares no code, header,
 * table or constant with the CUDA library and includes nothing from it.
 *
 * What it computes (FlashSampling: Fast and Memory-Efficient Exact Sampling):
 *  - the Gumbel-max rule of the method section: draw i.i.d. Gumbels g_i, form
 *    s_i = l~_i + g_i and return argmax_i s_i (the pages point to Algorithm I.1
 *    of the Appendix for it);
 *  - one untiled Gumbel-max over the whole vocabulary: the paper's exactness
 *    statement (tiled argmax gives the same maximizer, Appendix C) means the
 *    reference result is the full, untiled pass, which is what is written here;
 *  - l = H W^T of the LM head (Section 3 IO model: the GEMM reads W and H);
 *  - l~ = l / T, the one deterministic transform applied before the noise.
 *
 * Readings where the pages are silent (each one is listed in the design notes):
 *  - logits: bf16 inputs with f32 accumulation (the experimental setup's
 *    precision): each product of two bf16 values is exact in f32, and the
 *    sum runs in f32 in index order k = 0..D-1, rounded after every addition.
 *    An fp64 sum of the same products is kept for diagnostics only;
 *  - temperature: invT = 1.0f / T in f32, l~ = l * invT in f32; rows whose T is
 *    not finite or not > 0 get index -1 and score NaN (greedy is not part of the
 *    method, Section 5 GSM8K paragraph);
 *  - noise: Philox4x64-10 (Salmon, Moraes, Dror, Shaw, SC'11) with
 *    key = (seed, 0) and counter = (v >> 3, b, offset, 0); element v of row b
 *    takes 64-bit word (v & 7) >> 1 of that block, low half when v is even and
 *    high half when v is odd;
 *  - uniform: u = ((x >> 8) | 1) * 2^-24, so u is never 0 or 1;
 *  - Gumbel: g = -log(-log(u)) evaluated in double and rounded to f32;
 *  - score: s = l~ + g in f32; argmax keeps the first (lowest) index on ties,
 *    NaN never wins, and a row with no finite winner reports index -1.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fPIC -shared (oracle/build.py).
 * -ffp-contract=off keeps l * invT + g as two roundings, as specified.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------------------
 * Philox4x64-10 (SC'11, Section 4: the Philox family; 4 words of 64 bits,
 * 10 rounds).  Round: two 64x64->128 multiplications by the round multipliers,
 * xor of the high halves with the other two words and the round key, and the
 * fixed word permutation of the 4-word variant.  The key is bumped by the two
 * Weyl constants between rounds.
 * ------------------------------------------------------------------------- */
static const uint64_t PHILOX_M0 = 0xD2E7470EE14C6C93ULL;
static const uint64_t PHILOX_M1 = 0xCA5A826395121157ULL;
static const uint64_t PHILOX_W0 = 0x9E3779B97F4A7C15ULL; /* golden ratio */
static const uint64_t PHILOX_W1 = 0xBB67AE8584CAA73BULL; /* sqrt(3) - 1  */

static void mulhilo64(uint64_t a, uint64_t b, uint64_t *hi, uint64_t *lo) {
    unsigned __int128 p = (unsigned __int128)a * (unsigned __int128)b;
    *lo = (uint64_t)p;
    *hi = (uint64_t)(p >> 64);
}

void oracle_philox4x64_10(const uint64_t ctr_in[4], const uint64_t key_in[2],
                          uint64_t out[4]) {
    uint64_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint64_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += PHILOX_W0;
            k1 += PHILOX_W1;
        }
        uint64_t hi0, lo0, hi1, lo1;
        mulhilo64(PHILOX_M0, c0, &hi0, &lo0);
        mulhilo64(PHILOX_M1, c2, &hi1, &lo1);
        uint64_t n0 = hi1 ^ c1 ^ k0;
        uint64_t n1 = lo1;
        uint64_t n2 = hi0 ^ c3 ^ k1;
        uint64_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The 32-bit random word that element (b, v) draws. */
uint32_t oracle_noise_word(uint64_t seed, uint64_t offset, int64_t b, int64_t v) {
    uint64_t ctr[4] = {(uint64_t)v >> 3, (uint64_t)b, offset, 0};
    uint64_t key[2] = {seed, 0};
    uint64_t blk[4];
    oracle_philox4x64_10(ctr, key, blk);
    uint64_t w = blk[((uint64_t)v & 7) >> 1];
    return ((uint64_t)v & 1) ? (uint32_t)(w >> 32) : (uint32_t)(w & 0xFFFFFFFFULL);
}

/* u = ((x >> 8) | 1) / 2^24: an odd 24-bit numerator over 2^24. */
double oracle_uniform(uint32_t x) {
    uint32_t k = (x >> 8) | 1u;
    return (double)k / 16777216.0;
}

/* g = -log(-log(u)), in double, then rounded to f32. */
float oracle_gumbel_from_word(uint32_t x) {
    double u = oracle_uniform(x);
    double e = -log(u);
    return (float)(-log(e));
}

float oracle_gumbel(uint64_t seed, uint64_t offset, int64_t b, int64_t v) {
    return oracle_gumbel_from_word(oracle_noise_word(seed, offset, b, v));
}

/* Noise block for rows [b0, b0+nb) and vocab [v0, v0+nv): words and Gumbels,
 * row-major [nb, nv].  Either output may be NULL. */
void oracle_noise_block(uint64_t seed, uint64_t offset, int64_t b0, int64_t nb,
                        int64_t v0, int64_t nv, uint32_t *words, float *g,
                        int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < nb * nv; ++i) {
        int64_t b = b0 + i / nv;
        int64_t v = v0 + i % nv;
        uint32_t x = oracle_noise_word(seed, offset, b, v);
        if (words) words[i] = x;
        if (g) g[i] = oracle_gumbel_from_word(x);
    }
}

/* Vectorised forms used by the exhaustive tests: u and g for given words. */
void oracle_uniform_block(const uint32_t *x, int64_t n, double *u) {
    for (int64_t i = 0; i < n; ++i) u[i] = oracle_uniform(x[i]);
}

void oracle_gumbel_block(const uint32_t *x, int64_t n, float *g, int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) g[i] = oracle_gumbel_from_word(x[i]);
}

/* ---------------------------------------------------------------------------
 * LM-head logits l[b, v] = sum_k H[b, k] * W[v, k].
 * H is [B, D] and W is [V, D], both row-major bf16 given as raw 16-bit words.
 * bf16 -> f32 is exact, and so is the f32 product of two bf16 values (8 + 8
 * significant bits fit in 24).  The sum runs in f32 in index order
 * k = 0..D-1 and is rounded to f32 after every addition; -ffp-contract=off
 * keeps each product and addition apart (no fused multiply-add).
 * ------------------------------------------------------------------------- */
static float bf16_to_float(uint16_t h) {
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

static float dot_row(const uint16_t *h, const uint16_t *w, int64_t D) {
    float acc = 0.0f;
    for (int64_t k = 0; k < D; ++k) {
        float p = bf16_to_float(h[k]) * bf16_to_float(w[k]);
        acc = acc + p;
    }
    return acc;
}

/* Diagnostic only: the same exact products summed in fp64 in index order. */
static double dot_row64(const uint16_t *h, const uint16_t *w, int64_t D) {
    double acc = 0.0;
    for (int64_t k = 0; k < D; ++k)
        acc += (double)bf16_to_float(h[k]) * (double)bf16_to_float(w[k]);
    return acc;
}

void oracle_logits(const uint16_t *H, const uint16_t *W, int64_t B, int64_t V,
                   int64_t D, float *out, int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < B * V; ++i) {
        int64_t b = i / V, v = i % V;
        out[i] = dot_row(H + b * D, W + v * D, D);
    }
}

void oracle_logits64(const uint16_t *H, const uint16_t *W, int64_t B, int64_t V,
                     int64_t D, double *out, int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < B * V; ++i) {
        int64_t b = i / V, v = i % V;
        out[i] = dot_row64(H + b * D, W + v * D, D);
    }
}

/* ---------------------------------------------------------------------------
 * The full Gumbel-max pass for one row, given that row's f32 logits.
 *   invT = 1/T (f32), l~ = l * invT (f32), s = l~ + g (f32),
 *   idx = first v with the largest s; top2 = largest s over v != idx.
 * scores (optional, [V]) receives s for every v.
 * ------------------------------------------------------------------------- */
static int temperature_ok(float T) { return isfinite(T) && T > 0.0f; }

static void argmax_row(const float *s, int64_t V, int64_t *idx, float *best,
                       float *second) {
    float b1 = -INFINITY, b2 = -INFINITY;
    int64_t i1 = -1;
    for (int64_t v = 0; v < V; ++v) {
        float x = s[v];
        if (x > b1) {
            b2 = b1;
            b1 = x;
            i1 = v;
        } else if (x > b2) {
            b2 = x;
        }
    }
    *idx = i1;
    *best = b1;
    *second = b2;
}

#define ORACLE_NO_NOISE 1u

/* One row b of the full pass.  l32: that row's f32 logits [V].  s: scratch
 * [V] that receives the perturbed scores. */
static void sample_row(const float *l32, int64_t b, int64_t V, float Tb,
                       uint64_t seed, uint64_t offset, uint32_t flags, float *s,
                       int64_t *idx, float *best, float *second) {
    if (!temperature_ok(Tb)) {
        for (int64_t v = 0; v < V; ++v) s[v] = NAN;
        *idx = -1;
        *best = NAN;
        *second = NAN;
        return;
    }
    float invT = 1.0f / Tb;
    #pragma omp parallel for schedule(static)
    for (int64_t v = 0; v < V; ++v) {
        float lt = l32[v] * invT;
        float g = (flags & ORACLE_NO_NOISE) ? 0.0f : oracle_gumbel(seed, offset, b, v);
        s[v] = lt + g;
    }
    argmax_row(s, V, idx, best, second);
}

/* Sample one index per row from given f32 logits [B, V] (row-major).
 * T: per-row temperatures [B] (the caller broadcasts a scalar).
 * row_ids: NULL, or the row index b that each of the B given rows has in the
 * full batch (it keys the noise counter); NULL means 0..B-1.
 * out_idx [B], out_score [B], out_second [B]; out_scores [B, V] may be NULL. */
void oracle_sample_from_logits(const float *logits, int64_t B, int64_t V,
                               const float *T, const int64_t *row_ids, uint64_t seed,
                               uint64_t offset, uint32_t flags, int64_t *out_idx,
                               float *out_score, float *out_second, float *out_scores,
                               int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
    float *s = (float *)malloc(sizeof(float) * (size_t)(V > 0 ? V : 1));
    for (int64_t b = 0; b < B; ++b) {
        int64_t row = row_ids ? row_ids[b] : b;
        sample_row(logits + b * V, row, V, T[b], seed, offset, flags, s, &out_idx[b],
                   &out_score[b], &out_second[b]);
        if (out_scores) memcpy(out_scores + b * V, s, sizeof(float) * (size_t)V);
    }
    free(s);
}

/* The whole hot path from H and W: the f32 logits, then the full Gumbel-max
 * pass.  row_ids as for oracle_sample_from_logits.  out_logits [B, V] (f32,
 * optional) receives the logits the pass sampled from, for the logits
 * tolerance checks. */
void oracle_sample(const uint16_t *H, const uint16_t *W, int64_t B, int64_t V,
                   int64_t D, const float *T, const int64_t *row_ids, uint64_t seed,
                   uint64_t offset, uint32_t flags, int64_t *out_idx, float *out_score,
                   float *out_second, float *out_logits, int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
    float *l32 = (float *)malloc(sizeof(float) * (size_t)(V > 0 ? V : 1));
    float *s = (float *)malloc(sizeof(float) * (size_t)(V > 0 ? V : 1));
    for (int64_t b = 0; b < B; ++b) {
        const uint16_t *h = H + b * D;
        #pragma omp parallel for schedule(static)
        for (int64_t v = 0; v < V; ++v) l32[v] = dot_row(h, W + v * D, D);
        if (out_logits) memcpy(out_logits + b * V, l32, sizeof(float) * (size_t)V);
        int64_t row = row_ids ? row_ids[b] : b;
        sample_row(l32, row, V, T[b], seed, offset, flags, s, &out_idx[b],
                   &out_score[b], &out_second[b]);
    }
    free(l32);
    free(s);
}

/* ---------------------------------------------------------------------------
 * Log-probability of a sampled token under softmax(l~): l~[idx] - log sum_v
 * exp(l~[v]), with l~ = fl(l * fl(1/T)) in f32 as in the sampling pass and the
 * log-sum-exp evaluated in fp64 as (l~[idx] - max) - log sum exp(l~ - max).  This is the
 * per-shard log-mass that the grouped / tensor-parallel variant returns,
 * reduced here over the whole vocabulary.  Reading for non-finite
 * values (the pages are silent): the log-mass runs over the finite l~ only,
 * and a sampled token whose l~ is not finite gets NaN.  For each row of f32 logits
 * [B, V]: out[b] = logprob of idx[b] (NaN when idx[b] < 0 or T[b] invalid).
 * ------------------------------------------------------------------------- */
void oracle_logprob(const float *logits, int64_t B, int64_t V, const float *T,
                    const int64_t *idx, double *out) {
    for (int64_t b = 0; b < B; ++b) {
        float Tb = T[b];
        if (!temperature_ok(Tb) || idx[b] < 0 || idx[b] >= V) {
            out[b] = NAN;
            continue;
        }
        float invT = 1.0f / Tb;
        const float *l = logits + b * V;
        double win = (double)(l[idx[b]] * invT);
        double mx = -INFINITY;
        for (int64_t v = 0; v < V; ++v) {
            double x = (double)(l[v] * invT);
            if (isfinite(x) && x > mx) mx = x;
        }
        double sum = 0.0;
        for (int64_t v = 0; v < V; ++v) {
            double x = (double)(l[v] * invT);
            if (isfinite(x)) sum += exp(x - mx);
        }
        out[b] = (isfinite(win) && sum > 0.0) ? (win - mx) - log(sum) : NAN;
    }
}

/* ---------------------------------------------------------------------------
 * Deterministic transforms applied to the f32 logits before the temperature
 * (method section: Stage 1 applies deterministic transforms before the noise;
 * the pages do not list them -- this library offers the common ones), in this
 * order, each rounded to f32:
 *   l' = l + bias[v]                         (bias may be NULL)
 *   l' = c * tanh(l' / c)      if c > 0      (logit soft-capping)
 *   l' = -inf                  if mask given and bit (v & 31) of
 *                              mask[b * mask_words + (v >> 5)] is 0
 * then the usual l~ = l' * fl(1/T).  In place on logits [B, V].
 * ------------------------------------------------------------------------- */
void oracle_transform_logits(float *logits, int64_t B, int64_t V, const float *bias,
                             float softcap, const uint32_t *mask, int64_t mask_words) {
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t v = 0; v < V; ++v) {
            float l = logits[b * V + v];
            if (bias) l = l + bias[v];
            if (softcap > 0.0f) l = softcap * tanhf(l / softcap);
            if (mask && !((mask[b * mask_words + (v >> 5)] >> (v & 31)) & 1u)) l = -INFINITY;
            logits[b * V + v] = l;
        }
    }
}

/* ---------------------------------------------------------------------------
 * Grouped (hierarchical) sampling, the pages' variant for online and
 * tensor-parallel settings: each group of the vocabulary returns a local
 * sample and its local log-mass; a group is drawn with probability
 * proportional to exp(log-mass), and its local sample is returned.  Exact by
 * P(v) = P(group(v)) * P(v | group(v)).
 *
 * oracle_sample_shard: the local sample of rows [B] over the vocabulary slice
 * W_shard [Vs, D] whose first row has global index vocab_offset: the full
 * Gumbel-max pass over the slice with the noise of the global indices, plus
 * the log-mass log sum exp(l~) over the slice's finite l~ (fp64; -inf if
 * none; NaN for an invalid T).  out_idx are global indices.
 *
 * oracle_combine_groups: per row b, the group g maximising the f32 sum
 * logmass[g][b] + G(g) (f32 log-masses: the decision is taken in the
 * kernel's precision), G from Philox4x64-10 with key (seed, 0) and counter
 * (g >> 3, b, offset, 1) (word 3 = 1 separates these draws from the token
 * noise), ties to the lower g, NaN / -inf never win; out_idx[b] =
 * group_idx[g][b] (or -1), out_group[b] = g (or -1), and the two best sums.
 * ------------------------------------------------------------------------- */
static uint32_t group_noise_word(uint64_t seed, uint64_t offset, int64_t b, int64_t g) {
    uint64_t ctr[4] = {(uint64_t)g >> 3, (uint64_t)b, offset, 1};
    uint64_t key[2] = {seed, 0};
    uint64_t blk[4];
    oracle_philox4x64_10(ctr, key, blk);
    uint64_t w = blk[((uint64_t)g & 7) >> 1];
    return ((uint64_t)g & 1) ? (uint32_t)(w >> 32) : (uint32_t)(w & 0xFFFFFFFFULL);
}

float oracle_group_gumbel(uint64_t seed, uint64_t offset, int64_t b, int64_t g) {
    return oracle_gumbel_from_word(group_noise_word(seed, offset, b, g));
}

void oracle_sample_shard(const uint16_t *H, const uint16_t *W_shard, int64_t B, int64_t Vs,
                         int64_t D, int64_t vocab_offset, const float *T, uint64_t seed,
                         uint64_t offset, int64_t *out_idx, float *out_score,
                         float *out_second, double *out_logmass, int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
    float *lt = (float *)malloc(sizeof(float) * (size_t)(Vs > 0 ? Vs : 1));
    for (int64_t b = 0; b < B; ++b) {
        float Tb = T[b];
        if (!temperature_ok(Tb)) {
            out_idx[b] = -1;
            out_score[b] = NAN;
            out_second[b] = NAN;
            out_logmass[b] = NAN;
            continue;
        }
        float invT = 1.0f / Tb;
        const uint16_t *h = H + b * D;
        #pragma omp parallel for schedule(static)
        for (int64_t v = 0; v < Vs; ++v) lt[v] = dot_row(h, W_shard + v * D, D) * invT;
        float best = -INFINITY, second = -INFINITY;
        int64_t bi = -1;
        double mx = -INFINITY;
        for (int64_t v = 0; v < Vs; ++v) {
            float s = lt[v] + oracle_gumbel(seed, offset, b, vocab_offset + v);
            if (s > best) {
                second = best;
                best = s;
                bi = vocab_offset + v;
            } else if (s > second) {
                second = s;
            }
            if (isfinite(lt[v]) && (double)lt[v] > mx) mx = (double)lt[v];
        }
        double sum = 0.0;
        for (int64_t v = 0; v < Vs; ++v)
            if (isfinite(lt[v])) sum += exp((double)lt[v] - mx);
        out_idx[b] = bi;
        out_score[b] = best;
        out_second[b] = second;
        out_logmass[b] = sum > 0.0 ? mx + log(sum) : -INFINITY;
    }
    free(lt);
}

void oracle_combine_groups(int64_t n_groups, int64_t B, const int64_t *group_idx,
                           const float *group_logmass, uint64_t seed, uint64_t offset,
                           int64_t *out_idx, int64_t *out_group, float *out_best,
                           float *out_second) {
    for (int64_t b = 0; b < B; ++b) {
        float best = -INFINITY, second = -INFINITY;
        int64_t gbest = -1;
        for (int64_t g = 0; g < n_groups; ++g) {
            float s = group_logmass[g * B + b] + oracle_group_gumbel(seed, offset, b, g);
            if (s > best) {
                second = best;
                best = s;
                gbest = g;
            } else if (s > second) {
                second = s;
            }
        }
        out_group[b] = gbest;
        out_idx[b] = gbest >= 0 ? group_idx[gbest * B + b] : -1;
        out_best[b] = best;
        out_second[b] = second;
    }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

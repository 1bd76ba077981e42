// fs_stage1.cu -- Stage 1 of FlashSampling on sm_103a: the LM-head GEMM
// fused with temperature, Gumbel noise and a per-row tile argmax.
//
// "FlashSampling: Fast and Memory-Efficient Exact Sampling", method section:
// Stage 1 computes one batch tile and one vocabulary tile on chip, applies the
// deterministic transforms, adds Gumbel noise and keeps the tile-local
// maximizer for each row; each threadblock handles a contiguous vocabulary
// chunk.  Only (score, index) candidates leave the chip, never the [B, V]
// logits.
//
// GB300 design (one persistent CTA per SM, 512 threads = 16 warps):
//   warp 12     TMA producer: streams H [rows x 64] and W [<=256 x 64] k-blocks
//               (128-byte swizzled) into a ring of 4-6 shared-memory stages; a whole
//               W tile is one 256-row box (its 128-row half per CTA when
//               paired: multicast to both CTAs, or kept for a shared MMA),
//               tails are 64- and 16-row boxes.
//   warp 13     allocates 512 TMEM columns; one thread issues
//               tcgen05.mma (M=128, N<=256, K=16, bf16 -> f32; at large D
//               paired CTAs run one M=256 MMA over both, issued by the even
//               CTA) into one of two 256-column accumulators and commits to
//               mbarriers.
//   The producer and the MMA issuer share SM sub-partitions 0 and 1 with
//   busy epilogue warps, so they issue as few instructions per k-block as
//   possible (whole-tile boxes, precomputed descriptors).
//   warps 0-11, 14, 15  epilogue: tcgen05.ld of the accumulator (warp w reads
//               TMEM lane quarter w % 4: three warps for quarters 0 and 1, which
//               share their SM sub-partitions with the producer and the MMA
//               issuer, four for quarters 2 and 3; each takes its share of the
//               tile's columns), then
//               per element s = l * (1/T) + g with g from Philox4x64-10, and a
//               running per-row argmax across all tiles of the CTA.  The
//               epilogue of tile t overlaps the MMA of tile t+1 (double-buffered
//               TMEM).  At the end the column parts of each row are
//               merged through shared memory.  In the pair MMA, warps 14
//               and 15 instead sample the last column part of lane quarters
//               0 and 1, from raw logits that warps 0 and 1 pass through a
//               shared-memory ring, so that the sub-partitions of the TMA
//               producer and the MMA issuer carry less of the epilogue.
// Batch rows sit on the MMA M dimension, so each epilogue thread owns one row
// and scans its columns in increasing order: the lowest-index tie rule and
// the 8-wide Philox block both fall out without cross-lane exchange.
// CTA c works on batch tile c % nM and vocabulary partition c / nM
// (partitions are balanced in 16-row units), and writes one candidate per
// (row, partition).  Without clusters a partition is cut into balanced tiles
// of at most 256 rows plus a final 128-row tile, so that the one epilogue
// that cannot overlap an MMA (the last) is short; paired CTAs use plain
// 256-row tiles.  Each CTA (each cluster, when paired) starts its K loop at a
// different k-block, so the CTAs do not all request the same H line from L2
// at once.
// The epilogue screens every element with a cheap conservative bound
// (screen_lg2_tail / screen_bound): only elements that may beat the running
// best pay for the exact Gumbel, and the result equals the unscreened scan.
//
// Every wait is bounded: on expiry the CTA raises the device error word,
// tells its other warps to stop, drains its own TMA loads and MMAs, frees TMEM
// and returns.
#include <cuda_bf16.h>
#include <math.h>

#include <atomic>
#include <map>
#include <mutex>

#include "fs_internal.h"
#include "fs_noise.cuh"
#include "fs_ptx.cuh"

namespace fs {

__device__ uint32_t g_status_word = 0;


namespace {

constexpr uint32_t kStatusTimeout = 1u;

// Stage 1 launch forms (see stage1_kernel)
constexpr int kFormSingle = 0;
constexpr int kFormMulticast = 1;
constexpr int kFormPairMma = 2;
// Column hand-off ring (see the epilogue): per lane quarter 0 and 1,
// kExpSlots chunks of 16 columns x 32 rows of raw f32 logits, stored
// element-major (element i of lane l at i * 32 + l: conflict-free), after a
// 128-byte block of its full / empty barriers.
constexpr int kExpSlots = 4;
constexpr int kExpChunkFloats = 16 * 32;
constexpr int kExportBytes = 128 + 2 * kExpSlots * kExpChunkFloats * 4;
static_assert(4 * kExpSlots * 8 <= 128, "hand-off barriers");
// room behind the pair MMA's operand ring (6 stages of 32 KB)
static_assert(kRingBytes - 6 * (kABytes + kBBytes / 2) >= kExportBytes, "hand-off ring");
// the pair MMA serves paired calls with D at least this: with two batch
// tiles, or with more
constexpr int kPairMmaMinD2 = 4096;
constexpr int kPairMmaMinD = 6144;

__device__ __forceinline__ int round_up16(int x) { return (x + 15) & ~15; }

// Rows [r0, r1) of a partition of nu 16-row units.  A partition of at most
// 256 rows is one tile.  A larger one ends with a 128-row tile -- its
// epilogue is the one that cannot overlap an MMA, so it should be short --
// and splits the rest evenly into tiles of at most 256 rows, so that every
// pipeline stage still carries enough W bytes to keep HBM busy.  CTAs that
// share W tiles in a cluster (full_tiles) use plain 256-row tiles with the
// remainder last instead: each of them receives the whole tile, so they need
// the largest stages to keep enough bytes in flight.  Tile starts are
// multiples of 16 rows.
struct PartGeom {
    int r0, r1, nu, nmain, ntiles;
};

__device__ __forceinline__ PartGeom part_geom(int64_t u0, int64_t u1, int V, bool full_tiles) {
    constexpr int kTileUnits = kBN / kUnitRows;
    PartGeom g;
    g.r0 = static_cast<int>(u0 * kUnitRows);
    g.r1 = static_cast<int>(min(u1 * kUnitRows, static_cast<int64_t>(V)));
    g.nu = static_cast<int>(u1 - u0);
    if (full_tiles) {
        // 256-row tiles, the remainder last
        g.nmain = -1;
        g.ntiles = (g.r1 - g.r0 + kBN - 1) / kBN;
        return g;
    }
    if (g.nu <= kTileUnits) {
        g.nmain = 0;
        g.ntiles = (g.r1 > g.r0) ? 1 : 0;
    } else {
        g.nmain = (g.nu - kFinalTileUnits + kTileUnits - 1) / kTileUnits;
        g.ntiles = g.nmain + 1;
    }
    return g;
}

__device__ __forceinline__ void tile_geom(const PartGeom &g, int t, int &v0, int &tn) {
    if (g.nmain < 0) {
        v0 = g.r0 + kBN * t;
        tn = min(kBN, g.r1 - v0);
        return;
    }
    if (g.nmain == 0) {
        v0 = g.r0;
        tn = g.r1 - g.r0;
        return;
    }
    // Balanced split: the first `extra` main tiles take base + 1 units.  Tile
    // t starts at unit t * base + min(t, extra); no product exceeds the
    // partition's own unit count, so no overflow for any V < 2^31.
    const int main_units = g.nu - kFinalTileUnits;
    if (t < g.nmain) {
        const int base = main_units / g.nmain;
        const int extra = main_units - base * g.nmain;
        v0 = g.r0 + kUnitRows * (t * base + min(t, extra));
        tn = kUnitRows * (base + (t < extra ? 1 : 0));
    } else {
        v0 = g.r0 + kUnitRows * main_units;
        tn = g.r1 - v0;
    }
}

// First column of column part j (of np) of a tile of width tn: parts start
// on 16-column boundaries; part np ends at tn.
__device__ __forceinline__ int col_part_start(int j, int tn, int np) {
    if (j >= np) return tn;
    return min(tn, round_up16((j * tn + np - 1) / np));
}
// epilogue warps (column parts) of TMEM lane quarter q
__device__ __forceinline__ int quarter_parts(int q) { return q < 2 ? 3 : 4; }

// Element i (0..15) of a register array, by a chain of selects (an indexed
// load would move the array to local memory).
__device__ __forceinline__ float pick16(const float (&a)[16], int i) {
    float r = a[0];
#pragma unroll
    for (int k = 1; k < 16; ++k) r = (i == k) ? a[k] : r;
    return r;
}

__device__ __forceinline__ uint32_t pick16x(const uint32_t (&a)[8], const uint32_t (&b)[8], int i) {
    uint32_t r = a[0];
#pragma unroll
    for (int k = 1; k < 16; ++k) r = (i == k) ? (k < 8 ? a[k] : b[k - 8]) : r;
    return r;
}

// exp(x) from the hardware exp2 (relative error about 2^-22): the log-mass
// is a sum of positive terms, so this error does not accumulate.
__device__ __forceinline__ float exp2_approx_scaled(float x) {
    return ex2_approx(x * 1.4426950408889634f);
}

// Online log-sum-exp: add a finite element x to (m, s) = (max, sum exp(. - max)).
__device__ __forceinline__ void lse_add(float &m, float &s, float x) {
    if (x > m) {
        s = s * exp2_approx_scaled(m - x) + 1.0f;
        m = x;
    } else {
        s += exp2_approx_scaled(x - m);
    }
}

// Merge (m2, s2) into (m, s); an empty pair has m = -inf and s = 0.
__device__ __forceinline__ void lse_merge(float &m, float &s, float m2, float s2) {
    if (m2 > m) {
        s = s * exp2_approx_scaled(m - m2) + s2;
        m = m2;
    } else if (s2 > 0.0f) {
        s += s2 * exp2_approx_scaled(m2 - m);
    }
}

// The deterministic transforms of a 16-column chunk of row b, in place on
// the raw f32 accumulator bits: l += bias[v]; l = c * tanh(l / c) if c > 0;
// l = -inf where the row's allowed-token mask has a 0 bit.
__device__ __forceinline__ void apply_transforms(const Stage1Args &a, int b, int vbase,
                                                 int n_valid, uint32_t (&r)[16]) {
    float l[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) l[i] = __uint_as_float(r[i]);
    if (a.bias != nullptr) {
        if (n_valid == 16) {
            const float4 *bp = reinterpret_cast<const float4 *>(a.bias + vbase);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 bb = __ldg(bp + q);
                l[4 * q] = __fadd_rn(l[4 * q], bb.x);
                l[4 * q + 1] = __fadd_rn(l[4 * q + 1], bb.y);
                l[4 * q + 2] = __fadd_rn(l[4 * q + 2], bb.z);
                l[4 * q + 3] = __fadd_rn(l[4 * q + 3], bb.w);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (i < n_valid) l[i] = __fadd_rn(l[i], __ldg(a.bias + vbase + i));
        }
    }
    if (a.softcap > 0.0f) {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            l[i] = __fmul_rn(a.softcap, tanhf(__fdiv_rn(l[i], a.softcap)));
    }
    if (a.allow_mask != nullptr) {
        // vbase is a multiple of 16: the chunk's 16 bits sit in one word
        const uint32_t word = __ldg(a.allow_mask + static_cast<int64_t>(b) * a.mask_words +
                                    (vbase >> 5));
        const uint32_t bits = word >> (vbase & 31);
#pragma unroll
        for (int i = 0; i < 16; ++i)
            if (!((bits >> i) & 1u)) l[i] = -INFINITY;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(l[i]);
}

__device__ __forceinline__ void epilogue_barrier() {
    asm volatile("bar.sync 1, %0;" ::"n"(kNumEpiWarps * 32) : "memory");
}

__device__ __forceinline__ void raise_timeout(volatile int *abort_flag) {
    atomicOr(&g_status_word, kStatusTimeout);
    *abort_flag = 1;
}

// Stores n (<= 16) consecutive f32 values of one row.
__device__ __forceinline__ void store_f32_chunk(float *dst, int n, const uint32_t (&r)[16],
                                                bool vec_ok) {
    if (vec_ok && n == 16) {
        float4 *d4 = reinterpret_cast<float4 *>(dst);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            d4[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            if (i < n) dst[i] = __uint_as_float(r[i]);
    }
}

// Stores n (<= 16) consecutive values of one row rounded to bf16.
__device__ __forceinline__ void store_bf16_chunk(__nv_bfloat16 *dst, int n,
                                                 const uint32_t (&r)[16], bool vec_ok) {
    if (vec_ok && n == 16) {
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            uint32_t p[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                __nv_bfloat162 two = __floats2bfloat162_rn(__uint_as_float(r[8 * i + 2 * j]),
                                                           __uint_as_float(r[8 * i + 2 * j + 1]));
                p[j] = *reinterpret_cast<uint32_t *>(&two);
            }
            d4[i] = make_uint4(p[0], p[1], p[2], p[3]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            if (i < n) dst[i] = __float2bfloat16_rn(__uint_as_float(r[i]));
    }
}

// Running state of one sampled row in one epilogue thread: the best perturbed
// score and its index, and (log-probability modes) the log-mass of the
// elements seen, lse_m = max l~, lse_s = sum exp(l~ - lse_m), with best_lt =
// l~ of the best.
struct SampleRow {
    float best, lse_m, lse_s, best_lt, invT;
    int bidx, b;
    bool row_ok, t_ok;
    PhiloxRow prow;
};

__device__ __forceinline__ SampleRow sample_row(const Stage1Args &a, bool sampling, int b,
                                                bool row_ok) {
    SampleRow s;
    s.best = -INFINITY;
    s.bidx = -1;
    s.lse_m = -INFINITY;
    s.lse_s = 0.0f;
    s.best_lt = NAN;
    s.invT = 0.0f;
    s.t_ok = false;
    s.b = b;
    s.row_ok = row_ok;
    if (sampling && row_ok) {
        const float T = a.temps ? a.temps[b] : a.temp_scalar;
        s.t_ok = isfinite(T) && T > 0.0f;
        s.invT = __frcp_rn(T);
    }
    s.prow = philox_row(a.seed, a.offset, static_cast<uint64_t>(b));
    return s;
}

// One 16-column chunk of one row (raw f32 accumulator bits r, columns vbase ..
// vbase + n_valid - 1 of the partition's vocabulary): optional logits store and
// transforms, s = l * (1/T) + g with g from the Philox words (drawn here unless
// have_words), and the running best.  first_chunk is a warp-wide vote taken
// by the caller: every lane's best is still -inf.
template <int MODE>
__device__ __forceinline__ void sample_chunk(const Stage1Args &a, SampleRow &st,
                                             uint32_t (&r)[16], int vbase, int n_valid,
                                             bool first_chunk, bool have_words,
                                             uint32_t (&xa)[8], uint32_t (&xb)[8]) {
    constexpr bool kLogprob = (MODE == kModeSampleLogprob || MODE == kModeSampleXformLogprob);
    constexpr bool kXform = (MODE == kModeSampleXform || MODE == kModeSampleXformLogprob);
    if (MODE == kModeSampleStore && st.row_ok)
        store_f32_chunk(a.out_logits + static_cast<size_t>(st.b) * a.V + vbase, n_valid, r,
                        a.y_vec_ok != 0);
    if (kXform && st.row_ok && st.t_ok) apply_transforms(a, st.b, vbase, n_valid, r);
    if (!(st.row_ok && st.t_ok)) return;
    if (a.flags & 1u) {  // noise off
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float s = __fmul_rn(__uint_as_float(r[i]), st.invT);
            if (i < n_valid && s > st.best) {
                st.best = s;
                st.bidx = static_cast<int>(a.vocab_offset) + vbase + i;
                st.best_lt = s;
            }
            if (kLogprob && i < n_valid && isfinite(s)) lse_add(st.lse_m, st.lse_s, s);
        }
        return;
    }
    // Both Philox blocks of the chunk first (two independent chains for the
    // scheduler).
    if (!have_words) {
        const uint64_t v8 = static_cast<uint64_t>(a.vocab_offset + vbase) >> 3;
        noise_words8(st.prow, v8, xa);
        if (n_valid > 8) noise_words8(st.prow, v8 + 1, xb);
    }
    float lt[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) lt[i] = __fmul_rn(__uint_as_float(r[i]), st.invT);
    if (kLogprob) {
        // online log-sum-exp over the finite l~, rescaled once per chunk
        float cm = -INFINITY;
#pragma unroll
        for (int i = 0; i < 16; ++i)
            if (i < n_valid && isfinite(lt[i])) cm = fmaxf(cm, lt[i]);
        if (cm > st.lse_m) {
            st.lse_s *= exp2_approx_scaled(st.lse_m - cm);
            st.lse_m = cm;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i)
            if (i < n_valid && isfinite(lt[i])) st.lse_s += exp2_approx_scaled(lt[i] - st.lse_m);
    }
    if (first_chunk) {
        // every lane's best is still -inf: all 16 elements would survive the
        // screen, so score them directly
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t xi = i < 8 ? xa[i] : xb[i - 8];
            const float s = __fadd_rn(lt[i], gumbel_from_word(xi));
            if (i < n_valid && s > st.best) {
                st.best = s;
                st.bidx = static_cast<int>(a.vocab_offset) + vbase + i;
                if (kLogprob) st.best_lt = lt[i];
            }
        }
        return;
    }
    // A conservative screen per element against the best known before the
    // chunk (a lower bound of the running best); survivors are scored
    // exactly, lowest index first (keeps the tie rule).  A loop over the set
    // bits costs one iteration per survivor instead of a predicated
    // evaluation of every element.
    const float best0 = st.best;
    uint32_t pass = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t xi = i < 8 ? xa[i] : xb[i - 8];
        if (i < n_valid && screen_lg2_tail(xi) < screen_bound(lt[i], best0)) pass |= 1u << i;
    }
    while (pass) {
        const int i = __ffs(pass) - 1;
        pass &= pass - 1;
        const float s = __fadd_rn(pick16(lt, i), gumbel_from_word(pick16x(xa, xb, i)));
        if (s > st.best) {
            st.best = s;
            st.bidx = static_cast<int>(a.vocab_offset) + vbase + i;
            if (kLogprob) st.best_lt = pick16(lt, i);
        }
    }
}

}  // namespace

// FORM selects the launch form.
//   kFormSingle     one CTA per (batch tile, partition).
//   kFormMulticast  CTA pairs (2-CTA clusters) over two consecutive batch
//      tiles of the same vocabulary partition, each with its own M=128 MMA:
//      each CTA loads half of every W k-block and multicasts it to both, so
//      W crosses L2 -> SM once per pair.  A stage is refilled only after both
//      CTAs' MMAs have released it (each CTA's commit arrives on both CTAs'
//      empty barriers).
//   kFormPairMma    CTA pairs sharing one 256 x N MMA (.cta_group::2): each
//      CTA loads its own 128 H rows and half of the tile's W rows, so a stage
//      is 16 KB of H plus 16 KB of W per SM (6 stages fit instead of the 4 of
//      48 KB stages).  Both CTAs' loads of a stage complete on the leader's
//      (the even CTA's) full barrier, whose expected byte count covers both
//      halves, so the leader issues the MMAs of a stage once the whole pair's
//      data has landed, with no per-stage message between the CTAs.  Its
//      commits arrive on both CTAs' empty and full barriers.  Each CTA's
//      epilogue reads its own 128 accumulator lanes; the leader reuses an
//      accumulator once both CTAs' epilogue warps have released it (the
//      peer's warps arrive remotely on the leader's tempty_peer, once per
//      tile).
//   Both pair forms move the same bytes from L2; which is faster depends on
//   D and on the number of batch tiles (see launch_stage1).
template <int MODE, int FORM>
__global__ void __launch_bounds__(kThreads, 1)
    stage1_kernel(const __grid_constant__ CUtensorMap tmH, const __grid_constant__ CUtensorMap tmW16,
                  const __grid_constant__ CUtensorMap tmW64,
                  const __grid_constant__ CUtensorMap tmWhalf,
                  const __grid_constant__ CUtensorMap tmWfull, const Stage1Args a) {
    constexpr bool kSample = (MODE == kModeSample || MODE == kModeSampleStore ||
                              MODE == kModeSampleLogprob || MODE == kModeSampleXform ||
                              MODE == kModeSampleXformLogprob);
    constexpr bool kLogprob = (MODE == kModeSampleLogprob || MODE == kModeSampleXformLogprob);
    constexpr int CS = FORM == kFormSingle ? 1 : 2;  // CTAs per cluster
    constexpr bool kTwoSm = FORM == kFormPairMma;
    constexpr bool kMcast = FORM == kFormMulticast;
    constexpr uint16_t kClusterMask = static_cast<uint16_t>((1u << CS) - 1u);
    // bytes of one stage's W slot: half of a 256-row tile per CTA for the pair MMA
    constexpr int kWSlot = kTwoSm ? kBBytes / 2 : kBBytes;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
    // Shared memory: barriers and the combine area, then the ring: nst H
    // slots of a_stride bytes, then nst W slots.  A single batch tile loads
    // only round_up(B, 8) rows of H per stage, so its H slot shrinks to that
    // (in 1 KB swizzle atoms) and the ring holds more stages of W: 6 at
    // B <= 16, 5 at B <= 88, else 4.
    // A single batch tile of at most 64 (96) rows also sits in accumulator
    // lanes 64.. (32..): the MMA's A descriptor starts lane_off rows (128 B
    // each) before the H slot.  TMEM lane quarter q is read by the warps of SM
    // sub-partition q, so the epilogue of a small batch then runs on
    // sub-partitions 2-3, away from the TMA producer (0) and the MMA issuer
    // (1).  The A rows the MMA reads around the batch come from neighbouring
    // slots or from the area in front of the ring, always inside shared
    // memory, and feed lanes that no epilogue warp reads.
    const int a_stride = (a.nM == 1) ? (a.h_box_rows * (kBK * 2) + 1023) & ~1023 : kABytes;
    const int nst = min(kMaxStages, kRingBytes / (a_stride + kWSlot));
    const int lane_off = (a.nM != 1) ? 0 : (a.B <= 64 ? 64 : (a.B <= 96 ? 32 : 0));
    uint8_t *sA = smem + kPreRingBytes;
    uint8_t *sB = sA + nst * a_stride;
    // Column hand-off (sampling modes of the pair MMA): behind the operand
    // ring.  Measured: 1-2% faster for the pair MMA at D = 3584-8192; the
    // multicast pair at D = 2304 was 4% slower with it (there the epilogue
    // fills most of each tile's MMA time on every sub-partition), so it
    // runs without.
    uint8_t *sX = sB + nst * kWSlot;
    const bool exp_on = kSample && kTwoSm &&
                        kRingBytes - nst * (a_stride + kWSlot) >= kExportBytes;
    uint64_t *exp_full = reinterpret_cast<uint64_t *>(sX);  // [2][kExpSlots]
    uint64_t *exp_empty = exp_full + 2 * kExpSlots;         // [2][kExpSlots]
    float *exp_ring = reinterpret_cast<float *>(sX + 128);   // [2][kExpSlots][16][32]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    uint64_t *full_bar = bars;
    uint64_t *empty_bar = bars + kMaxStages;
    uint64_t *tfull_bar = bars + 2 * kMaxStages;
    uint64_t *tempty_bar = tfull_bar + 2;
    uint64_t *done_bar = tempty_bar + 2;
    uint64_t *tempty_peer = done_bar + 1;  // leader, pair MMA: the peer's epilogue is done
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty_peer + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *comb_s = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(bars) + 256);
    int *comb_i = reinterpret_cast<int *>(comb_s + kColParts * kBM);
    float *comb_lt = reinterpret_cast<float *>(comb_i + kColParts * kBM);
    float *comb_m = comb_lt + kColParts * kBM;
    float *comb_sum = comb_m + kColParts * kBM;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int m = blockIdx.x % a.nM;
    const int part = blockIdx.x / a.nM;
    const PartGeom geom = part_geom(static_cast<int64_t>(part) * a.U / a.P,
                                    static_cast<int64_t>(part + 1) * a.U / a.P, a.V, CS > 1);
    const uint32_t crank = (CS > 1) ? cluster_ctarank() : 0u;
    const int ntiles = geom.ntiles;
    const int nk = (a.D + kBK - 1) / kBK;
    // The CTAs of a cluster exchange W k-blocks, so they must walk the same
    // k sequence: rotate by cluster, not by CTA.
    const int kb_first = static_cast<int>((blockIdx.x / CS) % static_cast<unsigned>(nk));

    if (threadIdx.x == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(&full_bar[s], 1);
            // one commit per stage (the pair leader's for the pair MMA), two
            // for the multicast pair (both CTAs' MMAs read the stage's W)
            mbar_init(&empty_bar[s], kMcast ? CS : 1);
        }
        // Only epilogue warps whose TMEM lane quarter holds live batch rows
        // take part in the tile loop and release the accumulators (with the
        // column hand-off, three per quarter: warps 14 and 15 read no tensor
        // memory).
        auto live_warps = [&](int mt) {
            int n = 0;
            for (int qq = 0; qq < 4; ++qq)
                if (qq * 32 >= lane_off && (mt * kBM + qq * 32 - lane_off) < a.B)
                    n += exp_on ? 3 : quarter_parts(qq);
            return n;
        };
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull_bar[i], 1);
            mbar_init(&tempty_bar[i], live_warps(m));
            // the peer's batch tile is m + 1 (it holds at least one row: the
            // pair form runs only with an even number of batch tiles)
            mbar_init(&tempty_peer[i], kTwoSm ? max(1, live_warps(m + 1)) : 1);
        }
        mbar_init(done_bar, 1);
        if (exp_on)
            for (int i = 0; i < 2 * kExpSlots; ++i) {
                mbar_init(&exp_full[i], 32);   // every lane of the passing warp
                mbar_init(&exp_empty[i], 32);  // every lane of the receiving warp
            }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kWarpMma) {
        if constexpr (kTwoSm) {
            tmem_alloc_pair(tmem_slot, kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_slot, kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    // Paired CTAs: both CTAs' barriers (and tensor memory) must be set up
    // before either one's loads complete on, or its arrivals reach, the other.
    if (CS > 1) cluster_sync();
    const uint32_t tmem_base = *tmem_slot;

    // Programmatic dependent launch: everything above overlaps the previous
    // kernel of the stream.  Before waiting for it, the producer also warms L2
    // with the first W k-blocks of this CTA's first tile.  That is safe even if
    // the previous kernel writes W, because L2 is where writes become visible
    // and shared memory is filled only after the wait.  Every other global
    // access (H, the temperatures, the workspace) comes after the wait.
    if (warp == kWarpTma && lane == 0) {
        prefetch_tmap(&tmH);
        prefetch_tmap(&tmW64);
        prefetch_tmap(&tmW16);
        prefetch_tmap(CS > 1 ? &tmWhalf : &tmWfull);
        if (ntiles > 0 && !(a.flags & 0x100u)) {
            int v0, tn;
            tile_geom(geom, 0, v0, tn);
            const int nbox = (round_up16(tn) + 63) >> 6;  // 64-row boxes covering the tile
            const int nwarm = min(nk, nst + 2);
            int kb = kb_first;
            for (int jj = 0; jj < nwarm; ++jj) {
                for (int i = static_cast<int>(crank); i < nbox; i += CS)
                    tma_prefetch_l2_2d(&tmW64, kb * kBK, v0 + i * 64);
                if (++kb == nk) kb = 0;
            }
        }
    }
    griddep_wait();

    if (warp == kWarpTma) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_w = l2_policy_evict_first();
            const uint64_t pol_h = l2_policy_evict_last();
            const uint32_t h_bytes = static_cast<uint32_t>(a.h_box_rows) * (kBK * 2);
            int stage = 0;
            uint32_t phase = 0;
            int n_issued = 0;  // k-blocks whose loads were issued (for the drain)
            bool ok = true;
            // test hook (flag 0x100): issue nothing, so the consumers' first
            // bounded waits expire and the timeout path runs
            const int ntiles_loaded = (a.flags & 0x100u) ? 0 : ntiles;
            for (int t = 0; t < ntiles_loaded && ok; ++t) {
                int v0, tn;
                tile_geom(geom, t, v0, tn);
                const int tn16 = round_up16(tn);
                // W rows this CTA loads per stage: the whole tile, or for the
                // pair MMA its half of the tile rounded up to 32 rows (rows past
                // the tile feed accumulator columns that no epilogue reads)
                const int nw = kTwoSm ? ((tn + 31) & ~31) : tn16;
                const int wrows = kTwoSm ? nw / 2 : tn16;
                const int wrow0 = kTwoSm ? v0 + static_cast<int>(crank) * (nw / 2) : v0;
                const int n64 = wrows >> 6;
                const int n16 = (wrows & 63) >> 4;
                const uint32_t bytes = h_bytes + wrows * (kBK * 2);
                int kb = kb_first;
                for (int j = 0; j < nk; ++j) {
                    if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1u, a.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    uint8_t *dA = sA + stage * a_stride;
                    uint8_t *dB = sB + stage * kWSlot;
                    const int kx = kb * kBK;
                    if (kTwoSm) {
                        // both CTAs' bytes of the stage complete on the leader's
                        // full barrier; the leader expects them all (the peer's
                        // loads may land before that, which only takes the byte
                        // count below zero until the leader's arrival)
                        const uint32_t bar =
                            mapa_shared(smem_u32(&full_bar[stage]), 0u);
                        if (crank == 0) mbar_arrive_expect_tx(&full_bar[stage], 2 * bytes);
                        tma_load_2d_pair(dA, &tmH, bar, kx, m * kBM, pol_h);
                        if (wrows == kBN / 2) {
                            tma_load_2d_pair(dB, &tmWhalf, bar, kx, wrow0, pol_w);
                        } else {
                            for (int i = 0; i < n64; ++i)
                                tma_load_2d_pair(dB + i * 64 * (kBK * 2), &tmW64, bar, kx,
                                                 wrow0 + i * 64, pol_w);
                            for (int i = 0; i < n16; ++i)
                                tma_load_2d_pair(dB + (n64 * 64 + i * 16) * (kBK * 2), &tmW16, bar,
                                                 kx, wrow0 + n64 * 64 + i * 16, pol_w);
                        }
                        ++n_issued;
                        if (++stage == nst) {
                            stage = 0;
                            phase ^= 1u;
                        }
                        if (++kb == nk) kb = 0;
                        continue;
                    }
                    mbar_arrive_expect_tx(&full_bar[stage], bytes);
                    tma_load_2d(dA, &tmH, &full_bar[stage], kx, m * kBM, pol_h);
                    if (kMcast) {
                        // the stage's W is the whole tile in both CTAs; each
                        // CTA loads half of its boxes (its 128-row half of a
                        // whole tile, else box i when i % 2 == its rank) and
                        // multicasts them to both
                        if (tn16 == kBN) {
                            tma_load_2d_multicast(dB + crank * (kBN / 2) * (kBK * 2), &tmWhalf,
                                                  &full_bar[stage], kx,
                                                  v0 + static_cast<int>(crank) * (kBN / 2),
                                                  kClusterMask, pol_w);
                        } else {
                            for (int i = static_cast<int>(crank); i < n64 + n16; i += CS) {
                                const int r = i < n64 ? i * 64 : n64 * 64 + (i - n64) * 16;
                                tma_load_2d_multicast(dB + r * (kBK * 2), i < n64 ? &tmW64 : &tmW16,
                                                      &full_bar[stage], kx, v0 + r, kClusterMask,
                                                      pol_w);
                            }
                        }
                    } else if (tn16 == kBN) {
                        // a whole tile: one box (same shared-memory layout as the
                        // 64-row boxes)
                        tma_load_2d(dB, &tmWfull, &full_bar[stage], kx, v0, pol_w);
                    } else {
                        for (int i = 0; i < n64; ++i)
                            tma_load_2d(dB + i * 64 * (kBK * 2), &tmW64, &full_bar[stage], kx,
                                        v0 + i * 64, pol_w);
                        for (int i = 0; i < n16; ++i)
                            tma_load_2d(dB + (n64 * 64 + i * 16) * (kBK * 2), &tmW16,
                                        &full_bar[stage], kx, v0 + n64 * 64 + i * 16, pol_w);
                    }
                    ++n_issued;
                    if (++stage == nst) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    if (++kb == nk) kb = 0;
                }
            }
            if (!ok) raise_timeout(abort_flag);
            // Drain: every issued load must land before the CTA's shared
            // memory is released (immediate on the normal path).
            // The last load into stage s is load number s + nst * ((n_issued - 1 - s) / nst);
            // its full barrier completes with parity (that number / nst) & 1.
            // A pair-MMA peer's loads complete on the leader's barriers, which
            // the leader drains (both CTAs stay resident until the cluster
            // barrier at the end).  A multicast CTA's barriers complete only
            // once its peer's halves have landed too.
            for (int s = 0; s < nst && s < n_issued && !(kTwoSm && crank != 0); ++s) {
                const int last = s + nst * ((n_issued - 1 - s) / nst);
                mbar_wait_bounded(&full_bar[s], static_cast<uint32_t>(last / nst) & 1u,
                                  a.timeout_ns, nullptr);
            }
        }
    } else if (warp == kWarpMma && kTwoSm && crank != 0) {
        // pair MMA, peer CTA: the leader issues every MMA; nothing to do here
    } else if (warp == kWarpMma) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            // lane_off rows before the H slot: H row r feeds accumulator lane lane_off + r
            const uint64_t a_desc0 =
                sw128_kmajor_desc(smem_u32(sA) - static_cast<uint32_t>(lane_off * (kBK * 2)));
            const uint64_t b_desc0 = sw128_kmajor_desc(smem_u32(sB));
            for (int t = 0; t < ntiles && ok; ++t) {
                const int acc = t & 1;
                const uint32_t aphase = static_cast<uint32_t>(t >> 1) & 1u;
                if (!mbar_wait_bounded(&tempty_bar[acc], aphase ^ 1u, a.timeout_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                // pair MMA: the peer's epilogue must have released it too
                if (kTwoSm && !mbar_wait_bounded_cluster(&tempty_peer[acc], aphase ^ 1u,
                                                         a.timeout_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                int v0, tn;
                tile_geom(geom, t, v0, tn);
                const uint32_t idesc =
                    kTwoSm ? idesc_bf16_f32(2 * kBM, static_cast<uint32_t>((tn + 31) & ~31))
                           : idesc_bf16_f32(kBM, static_cast<uint32_t>(round_up16(tn)));
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
                for (int j = 0; j < nk; ++j) {
                    if (!mbar_wait_bounded(&full_bar[stage], phase, a.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    {
                        // descriptors differ from stage 0's by the stage offset and
                        // from each other by 32 bytes of K (both in 16-byte units)
                        const uint64_t ad = a_desc0 + static_cast<uint64_t>(stage * (a_stride >> 4));
                        const uint64_t bd = b_desc0 + static_cast<uint64_t>(stage * (kWSlot >> 4));
#pragma unroll
                        for (int ks = 0; ks < kBK / kUmmaK; ++ks) {
                            if constexpr (kTwoSm)
                                umma_bf16_ss_pair(d_tmem, ad + 2 * ks, bd + 2 * ks, idesc,
                                                  (j | ks) != 0 ? 1u : 0u);
                            else
                                umma_bf16_ss(d_tmem, ad + 2 * ks, bd + 2 * ks, idesc,
                                             (j | ks) != 0 ? 1u : 0u);
                        }
                    }
                    if constexpr (kTwoSm)
                        umma_commit_pair_multicast(&empty_bar[stage], kClusterMask);
                    else if constexpr (kMcast)
                        umma_commit_multicast(&empty_bar[stage], kClusterMask);
                    else
                        umma_commit(&empty_bar[stage]);
                    if (++stage == nst) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) {
                    if constexpr (kTwoSm)
                        umma_commit_pair_multicast(&tfull_bar[acc], kClusterMask);
                    else
                        umma_commit(&tfull_bar[acc]);
                }
            }
            if (!ok) raise_timeout(abort_flag);
            // Retire every MMA this thread issued before TMEM is freed.
            if constexpr (kTwoSm)
                umma_commit_pair_multicast(done_bar, 1u);
            else
                umma_commit(done_bar);
            mbar_wait_bounded(done_bar, 0, a.timeout_ns, nullptr);
        }
    } else {
        // ------------------------------------------------ epilogue warps
        const int q = warp & 3;   // TMEM lane quarter (the warp's rank in its warpgroup)
        // Roles.  Without the column hand-off, warp w reads lane quarter q =
        // w % 4 and takes column part w / 4 of quarter_parts(q) (warps 14 and
        // 15: part 3).  With it, warps 0-11 take parts 0-2: of four parts in
        // quarters 0 and 1 and of three in quarters 2 and 3.  Part 3 of
        // quarters 0 and 1 is sampled by warps 14 and 15 on sub-partitions 2
        // and 3, from the raw logits that warps 0 and 1 pass through the
        // hand-off ring, so that sub-partitions 0 and 1 (TMA producer, MMA
        // issuer) carry less of the epilogue.
        const bool importer = exp_on && warp >= 14;
        const int j = warp < 12 ? (warp >> 2) : 3;  // column part of the tile
        const int np = exp_on ? (q < 2 ? 4 : 3) : quarter_parts(q);
        const int rq = importer ? q - 2 : q;  // lane quarter of the rows this warp samples
        const int tl = rq * 32 + lane;        // accumulator row
        const int row = tl - lane_off;        // row within the batch tile
        const int b = m * kBM + row;
        const bool quarter_live = rq * 32 >= lane_off && (m * kBM + rq * 32 - lane_off) < a.B;
        const bool reads_tmem = !importer && quarter_live;
        const bool exporter = exp_on && !importer && q < 2 && j == 0 && quarter_live;
        SampleRow st = sample_row(a, kSample, b, row >= 0 && b < a.B);
        const bool no_noise = (a.flags & 1u) != 0;
        bool ok = true;
        int xcnt = 0;  // chunks passed through the hand-off ring so far
        // Warps without live rows skip the tile loop (they are not counted by
        // the accumulator-release barrier) and wait at the combine barrier.
        for (int t = 0; t < (reads_tmem ? ntiles : 0); ++t) {
            const int acc = t & 1;
            const uint32_t aphase = static_cast<uint32_t>(t >> 1) & 1u;
            // The last tile's epilogue is the one no MMA hides.  Its noise
            // depends only on (row, column), so it is computed while that
            // tile's MMA still runs and parked in the other accumulator:
            // tile t-1 has released it (all epilogue warps arrived on its
            // empty barrier) and no later MMA writes it again.
            const bool pre_noise = kSample && !no_noise && t >= 1 && t == ntiles - 1;  // warp-uniform
            if (pre_noise) {
                if (!mbar_wait_bounded_backoff(&tempty_bar[acc ^ 1],
                                               static_cast<uint32_t>((t - 1) >> 1) & 1u,
                                               a.timeout_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                int v0p, tnp;
                tile_geom(geom, t, v0p, tnp);
                const int lo = col_part_start(j, tnp, np);
                const int hi = col_part_start(j + 1, tnp, np);
                for (int c0 = lo; c0 < hi; c0 += 16) {
                    uint32_t wa[8], wb[8], w[16];
                    const uint64_t v8 = static_cast<uint64_t>(a.vocab_offset + v0p + c0) >> 3;
                    noise_words8(st.prow, v8, wa);
                    noise_words8(st.prow, v8 + 1, wb);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        w[i] = wa[i];
                        w[8 + i] = wb[i];
                    }
                    tmem_st16_wait(tmem_base + static_cast<uint32_t>((acc ^ 1) * kBN + c0) +
                                       (static_cast<uint32_t>(q * 32) << 16),
                                   w);
                }
            }
            if (!mbar_wait_bounded_backoff(&tfull_bar[acc], aphase, a.timeout_ns, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            int v0, tn;
            tile_geom(geom, t, v0, tn);
            if (exporter) {
                // part 3 of this quarter's rows, raw, into the hand-off ring
                uint64_t *xfull = exp_full + q * kExpSlots;
                uint64_t *xempty = exp_empty + q * kExpSlots;
                for (int c0 = col_part_start(3, tn, 4); c0 < tn; c0 += 16, ++xcnt) {
                    const int slot = xcnt % kExpSlots;
                    if (!mbar_wait_bounded_backoff(&xempty[slot],
                                                   (static_cast<uint32_t>(xcnt / kExpSlots) & 1u) ^ 1u,
                                                   a.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    __syncwarp();
                    uint32_t r[16];
                    tmem_ld16_wait(tmem_base + static_cast<uint32_t>(acc * kBN + c0) +
                                       (static_cast<uint32_t>(q * 32) << 16),
                                   r);
                    float *dst = exp_ring + (q * kExpSlots + slot) * kExpChunkFloats;
#pragma unroll
                    for (int i = 0; i < 16; ++i) dst[i * 32 + lane] = __uint_as_float(r[i]);
                    mbar_arrive(&xfull[slot]);  // each lane: its own stores are released
                }
                if (!ok) break;
            }
            const int c_lo = col_part_start(j, tn, np);
            const int c_hi = col_part_start(j + 1, tn, np);
            for (int c0 = c_lo; c0 < c_hi; c0 += 16) {
                uint32_t r[16];
                tmem_ld16_wait(tmem_base + static_cast<uint32_t>(acc * kBN + c0) +
                                   (static_cast<uint32_t>(q * 32) << 16),
                               r);
                // the parked noise of the last tile, read by the whole (converged) warp
                uint32_t xa[8], xb[8];
                if (pre_noise) {
                    uint32_t w[16];
                    tmem_ld16_wait(tmem_base + static_cast<uint32_t>((acc ^ 1) * kBN + c0) +
                                       (static_cast<uint32_t>(q * 32) << 16),
                                   w);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        xa[i] = w[i];
                        xb[i] = w[8 + i];
                    }
                }
                const int n_valid = min(16, c_hi - c0);
                const int vbase = v0 + c0;
                if (kSample) {
                    // warp-wide vote while the warp is converged; lanes without
                    // a live row keep best = -inf and never block it
                    const bool first_chunk = __all_sync(0xffffffffu, st.best == -INFINITY);
                    sample_chunk<MODE>(a, st, r, vbase, n_valid, first_chunk, pre_noise, xa, xb);
                } else if (st.row_ok) {
                    if (MODE == kModeGemmF32)
                        store_f32_chunk(static_cast<float *>(a.out_y) +
                                            static_cast<size_t>(b) * a.V + vbase,
                                        n_valid, r, a.y_vec_ok != 0);
                    else
                        store_bf16_chunk(static_cast<__nv_bfloat16 *>(a.out_y) +
                                             static_cast<size_t>(b) * a.V + vbase,
                                         n_valid, r, a.y_vec_ok != 0);
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&tempty_bar[acc]);
                // pair MMA: the leader reuses the accumulator only once the
                // peer's warps have released it as well
                if (kTwoSm && crank != 0)
                    mbar_arrive_cluster(mapa_shared(smem_u32(&tempty_peer[acc]), 0u));
            }
        }
        // Warps 14 and 15 with the hand-off: part 3 of quarter 0 or 1, chunk
        // by chunk as the ring fills.  They never touch tensor memory, so the
        // accumulators are released without them.
        if (kSample && importer && quarter_live) {
            uint64_t *xfull = exp_full + rq * kExpSlots;
            uint64_t *xempty = exp_empty + rq * kExpSlots;
            for (int t = 0; t < ntiles && ok; ++t) {
                int v0, tn;
                tile_geom(geom, t, v0, tn);
                for (int c0 = col_part_start(3, tn, 4); c0 < tn; c0 += 16, ++xcnt) {
                    const int slot = xcnt % kExpSlots;
                    if (!mbar_wait_bounded_backoff(&xfull[slot],
                                                   static_cast<uint32_t>(xcnt / kExpSlots) & 1u,
                                                   a.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    __syncwarp();
                    uint32_t r[16];
                    const float *src = exp_ring + (rq * kExpSlots + slot) * kExpChunkFloats;
#pragma unroll
                    for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(src[i * 32 + lane]);
                    mbar_arrive(&xempty[slot]);  // each lane, after its loads
                    const bool first_chunk = __all_sync(0xffffffffu, st.best == -INFINITY);
                    uint32_t xa[8], xb[8];
                    sample_chunk<MODE>(a, st, r, v0 + c0, min(16, tn - c0), first_chunk, false,
                                       xa, xb);
                }
            }
        }
        if (!ok) raise_timeout(abort_flag);
        if (kSample) {
            // Combine the column parts' bests of each row (tie: lower index),
            // then one candidate per (row, partition).
            comb_s[j * kBM + tl] = st.best;
            comb_i[j * kBM + tl] = st.bidx;
            if (kLogprob) {
                comb_lt[j * kBM + tl] = st.best_lt;
                comb_m[j * kBM + tl] = st.lse_m;
                comb_sum[j * kBM + tl] = st.lse_s;
            }
            epilogue_barrier();
            if (j == 0 && st.row_ok) {
                float best = st.best, best_lt = st.best_lt, lse_m = st.lse_m, lse_s = st.lse_s;
                int bidx = st.bidx;
#pragma unroll
                for (int jj = 1; jj < np; ++jj) {
                    const float s = comb_s[jj * kBM + tl];
                    const int i = comb_i[jj * kBM + tl];
                    if (s > best ||
                        (s == best && static_cast<uint32_t>(i) < static_cast<uint32_t>(bidx))) {
                        best = s;
                        bidx = i;
                        if (kLogprob) best_lt = comb_lt[jj * kBM + tl];
                    }
                    if (kLogprob)
                        lse_merge(lse_m, lse_s, comb_m[jj * kBM + tl], comb_sum[jj * kBM + tl]);
                }
                const size_t o = static_cast<size_t>(part) * a.B + b;
                a.cand_score[o] = best;
                a.cand_idx[o] = bidx;
                if (kLogprob) {
                    a.cand_lt[o] = best_lt;
                    a.cand_m[o] = lse_m;
                    a.cand_s[o] = lse_s;
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    // This CTA's candidates are written: Stage 2 (launched with programmatic
    // serialization) may now be scheduled; it still waits for the whole grid
    // before reading.  Triggering only here keeps its blocks off the SMs while
    // the epilogues run.
    griddep_launch_dependents();
    // Paired CTAs after a timeout anywhere (the device error word is set):
    // a pair-MMA peer's loads complete only on the leader's barriers, and the
    // leader drains no further than the phases it armed; a multicast CTA's
    // drain cannot account for loads its peer issued after it stopped.  So
    // such a CTA gives any load still in flight a bounded 100 us to land
    // before the pair releases its shared memory.  On the normal path every
    // load was consumed by an MMA.
    if (((kTwoSm && crank != 0) || kMcast) && threadIdx.x == 0 &&
        *reinterpret_cast<volatile uint32_t *>(&g_status_word) != 0u) {
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 100000ull) {
        }
    }
    // Paired CTAs: neither leaves while the leader's MMAs may still read the
    // peer's shared memory or write its tensor memory, or while the other
    // CTA's multicast loads, commits or arrivals may still reach it.
    if (CS > 1) cluster_sync();
    if (warp == kWarpMma) {
        __syncwarp();
        if constexpr (kTwoSm)
            tmem_dealloc_pair(tmem_base, kTmemCols);
        else
            tmem_dealloc(tmem_base, kTmemCols);
    }
}

template <int MODE, int FORM>
static cudaError_t launch_mode(const CUtensorMap &tmH, const WMaps &wm, const Stage1Args &a,
                               int grid,
                               cudaStream_t stream) {
    constexpr int CS = FORM == kFormSingle ? 1 : 2;
    static std::atomic<uint32_t> configured_mask{0};  // per device (device ordinals < 32)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 32 || !(configured_mask.load() & (1u << dev))) {
        e = cudaFuncSetAttribute(stage1_kernel<MODE, FORM>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        if (CS > 1) {
            e = cudaFuncSetAttribute(stage1_kernel<MODE, FORM>,
                                     cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
            if (e != cudaSuccess) return e;
        }
        if (dev < 32) configured_mask.fetch_or(1u << dev);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // the prologue may overlap the previous kernel (see griddep_wait in the kernel)
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, stage1_kernel<MODE, FORM>, tmH, wm.w16, wm.w64, wm.w128,
                              wm.w256, a);
}

// How many 2-CTA clusters of Stage 1's pair forms the current device can
// hold at once (cached per device; 0 if the query fails).  Both pair forms
// launch with the same block size and dynamic shared memory, and one block
// fits per SM, so one query serves both.
static int max_pair_clusters() {
    static std::mutex mu;
    static int cached[64];
    static bool known[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (!known[dev]) {
        int n = 0;
        if (cudaFuncSetAttribute(stage1_kernel<kModeSample, kFormPairMma>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBytes) == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(2);
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = kSmemBytes;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&n, stage1_kernel<kModeSample, kFormPairMma>, &cfg) !=
                cudaSuccess)
                n = 0;
        }
        cudaGetLastError();  // a failed query leaves no sticky error
        cached[dev] = n;
        known[dev] = true;
    }
    return cached[dev];
}

template <int FORM>
static cudaError_t launch_form(int mode, const CUtensorMap &tmH, const WMaps &wm,
                               const Stage1Args &a, int grid, cudaStream_t stream) {
    switch (mode) {
        case kModeSample: return launch_mode<kModeSample, FORM>(tmH, wm, a, grid, stream);
        case kModeSampleStore:
            return launch_mode<kModeSampleStore, FORM>(tmH, wm, a, grid, stream);
        case kModeGemmBf16: return launch_mode<kModeGemmBf16, FORM>(tmH, wm, a, grid, stream);
        case kModeGemmF32: return launch_mode<kModeGemmF32, FORM>(tmH, wm, a, grid, stream);
        case kModeSampleLogprob:
            return launch_mode<kModeSampleLogprob, FORM>(tmH, wm, a, grid, stream);
        case kModeSampleXform:
            return launch_mode<kModeSampleXform, FORM>(tmH, wm, a, grid, stream);
        case kModeSampleXformLogprob:
            return launch_mode<kModeSampleXformLogprob, FORM>(tmH, wm, a, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

int stage1_form(int nM, int D, int grid) {
    // Pairs only when batch tiles come in pairs and every pair fits at once.
    const bool pair = (nM % 2 == 0) && (2 * max_pair_clusters() >= grid);
    if (!pair) return kFormSingle;
    // Measured on GB300 with the noise on (V = 128 K - 256 K): with two batch
    // tiles the pair MMA is ahead from D = 4096 (1.5-4%) and behind at 3584
    // (1.4%); with four it is behind at D <= 4096 (2.4-3.4%), even at 5120
    // and ahead from 6144 (1%).
    const int min_d = nM == 2 ? kPairMmaMinD2 : kPairMmaMinD;
    return D >= min_d ? kFormPairMma : kFormMulticast;
}

cudaError_t launch_stage1(int mode, const CUtensorMap &tmH, const WMaps &wm,
                          const Stage1Args &a, int grid,
                          cudaStream_t stream) {
    switch (stage1_form(a.nM, a.D, grid)) {
        case kFormPairMma: return launch_form<kFormPairMma>(mode, tmH, wm, a, grid, stream);
        case kFormMulticast: return launch_form<kFormMulticast>(mode, tmH, wm, a, grid, stream);
        default: return launch_form<kFormSingle>(mode, tmH, wm, a, grid, stream);
    }
}

cudaError_t status_word_address(uint32_t **out) {
    // A context that is destroyed and created again (cudaDeviceReset) loads
    // the module anew, so the cache is keyed by context, not by device.
    static std::mutex mu;
    static std::map<unsigned long long, uint32_t *> by_context;
    unsigned long long ctx = 0;
    bool have_ctx = current_context_id(&ctx);
    std::lock_guard<std::mutex> lock(mu);
    if (have_ctx) {
        auto it = by_context.find(ctx);
        if (it != by_context.end()) {
            *out = it->second;
            return cudaSuccess;
        }
    }
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_status_word);
    if (e != cudaSuccess) return e;
    // the lookup itself makes the device's primary context current if none was
    if (have_ctx || current_context_id(&ctx)) by_context[ctx] = static_cast<uint32_t *>(p);
    *out = static_cast<uint32_t *>(p);
    return cudaSuccess;
}

cudaError_t read_and_clear_status(cudaStream_t stream, uint32_t *word) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    uint32_t w = 0;
    e = cudaMemcpyFromSymbol(&w, g_status_word, sizeof(w));
    if (e != cudaSuccess) return e;
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero));
    if (e != cudaSuccess) return e;
    *word = w;
    return cudaSuccess;
}

}  // namespace fs

// fs_internal.h -- declarations shared by the library's translation units.
// Not part of the public C ABI (include/fs_sample.h is).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace fs {

// ---- Stage 1 tiling ------------------------------------------------------
// One CTA per SM, persistent over its share of the vocabulary.  A tile is
// 128 batch rows (MMA M, TMEM lanes) x up to 256 vocabulary rows (MMA N, TMEM
// columns); K advances 64 bf16 (one 128-byte swizzle span) per pipeline stage.
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kStages = 4;
constexpr int kUmmaK = 16;
constexpr int kABytes = kBM * kBK * 2;  // 16 KiB: H tile
constexpr int kBBytes = kBN * kBK * 2;  // 32 KiB: W tile
constexpr int kColParts = 4;                      // most epilogue warps per TMEM lane quarter
constexpr int kNumEpiWarps = 14;                  // 3 + 3 + 4 + 4
constexpr int kWarpTma = 12;                      // sub-partition 0
constexpr int kWarpMma = 13;                      // sub-partition 1
constexpr int kThreads = 16 * 32;                 // 512
constexpr int kTmemCols = 512;  // two 256-column accumulators
constexpr int kCombineBytes = kColParts * kBM * 20;  // per-row results of the column parts
// Dynamic shared memory: the per-CTA maximum.  The ring takes what the
// alignment slack, the barriers and the combine area leave: 4 stages for a
// full batch tile, and more when a small batch shrinks each stage's H slot.
constexpr int kSmemBytes = 232448;
// Barriers (256 B) and the combine area sit in front of the ring, rounded up
// to the 1 KB swizzle atom; a small batch's MMA reads up to 8 KB in front of
// its first H slot from there (see the kernel).
constexpr int kPreRingBytes = (256 + kCombineBytes + 1023) & ~1023;
constexpr int kRingBytes = kSmemBytes - 1024 - kPreRingBytes;
static_assert(kPreRingBytes >= 64 * kBK * 2, "room for a 64-lane offset of the A operand");
constexpr int kMaxStages = 8;
static_assert(kStages * (kABytes + kBBytes) <= kRingBytes, "ring of full batch tiles");
constexpr int kFinalTileUnits = 8;  // last tile of a partition: 128 rows
constexpr int kUnitRows = 16;  // vocabulary partitions are multiples of 16 rows

// ---- materialised-logits sampler ------------------------------------------
// A block scans one chunk of one row; the chunk (a multiple of one step,
// 256 threads x 8 entries) grows with B * V up to 64 K entries, aiming at
// about 4 blocks per SM, so that each thread scans a long run of its row and
// the screen has a good running best to reject against.
constexpr int kLogitsThreads = 256;
constexpr int kLogitsStep = kLogitsThreads * 8;
constexpr int kLogitsMaxChunk = 65536;

enum Stage1Mode : int {
    kModeSample = 0,       // fused: GEMM + temperature + Gumbel + tile argmax
    kModeSampleStore = 1,  // same, plus f32 logits written to HBM
    kModeGemmBf16 = 2,     // unfused GEMM: Y written as bf16, no sampling
    kModeGemmF32 = 3,      // unfused GEMM: Y written as f32, no sampling
    kModeSampleLogprob = 4,  // fused sampling plus the online log-mass of each row
    kModeSampleXform = 5,    // fused sampling after bias / soft-cap / token mask
    kModeSampleXformLogprob = 6,  // both
};

struct Plan {
    int64_t B, V, D;
    int nM;        // batch tiles of 128 rows
    int P;         // vocabulary partitions (one per CTA column)
    int G;         // CTAs launched = P * nM
    int nCand;     // candidate slots per row (one per partition)
    int64_t U;     // vocabulary units of 16 rows
    int maxTiles;  // max vocabulary tiles per CTA
    int nChunks;   // blocks per row of the materialised-logits sampler
    int logitsChunk;  // vocabulary entries per block of that sampler
    // Workspace bytes.  Every call lays out its candidate arrays, each
    // [slots][B] of 4-byte values rounded up to 256 B, with the slots it uses:
    // nCand for the fused calls, nChunks for the materialised-logits sampler.
    size_t wsBytes;        // fs_workspace_size: five arrays of max(nCand, nChunks) slots
    size_t wsSampleBytes;  // fused sampling: two arrays (score, index) of nCand slots
    size_t wsLogprobBytes; // fused sampling with log-masses: five arrays of nCand slots
    size_t wsLogitsBytes;  // materialised-logits sampler: two arrays of nChunks slots
};

bool make_plan(int64_t B, int64_t V, int64_t D, int num_sms, Plan *plan);

// Plan::wsSampleBytes for (B, V, D) on the current device (0 on a bad
// argument or without a usable device): the candidate bytes that
// fs_sample_ex, fs_stage1 and fs_stage2 need.
size_t sample_workspace_bytes(int64_t B, int64_t V, int64_t D);


struct Stage1Args {
    int32_t B, V, D;
    int32_t nM, P;
    int64_t U;
    const float *temps;  // nullable device [B]
    float temp_scalar;
    uint64_t seed, offset;
    uint32_t flags;
    float *cand_score;  // [nCand][B]
    int32_t *cand_idx;  // [nCand][B]
    float *cand_lt;     // [nCand][B] winner's l*invT          (kModeSampleLogprob)
    float *cand_m;      // [nCand][B] running max of l*invT      (kModeSampleLogprob)
    float *cand_s;      // [nCand][B] sum of exp(l*invT - max)  (kModeSampleLogprob)
    float *out_logits;  // [B][V] f32 (kModeSampleStore)
    void *out_y;        // [B][V] bf16/f32 (GEMM modes)
    int y_vec_ok;       // row starts of Y / out_logits are 16-byte aligned
    int h_box_rows;     // rows of the H tensor-map box (8..128; rows above are not loaded)
    int64_t vocab_offset;  // global index of W's first row (a multiple of 16): the
                           // noise and the candidate indices use global indices
    const float *bias;  // nullable [V], 16-byte aligned          (transform modes)
    float softcap;      // > 0: l = c * tanh(l / c)              (transform modes)
    const uint32_t *allow_mask;  // nullable [B][mask_words]     (transform modes)
    int64_t mask_words;
    uint64_t timeout_ns;
};

// W is read through four tensor maps with boxes of 16, 64, 128 and 256 rows
// (all 64 columns wide): whole tiles in one box per CTA, tails in 64- and
// 16-row boxes.
struct WMaps {
    CUtensorMap w16, w64, w128, w256;
};

cudaError_t launch_stage1(int mode, const CUtensorMap &tmH, const WMaps &wm,
                          const Stage1Args &a, int grid,
                          cudaStream_t stream);
// The launch form launch_stage1 takes on the current device for nM batch
// tiles, depth D and `grid` CTAs (FS_STAGE1_* of fs_sample.h).
int stage1_form(int nM, int D, int grid);

// Stage 2 reads Stage 1's device error word (status_word_address): while it
// is set, every row gets out_idx = -1 and NaN scores, so a call whose Stage 1
// gave up a bounded wait never returns tokens from a partial candidate buffer.
cudaError_t launch_stage2(const float *cand_score, const int32_t *cand_idx, int nCand,
                          int64_t B, const float *temps, float temp_scalar, int64_t *out_idx,
                          float *out_score, cudaStream_t stream);

// Stage 2 with the log-mass merge: also writes out_logprob [B] and/or the
// row's log-mass out_logmass [B] (either may be null).
cudaError_t launch_stage2_logprob(const float *cand_score, const int32_t *cand_idx,
                                  const float *cand_lt, const float *cand_m, const float *cand_s,
                                  int nCand, int64_t B, const float *temps, float temp_scalar,
                                  int64_t *out_idx, float *out_score, float *out_logprob,
                                  cudaStream_t stream, float *out_logmass = nullptr);

// Grouped sampler: per row, the group maximising log-mass + Gumbel (group noise).
cudaError_t launch_combine_groups(int64_t n_groups, int64_t B, const int64_t *group_idx,
                                  const float *group_logmass, uint64_t seed, uint64_t offset,
                                  int64_t *out_idx, int64_t *out_group, cudaStream_t stream);

cudaError_t launch_logits_sample(const void *Y, int y_dtype, int64_t B, int64_t V,
                                 const float *temps, float temp_scalar, uint64_t seed,
                                 uint64_t offset, uint32_t flags, float *cand_score,
                                 int32_t *cand_idx, int nChunks, int chunk,
                                 cudaStream_t stream);

cudaError_t launch_upload(const void *src, void *dst, int64_t bytes, const float *tsrc,
                          float *tdst, int64_t nt, cudaStream_t stream);
cudaError_t launch_debug_gumbel(const uint32_t *words, int64_t n, float *out_g,
                                cudaStream_t stream);
cudaError_t launch_debug_noise(uint64_t seed, uint64_t offset, int64_t b0, int64_t nb,
                               int64_t V, uint32_t *out_words, float *out_g,
                               cudaStream_t stream);

// Device error word of Stage 1 (bit 0: a bounded wait expired).
cudaError_t read_and_clear_status(cudaStream_t stream, uint32_t *word);

// Device address of that word in the current CUDA context, for the kernels of
// other translation units (looked up once per context, then cached).
cudaError_t status_word_address(uint32_t **out);

// Identifier of the CUDA context current on this thread (unique for the life
// of the process, unlike a context handle, which a destroyed context may pass
// on); false when no context is current or the driver lacks the query.
bool current_context_id(unsigned long long *id);

}  // namespace fs

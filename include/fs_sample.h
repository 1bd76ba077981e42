/*
 * fs_sample.h -- C ABI of the GB300 (sm_103a) fused LM-head + exact sampling
 * library (libfs_sample.so).
 *
 * The operation ("FlashSampling: Fast and Memory-Efficient Exact Sampling",
 * arXiv 2603.15854):
 *   - the LM-head GEMM l = H W^T with H [B, D] hidden states and W [V, D]
 *     vocabulary-major weights, both bf16 (the experimental setup's
 *     precision);
 *   - exact categorical sampling from softmax(l / T) by the Gumbel-max trick:
 *     draw i.i.d. Gumbels g, form s = l/T + g, return argmax s (method
 *     section, Algorithm I.1 of the Appendix);
 *   - fused in two stages (method section, "Stage 1 (Fused Kernel)" /
 *     "Stage 2 (Reduction)"): Stage 1 computes logits tile by tile on chip,
 *     applies the temperature, adds the noise and keeps one maximizer per row
 *     and per vocabulary tile, never writing the [B, V] logits to HBM; Stage 2
 *     reduces the small candidate buffer to one token per row.  Exactness:
 *     argmax decomposes over a partition of the vocabulary (Appendix C).
 *
 * Conventions shared by every entry point
 *   - Pointers named H, W, Y, out_*, temperatures and workspace are DEVICE
 *     pointers into memory the caller owns.  The library never frees them and
 *     keeps none of them after the call returns.
 *   - H and W must be 16-byte aligned and D must be a multiple of 8 (the
 *     tensor-memory-access unit needs 16-byte rows); otherwise the call
 *     returns FS_ERR_UNSUPPORTED and launches nothing.
 *   - H and W must be device memory of the current GPU (cudaMalloc-family or
 *     pool memory of that device).  Stage 1 reads them with tensor-memory
 *     loads, and in its paired forms (two CTAs of a cluster) a W box is
 *     multicast to both CTAs, or both CTAs' loads complete on one CTA's
 *     barrier to feed one MMA; those loads are kept to the calling GPU's own
 *     memory.  Page-locked host memory, another
 *     GPU's memory (peer access) and managed memory are refused with
 *     FS_ERR_UNSUPPORTED before anything is launched.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous on `stream`: a returned FS_OK means the
 *     work was enqueued; device-side errors surface at the caller's next
 *     synchronisation or through fs_get_device_status().
 *   - A bad argument returns an error status and launches nothing.  The reason
 *     is available from fs_last_error_string() (thread-local).
 *   - The sampled token of row b is a deterministic function of
 *     (H[b], W, T_b, seed, offset, b).  A decoder advances `offset` per step.
 *   - Noise: element (b, v) draws 32 random bits from Philox4x64-10 (Salmon et
 *     al., SC'11) with key (seed, 0) and counter (v >> 3, b, offset, 0): half
 *     (v & 1) of 64-bit output word (v & 7) >> 1.  u = ((x >> 8) | 1) * 2^-24,
 *     g = -log(-log(u)).  The score is s = fl(fl(l * fl(1/T)) + g) in f32.
 *     Ties in s go to the lowest vocabulary index; NaN never wins.
 *   - Temperatures: `temperature` (scalar) is used when `temperatures` is
 *     NULL, otherwise `temperatures` is a device f32 [B] array of per-row
 *     values.  A scalar that is not finite or not > 0 is rejected with
 *     FS_ERR_INVALID_ARG.  A per-row value that is not finite or not > 0 gives
 *     that row out_idx = -1 and out_score = NaN (greedy decoding is not part
 *     of the method).
 */
#ifndef FS_SAMPLE_H
#define FS_SAMPLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fs_status {
    FS_OK = 0,
    FS_ERR_INVALID_ARG = 1, /* null pointer, size < 1, bad scalar temperature  */
    FS_ERR_UNSUPPORTED = 2, /* alignment / D % 8 / size limits / no device      */
    FS_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed              */
    FS_ERR_TIMEOUT = 4,     /* a kernel gave up a bounded wait (device word)     */
    FS_ERR_NO_MEMORY = 5,   /* workspace allocation failed or is too small       */
} fs_status;

/* Flags of fs_sample_ex / fs_stage1 / fs_sample_from_logits. */
#define FS_FLAG_NO_NOISE 0x1u     /* g = 0: plain argmax of l/T (tie tests only)  */
#define FS_FLAG_STORE_LOGITS 0x2u /* also write f32 logits l (before 1/T) to      \
                                     out_logits [B, V]: the logits-store flag the  \
                                     IO-model check uses (Section 3)               */

/* Test hook of fs_stage1 / fs_sample_ex: Stage 1's loader issues no loads,
 * so the first bounded wait of every CTA expires (after FS_WAIT_TIMEOUT_MS,
 * default 4000 ms, read from the environment once per process); the kernel
 * then sets the device error word, stops and returns, and
 * fs_get_device_status reports FS_ERR_TIMEOUT.  Exercises the failure path
 * without a fault; never use it outside tests. */
#define FS_FLAG_TEST_NO_LOADS 0x100u

/* dtype codes of materialised logits Y. */
#define FS_DTYPE_BF16 0
#define FS_DTYPE_F32 1

/* Upper limits checked on the host. */
#define FS_MAX_VOCAB 2147483647LL /* indices are stored as int32 candidates */
#define FS_MAX_BATCH 16777216LL

/* ---------------------------------------------------------------------------
 * fs_sample -- the whole hot path: Stage 1 then Stage 2.
 *   H            device bf16 [B, D], row-major (row stride D elements)
 *   W            device bf16 [V, D], row-major (row stride D elements)
 *   temperature  scalar T (used when temperatures == NULL)
 *   temperatures NULL or device f32 [B]
 *   seed, offset Philox key word and counter word (see Noise above)
 *   out_idx      device int64 [B]: sampled token per row (-1: invalid row T)
 *   out_score    NULL or device f32 [B]: the winning perturbed score s
 * Candidate workspace: a buffer cached per (device, stream) inside the
 * library, grown stream-ordered with cudaMallocAsync/cudaFreeAsync.  Calls on
 * one stream reuse it in order.  fs_release_workspaces() frees the cache.
 * Returns FS_ERR_NO_MEMORY if the workspace cannot be grown.  While `stream`
 * is being captured into a CUDA graph the cache does not grow (memory
 * allocated then would belong to the graph): a call that needs more than an
 * earlier call of the same stream left returns FS_ERR_UNSUPPORTED; make one
 * call of the same size before capturing, or use fs_sample_ex.
 * ------------------------------------------------------------------------- */
fs_status fs_sample(const void *H, const void *W, int64_t B, int64_t V, int64_t D,
                    float temperature, const float *temperatures, uint64_t seed,
                    uint64_t offset, int64_t *out_idx, float *out_score, void *stream);

/* ---------------------------------------------------------------------------
 * fs_sample_host -- fs_sample with the per-call data in HOST memory, for a
 * decode loop whose hidden states and sampled tokens live on the host.  The
 * weights stay resident on the device (method section: W is read from HBM
 * once per call).
 *   H_host            host bf16 [B, D], row-major; must stay unchanged until
 *                     `stream` reaches the end of the call
 *   W                 device bf16 [V, D], row-major, 16-byte aligned
 *   temperatures_host NULL or host f32 [B] (same lifetime rule as H_host)
 *   out_idx_host      host int64 [B]; valid once `stream` has reached the end
 *                     of this call (cudaStreamSynchronize or an event)
 *   out_score_host    NULL or host f32 [B], as out_idx_host
 * Order of work: H (and the temperatures) are copied into one of two device
 * slots used alternately, then `stream` runs Stage 1 and Stage 2.
 *   - Page-locked inputs (16-byte aligned H) are copied by a small kernel on
 *     `stream` that reads them through their mapped device address.  It is
 *     launched with programmatic dependent launch like both stages, so
 *     back-to-back calls keep overlapping their set-up.
 *   - Pageable inputs are copied by the CUDA runtime (staged before the call
 *     returns) on an internal upload stream that waits for the previous reader
 *     of the slot; `stream` waits for that copy.
 * Page-locked outputs are written by Stage 2 directly through their mapped
 * device address; pageable outputs are staged on the device and copied back
 * on `stream` (that copy completes before the call returns).  While `stream`
 * is being captured into a CUDA graph, pageable inputs are copied on `stream`
 * itself (page-locked buffers are recommended), and the device staging must
 * already exist from an earlier call of the same size on that stream (else
 * FS_ERR_UNSUPPORTED, as for fs_sample).
 * Device state (upload stream, events, slots) is cached per (device, stream)
 * and freed by fs_release_workspaces().  Host pointers need no particular
 * alignment beyond their element size for page-locked outputs.  Results are
 * bit-identical to fs_sample on the same data.
 * ------------------------------------------------------------------------- */
fs_status fs_sample_host(const void *H_host, const void *W, int64_t B, int64_t V, int64_t D,
                         float temperature, const float *temperatures_host, uint64_t seed,
                         uint64_t offset, int64_t *out_idx_host, float *out_score_host,
                         void *stream);

/* Bytes of caller workspace for (B, V, D) on the current device: enough for
 * every entry point that takes a workspace.  It holds five equal candidate
 * arrays; the calls that sample without a log-probability (fs_sample_ex,
 * fs_stage1/fs_stage2, fs_sample_from_logits, fs_sample_unfused and
 * fs_sample_transformed without out_logprob) use only the first two and
 * accept any ws_bytes >= 2/5 of this size.
 * Returns 0 on a bad argument or when no device is visible. */
size_t fs_workspace_size(int64_t B, int64_t V, int64_t D);

/* ---------------------------------------------------------------------------
 * fs_sample_ex -- fs_sample with a caller workspace and flags.
 *   flags       FS_FLAG_NO_NOISE | FS_FLAG_STORE_LOGITS
 *   out_logits  device f32 [B, V] row-major; required iff FS_FLAG_STORE_LOGITS
 *               (receives l = H W^T before the temperature; the fused path
 *               otherwise never materialises it)
 *   workspace   device buffer of ws_bytes >= fs_workspace_size(B, V, D),
 *               16-byte aligned; FS_ERR_NO_MEMORY if smaller
 * ------------------------------------------------------------------------- */
fs_status fs_sample_ex(const void *H, const void *W, int64_t B, int64_t V, int64_t D,
                       float temperature, const float *temperatures, uint64_t seed,
                       uint64_t offset, uint32_t flags, int64_t *out_idx,
                       float *out_score, float *out_logits, void *workspace,
                       size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * The two stages separately (method section, Stage 1 / Stage 2).
 * fs_stage1 runs the fused GEMM + temperature + Gumbel + tile-argmax kernel
 * and leaves one (score, index) candidate per (row, candidate slot) in
 * `workspace`; fs_stage2 reduces them to out_idx / out_score.  Both must be
 * called with the same (B, V, D) on the same device; fs_stage2 also needs the
 * temperatures to mark invalid rows.  fs_sample_ex == fs_stage1 + fs_stage2.
 * Argument meanings as for fs_sample_ex.
 * ------------------------------------------------------------------------- */
fs_status fs_stage1(const void *H, const void *W, int64_t B, int64_t V, int64_t D,
                    float temperature, const float *temperatures, uint64_t seed,
                    uint64_t offset, uint32_t flags, float *out_logits,
                    void *workspace, size_t ws_bytes, void *stream);
fs_status fs_stage2(int64_t B, int64_t V, int64_t D, float temperature,
                    const float *temperatures, int64_t *out_idx, float *out_score,
                    const void *workspace, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * fs_sample_logprob -- fs_sample_ex that also returns the log-probability of
 * each sampled token under softmax(l~), l~ = l * fl(1/T):
 *   out_logprob[b] = l~[idx] - log sum_v exp(l~[v]).
 * Stage 1 keeps, besides the per-row maximizer, each partition's log-mass
 * (max l~, sum exp(l~ - max)) -- the online-normalizer analogy of the method
 * section and the per-shard sample plus log-mass of the grouped /
 * tensor-parallel variant (Section 4) -- and Stage 2 merges them over the
 * whole vocabulary.  Elements with a non-finite l~ are left out of the sum; a
 * row whose sampled l~ is not finite, or with an invalid temperature, gets
 * NaN.  The logits are never written to HBM.  Costs one exp2 per element on
 * top of fs_sample.
 *   out_logprob  device f32 [B] (required)
 *   workspace    as fs_sample_ex (fs_workspace_size covers this call)
 * Indices and scores are identical to fs_sample_ex's.
 * ------------------------------------------------------------------------- */
fs_status fs_sample_logprob(const void *H, const void *W, int64_t B, int64_t V, int64_t D,
                            float temperature, const float *temperatures, uint64_t seed,
                            uint64_t offset, int64_t *out_idx, float *out_score,
                            float *out_logprob, void *workspace, size_t ws_bytes,
                            void *stream);

/* ---------------------------------------------------------------------------
 * fs_sample_transformed -- the fused path with deterministic transforms
 * applied to the f32 logits in the Stage 1 epilogue, before the temperature
 * (method section: Stage 1 applies deterministic transforms before the
 * noise; the pages do not list them).  In this order, each rounded to f32:
 *   l' = l + bias[v]                   bias: nullable device f32 [V], 16-byte aligned
 *   l' = c * tanh(l' / c)   if c > 0   softcap: logit soft-capping (0 = off)
 *   l' = -inf               where bit (v & 31) of allow_mask[b * mask_words + (v >> 5)]
 *                           is 0 (allow_mask: nullable device uint32 [B][mask_words],
 *                           mask_words >= ceil(V / 32); constrained decoding)
 * then l~ = l' * fl(1/T), s = l~ + g and the argmax as in fs_sample.
 *   tf           required; a zero-initialised struct means no transform
 *   flags        FS_FLAG_NO_NOISE only
 *   out_logprob  nullable device f32 [B]: as fs_sample_logprob, over l~
 *   workspace    as fs_sample_ex
 * A row whose tokens are all masked gets out_idx = -1 and score -inf.
 * ------------------------------------------------------------------------- */
typedef struct fs_transforms {
    const float *bias;
    float softcap;
    const uint32_t *allow_mask;
    int64_t mask_words;
} fs_transforms;

fs_status fs_sample_transformed(const void *H, const void *W, int64_t B, int64_t V, int64_t D,
                                const fs_transforms *tf, float temperature,
                                const float *temperatures, uint64_t seed, uint64_t offset,
                                uint32_t flags, int64_t *out_idx, float *out_score,
                                float *out_logprob, void *workspace, size_t ws_bytes,
                                void *stream);

/* ---------------------------------------------------------------------------
 * Grouped (hierarchical) sampling -- the pages' variant for online and
 * tensor-parallel settings (abstract; Section 4: each vocabulary shard returns
 * its own sample and log-mass), exact by the hierarchical
 * factorisation P(v) = P(group(v)) P(v | group(v)).
 *
 * fs_sample_shard   the fused path over one vocabulary shard W_shard
 *                   [V_shard, D] whose first row has global index
 *                   vocab_offset (a multiple of 16): the noise of every
 *                   element is that of its global index, out_idx holds global
 *                   indices, and out_logmass [B] (required, device f32) the
 *                   shard's log sum exp(l~) over its finite l~ (-inf if none,
 *                   NaN for an invalid T).  out_idx / out_score equal what the
 *                   unsharded call computes restricted to the shard.
 * fs_combine_groups per row b, draw group g with probability proportional to
 *                   exp(group_logmass[g][b]) -- argmax_g of the f32 sum
 *                   group_logmass[g][b] + G_g, G from Philox4x64-10 with key
 *                   (seed, 0) and counter (g >> 3, b, offset, 1) (word 3 = 1:
 *                   apart from the token noise) -- and return
 *                   out_idx[b] = group_idx[g][b].  group_idx: device int64
 *                   [n_groups][B]; group_logmass: device f32 [n_groups][B];
 *                   out_group: nullable device int64 [B].  Ties go to the
 *                   lower g; NaN and -inf never win (-1 if no group can).
 * Use the same (seed, offset) in the shard calls and a fresh seed for the
 * combine.  The result is an exact sample from softmax(l~) over the union of
 * the shards, but a different one from fs_sample's with the same seed.
 * ------------------------------------------------------------------------- */
fs_status fs_sample_shard(const void *H, const void *W_shard, int64_t B, int64_t V_shard,
                          int64_t D, int64_t vocab_offset, float temperature,
                          const float *temperatures, uint64_t seed, uint64_t offset,
                          int64_t *out_idx, float *out_score, float *out_logmass,
                          void *workspace, size_t ws_bytes, void *stream);
fs_status fs_combine_groups(int64_t n_groups, int64_t B, const int64_t *group_idx,
                            const float *group_logmass, uint64_t seed, uint64_t offset,
                            int64_t *out_idx, int64_t *out_group, void *stream);

/* ---------------------------------------------------------------------------
 * Unfused comparator: the baseline the IO model of Section 3 describes, a
 * GEMM that writes the logits Y to HBM followed by a sampling pass that reads
 * them back.  Same noise, temperature and tie rule as the fused path.
 *
 * fs_logits_gemm        Y = H W^T, written as bf16 or f32 [B, V] row-major.
 * fs_sample_from_logits Gumbel-max over materialised logits Y [B, V]
 *                       (bf16 or f32, row-major, row stride V); flags:
 *                       FS_FLAG_NO_NOISE only.  workspace as fs_sample_ex.
 * fs_sample_unfused     fs_logits_gemm then fs_sample_from_logits; Y is a
 *                       caller buffer of B*V elements of y_dtype.
 * With y_dtype = FS_DTYPE_F32 the unfused path samples exactly what the fused
 * path samples; with FS_DTYPE_BF16 the logits are rounded to bf16 first.
 * ------------------------------------------------------------------------- */
fs_status fs_logits_gemm(const void *H, const void *W, int64_t B, int64_t V, int64_t D,
                         void *Y, int y_dtype, void *stream);
fs_status fs_sample_from_logits(const void *Y, int y_dtype, int64_t B, int64_t V,
                                float temperature, const float *temperatures,
                                uint64_t seed, uint64_t offset, uint32_t flags,
                                int64_t *out_idx, float *out_score, void *workspace,
                                size_t ws_bytes, void *stream);
fs_status fs_sample_unfused(const void *H, const void *W, int64_t B, int64_t V,
                            int64_t D, float temperature, const float *temperatures,
                            uint64_t seed, uint64_t offset, void *Y, int y_dtype,
                            int64_t *out_idx, float *out_score, void *workspace,
                            size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * fs_debug_noise -- test hook: the random word and Gumbel of every element
 * (b, v) for rows b0 .. b0+nb-1 and vocabulary 0 .. V-1, computed by the
 * same device functions as the Stage 1 epilogue.
 *   out_words  NULL or device uint32 [nb, V];  out_g  NULL or device f32 [nb, V]
 * ------------------------------------------------------------------------- */
fs_status fs_debug_noise(uint64_t seed, uint64_t offset, int64_t b0, int64_t nb,
                         int64_t V, uint32_t *out_words, float *out_g, void *stream);

/* ---------------------------------------------------------------------------
 * fs_debug_gumbel -- test hook: g = -log(-log(u)) of given 32-bit random
 * words (u = ((x >> 8) | 1) * 2^-24, see Noise above), by the device function
 * every sampling kernel uses.
 *   words  device uint32 [n];  out_g  device f32 [n];  both 4-byte aligned
 * ------------------------------------------------------------------------- */
fs_status fs_debug_gumbel(const uint32_t *words, int64_t n, float *out_g, void *stream);

/* ---------------------------------------------------------------------------
 * fs_get_device_status -- synchronise `stream`, then read and clear the
 * library's device error word on the current device.  *out_word (may be
 * NULL) receives the raw bits: 1 = a bounded wait inside a kernel expired.
 * Returns FS_ERR_TIMEOUT if any bit was set, FS_ERR_CUDA if a CUDA call
 * failed, FS_OK otherwise.
 * While the word is set, every Stage 2 (of any sampling entry point) writes
 * out_idx = -1 and NaN to out_score / out_logprob / out_logmass for every
 * row instead of reducing candidates, so a call whose Stage 1 gave up never
 * returns tokens; clearing the word here restores normal results.
 * ------------------------------------------------------------------------- */
fs_status fs_get_device_status(void *stream, uint32_t *out_word);

/* ---------------------------------------------------------------------------
 * fs_plan_info -- host-only description of the Stage 1 schedule for
 * (B, V, D) on a GPU with num_sms SMs; launches nothing and needs no device.
 *   out[0] batch tiles of 128 rows (nM)       out[1] vocabulary partitions (P)
 *   out[2] CTAs launched (P * nM)             out[3] candidate slots per row
 *   out[4] workspace bytes                    out[5] max vocab tiles per CTA
 * ------------------------------------------------------------------------- */
fs_status fs_plan_info(int64_t B, int64_t V, int64_t D, int num_sms, int64_t out[6]);

/* ---------------------------------------------------------------------------
 * fs_stage1_form -- which form of Stage 1 (method section: one batch tile x
 * one vocabulary tile per step, here in one of three launch forms) the
 * sampling and GEMM entry points launch for (B, V, D) on the current GPU.
 * Launches nothing; the first call per device queries how many 2-CTA
 * clusters fit at once.
 *   FS_STAGE1_ONE_CTA          one CTA per (batch tile, vocabulary partition):
 *                              one or an odd number of 128-row batch tiles,
 *                              or pairs that would not all fit at once
 *   FS_STAGE1_MULTICAST_PAIR   2-CTA clusters over two batch tiles, each CTA
 *                              its own 128-row MMA on W boxes multicast to
 *                              both (an even number of batch tiles, D below
 *                              4096 with two of them, below 6144 with more)
 *   FS_STAGE1_PAIR_MMA         2-CTA clusters sharing one 256-row MMA
 *                              (tcgen05 cta_group::2) for larger D
 * Every form computes the same samples.  Returns FS_ERR_INVALID_ARG for a
 * NULL out_form or a bad shape, FS_ERR_UNSUPPORTED / FS_ERR_CUDA when the
 * current device is not an sm_103 GPU or cannot be queried.
 * ------------------------------------------------------------------------- */
enum { FS_STAGE1_ONE_CTA = 0, FS_STAGE1_MULTICAST_PAIR = 1, FS_STAGE1_PAIR_MMA = 2 };
fs_status fs_stage1_form(int64_t B, int64_t V, int64_t D, int *out_form);

/* ---------------------------------------------------------------------------
 * fs_sample_noalloc -- fs_sample that allocates no device memory.  The paper
 * has no counterpart: this is a library convenience.  It is for callers that
 * cannot allocate: applications that reserve all device memory up front and
 * forbid allocation afterwards (an inference server's own memory pool, a
 * plug-in whose host owns the allocator), and decode loops that cannot afford
 * cudaMalloc's possible device synchronisation.
 * Arguments, results and errors are those of fs_sample.  The candidate
 * scratch is a static array of FS_NOALLOC_SCRATCH_BYTES inside the library's
 * device memory (held on every GPU that loads the library until the process
 * exits).  A call keeps two candidate arrays (score, index) of P x B
 * four-byte values each, rounded up to 256 bytes, where P = the vocabulary
 * partitions of Stage 1 = min(floor(SMs / ceil(B / 128)), ceil(V / 16)), at
 * least 1; a call that needs more than the array returns FS_ERR_UNSUPPORTED
 * and launches nothing (on a 152-SM GPU every B up to 131072 fits).
 * The first call in each CUDA context looks up the array's device address
 * (cudaGetSymbolAddress), so make that first call before any stream capture.
 * All calls share the array: calls whose kernels overlap on the GPU (other
 * streams, other host threads) race on it and must be serialised by the
 * caller.  Nothing in it needs clearing between calls.
 * ------------------------------------------------------------------------- */
#define FS_NOALLOC_SCRATCH_BYTES (1 << 20)
fs_status fs_sample_noalloc(const void *H, const void *W, int64_t B, int64_t V, int64_t D,
                            float temperature, const float *temperatures, uint64_t seed,
                            uint64_t offset, int64_t *out_idx, float *out_score,
                            void *stream);

/* Frees every workspace cached by fs_sample and every staging block, upload
 * stream and event cached by fs_sample_host (all devices and streams).  It
 * synchronises the device (cudaFree).  The caller must make sure that no
 * other library call runs concurrently on another host thread, and that no
 * work of those calls still needs the freed memory. */
fs_status fs_release_workspaces(void);

/* Thread-local text for the last non-FS_OK status of this thread. */
const char *fs_last_error_string(void);

/* Library version string. */
const char *fs_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FS_SAMPLE_H */

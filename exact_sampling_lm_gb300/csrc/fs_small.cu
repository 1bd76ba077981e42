// fs_small.cu -- the small kernels around Stage 1:
//   * Stage 2 ("FlashSampling: Fast and Memory-Efficient Exact Sampling",
//     method section, Stage 2): argmax over the candidate buffer of shape
//     [candidate slots, B], one warp per row; a variant that also merges the
//     partitions' log-masses into the sampled token's log-probability;
//   * the group combine of grouped sampling (a group drawn by its log-mass);
//   * the sampling pass of the unfused comparator (the IO-model section's
//     baseline, which samples from logits that a GEMM has written out);
//   * the upload of a host-buffer call's page-locked inputs;
//   * debug kernels exposing the epilogue's noise functions for tests.
// All sampling kernels use the same noise functions and tie rule as Stage 1:
// higher score wins, equal scores go to the lower vocabulary index, NaN never
// wins.
#include <cuda_bf16.h>
#include <math.h>

#include "fs_internal.h"
#include "fs_noise.cuh"
#include "fs_ptx.cuh"

namespace fs {

namespace {

// (s, i) beats (best, bi)?  Indices compare as unsigned so that the "no
// candidate" index -1 loses every tie.
__device__ __forceinline__ bool better(float s, uint32_t i, float best, uint32_t bi) {
    return s > best || (s == best && i < bi);
}

__device__ __forceinline__ void warp_argmax(float &best, uint32_t &bi) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        const float s = __shfl_xor_sync(0xffffffffu, best, d);
        const uint32_t i = __shfl_xor_sync(0xffffffffu, bi, d);
        if (better(s, i, best, bi)) {
            best = s;
            bi = i;
        }
    }
}

__device__ __forceinline__ bool temperature_ok(float T) { return isfinite(T) && T > 0.0f; }

}  // namespace

// ------------------------------------------------------------------ Stage 2
constexpr int kStage2Warps = 8;

__global__ void __launch_bounds__(kStage2Warps * 32)
    stage2_kernel(const float *__restrict__ cand_score, const int32_t *__restrict__ cand_idx,
                  int nCand, int64_t B, const float *__restrict__ temps, float temp_scalar,
                  int64_t *__restrict__ out_idx, float *__restrict__ out_score,
                  const uint32_t *__restrict__ status) {
    // The next kernel of the stream (the next call's Stage 1) may launch now:
    // it only sets itself up before waiting for this grid.  Launched with
    // programmatic serialization itself: wait for the producing grid.
    griddep_launch_dependents();
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int64_t b = static_cast<int64_t>(blockIdx.x) * kStage2Warps + (threadIdx.x >> 5);
    if (b >= B) return;
    if (*status != 0u) {
        // a Stage 1 gave up a bounded wait: its candidates are incomplete
        if (lane == 0) {
            out_idx[b] = -1;
            if (out_score) out_score[b] = __int_as_float(0x7fc00000);
        }
        return;
    }
    float best = -INFINITY;
    uint32_t bi = 0xFFFFFFFFu;
    for (int i = lane; i < nCand; i += 32) {
        const float s = cand_score[static_cast<int64_t>(i) * B + b];
        const uint32_t id = static_cast<uint32_t>(cand_idx[static_cast<int64_t>(i) * B + b]);
        if (better(s, id, best, bi)) {
            best = s;
            bi = id;
        }
    }
    warp_argmax(best, bi);
    if (lane == 0) {
        const float T = temps ? temps[b] : temp_scalar;
        const bool ok = temperature_ok(T);
        out_idx[b] = (ok && bi != 0xFFFFFFFFu) ? static_cast<int64_t>(bi) : -1;
        if (out_score) out_score[b] = ok ? best : __int_as_float(0x7fc00000);
    }
}

cudaError_t launch_stage2(const float *cand_score, const int32_t *cand_idx, int nCand,
                          int64_t B, const float *temps, float temp_scalar, int64_t *out_idx,
                          float *out_score, cudaStream_t stream) {
    const int64_t blocks = (B + kStage2Warps - 1) / kStage2Warps;
    // Programmatic dependent launch: the blocks may be scheduled while the
    // producing kernel finishes; griddep_wait() orders the reads.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kStage2Warps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    uint32_t *status = nullptr;
    cudaError_t e = status_word_address(&status);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, stage2_kernel, cand_score, cand_idx, nCand, B, temps,
                              temp_scalar, out_idx, out_score, static_cast<const uint32_t *>(status));
}

// ------------------------------------------------------------------ host-buffer upload
// Copies a call's H (n16 16-byte units) and per-row temperatures (nt floats)
// from page-locked host memory, through its mapped device address, into the
// call's device slot.  Launched with programmatic serialization and
// triggering its dependents at once: it reads only host memory written before
// the call and writes a slot that the Stage 1 two calls back has finished
// loading (that Stage 1 triggered the Stage 2 whose start let this kernel
// launch), so it needs no wait; the next Stage 1 waits for it before reading
// the slot.
__global__ void upload_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst, int64_t n16,
                              const float *__restrict__ tsrc, float *__restrict__ tdst,
                              int64_t nt) {
    griddep_launch_dependents();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
         i += stride)
        dst[i] = src[i];
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nt;
         i += stride)
        tdst[i] = tsrc[i];
}

cudaError_t launch_upload(const void *src, void *dst, int64_t bytes, const float *tsrc,
                          float *tdst, int64_t nt, cudaStream_t stream) {
    const int64_t n16 = bytes / 16;
    int64_t blocks = (n16 + 255) / 256;
    if (blocks > 256) blocks = 256;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, upload_kernel, static_cast<const uint4 *>(src),
                              static_cast<uint4 *>(dst), n16, tsrc, tdst, nt);
}

// ------------------------------------------------------------------ Stage 2 with log-mass
// Besides the argmax, each row merges the partitions' log-masses
// (m_j, s_j) = (max l~, sum exp(l~ - max)) over the finite l~ into
// (M, S) and returns log p(idx) = (l~[idx] - M) - log S, the log-probability
// of the sampled token under softmax(l~) (the grouped variant's "local
// log-mass" summaries, reduced over the whole vocabulary).
__device__ __forceinline__ void lse_merge_acc(float &m, float &s, float m2, float s2) {
    if (!(s2 > 0.0f)) return;
    if (m2 > m) {
        s = s * expf(m - m2) + s2;
        m = m2;
    } else {
        s += s2 * expf(m2 - m);
    }
}

__global__ void __launch_bounds__(kStage2Warps * 32)
    stage2_logprob_kernel(const float *__restrict__ cand_score,
                          const int32_t *__restrict__ cand_idx, const float *__restrict__ cand_lt,
                          const float *__restrict__ cand_m, const float *__restrict__ cand_s,
                          int nCand, int64_t B, const float *__restrict__ temps,
                          float temp_scalar, int64_t *__restrict__ out_idx,
                          float *__restrict__ out_score, float *__restrict__ out_logprob,
                          float *__restrict__ out_logmass, const uint32_t *__restrict__ status) {
    griddep_launch_dependents();  // as in stage2_kernel
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int64_t b = static_cast<int64_t>(blockIdx.x) * kStage2Warps + (threadIdx.x >> 5);
    if (b >= B) return;
    if (*status != 0u) {  // as in stage2_kernel
        if (lane == 0) {
            const float nan = __int_as_float(0x7fc00000);
            out_idx[b] = -1;
            if (out_score) out_score[b] = nan;
            if (out_logprob) out_logprob[b] = nan;
            if (out_logmass) out_logmass[b] = nan;
        }
        return;
    }
    float best = -INFINITY, blt = __int_as_float(0x7fc00000);
    uint32_t bi = 0xFFFFFFFFu;
    float m = -INFINITY, sum = 0.0f;
    for (int i = lane; i < nCand; i += 32) {
        const int64_t o = static_cast<int64_t>(i) * B + b;
        const float sc = cand_score[o];
        const uint32_t id = static_cast<uint32_t>(cand_idx[o]);
        if (better(sc, id, best, bi)) {
            best = sc;
            bi = id;
            blt = cand_lt[o];
        }
        lse_merge_acc(m, sum, cand_m[o], cand_s[o]);
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        const float sc = __shfl_xor_sync(0xffffffffu, best, d);
        const uint32_t id = __shfl_xor_sync(0xffffffffu, bi, d);
        const float lt2 = __shfl_xor_sync(0xffffffffu, blt, d);
        const float m2 = __shfl_xor_sync(0xffffffffu, m, d);
        const float s2 = __shfl_xor_sync(0xffffffffu, sum, d);
        if (better(sc, id, best, bi)) {
            best = sc;
            bi = id;
            blt = lt2;
        }
        lse_merge_acc(m, sum, m2, s2);
    }
    if (lane == 0) {
        const float T = temps ? temps[b] : temp_scalar;
        const bool ok = temperature_ok(T);
        const bool found = ok && bi != 0xFFFFFFFFu;
        out_idx[b] = found ? static_cast<int64_t>(bi) : -1;
        if (out_score) out_score[b] = ok ? best : __int_as_float(0x7fc00000);
        const bool lp_ok = found && isfinite(blt) && sum > 0.0f;
        if (out_logprob)
            out_logprob[b] = lp_ok ? (blt - m) - logf(sum) : __int_as_float(0x7fc00000);
        if (out_logmass)
            out_logmass[b] = !ok ? __int_as_float(0x7fc00000)
                                 : (sum > 0.0f ? m + logf(sum) : -INFINITY);
    }
}

cudaError_t launch_stage2_logprob(const float *cand_score, const int32_t *cand_idx,
                                  const float *cand_lt, const float *cand_m, const float *cand_s,
                                  int nCand, int64_t B, const float *temps, float temp_scalar,
                                  int64_t *out_idx, float *out_score, float *out_logprob,
                                  cudaStream_t stream, float *out_logmass) {
    const int64_t blocks = (B + kStage2Warps - 1) / kStage2Warps;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kStage2Warps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    uint32_t *status = nullptr;
    cudaError_t e = status_word_address(&status);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, stage2_logprob_kernel, cand_score, cand_idx, cand_lt, cand_m,
                              cand_s, nCand, B, temps, temp_scalar, out_idx, out_score,
                              out_logprob, out_logmass, static_cast<const uint32_t *>(status));
}

// ------------------------------------------------------------------ grouped sampler
// The pages' grouped variant: every group of the vocabulary has returned a
// local sample and its log-mass; per row, draw group g with probability
// proportional to exp(logmass[g]) -- as argmax_g logmass[g] + G_g with
// Gumbels from Philox4x64-10, key (seed, 0), counter (g >> 3, b, offset, 1)
// (word 3 = 1 keeps these draws apart from the token noise) -- and return
// that group's sample.  One thread per row; ties go to the lower g, NaN and
// -inf never win.
__global__ void combine_groups_kernel(int64_t n_groups, int64_t B,
                                      const int64_t *__restrict__ group_idx,
                                      const float *__restrict__ group_logmass, uint64_t seed,
                                      uint64_t offset, int64_t *__restrict__ out_idx,
                                      int64_t *__restrict__ out_group) {
    const int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (b >= B) return;
    float best = -INFINITY;
    int64_t gbest = -1;
    for (int64_t g8 = 0; g8 * 8 < n_groups; ++g8) {
        uint64_t w[4];
        philox4x64_10_block(static_cast<uint64_t>(g8), static_cast<uint64_t>(b), offset, 1ull,
                            seed, w);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int64_t g = g8 * 8 + e;
            if (g < n_groups) {
                const uint32_t x = (e & 1) ? static_cast<uint32_t>(w[e >> 1] >> 32)
                                           : static_cast<uint32_t>(w[e >> 1]);
                const float s = __fadd_rn(group_logmass[g * B + b], gumbel_from_word(x));
                if (s > best) {
                    best = s;
                    gbest = g;
                }
            }
        }
    }
    out_idx[b] = gbest >= 0 ? group_idx[gbest * B + b] : -1;
    if (out_group) out_group[b] = gbest;
}

cudaError_t launch_combine_groups(int64_t n_groups, int64_t B, const int64_t *group_idx,
                                  const float *group_logmass, uint64_t seed, uint64_t offset,
                                  int64_t *out_idx, int64_t *out_group, cudaStream_t stream) {
    const int64_t blocks = (B + 127) / 128;
    combine_groups_kernel<<<static_cast<unsigned>(blocks), 128, 0, stream>>>(
        n_groups, B, group_idx, group_logmass, seed, offset, out_idx, out_group);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ unfused sampling pass
// Block (chunk, row): 256 threads scan `chunk` logits of one row, 8 per
// thread per step (one Philox call), then reduce to one candidate.  Like the
// Stage 1 epilogue, each step screens its 8 elements against the thread's
// best before the step (screen_lg2_tail / screen_bound) and pays for the
// exact Gumbel only for the survivors, lowest index first; the screen is
// conservative, so the result equals scoring every element.  A thread
// scores its first element exactly and screens the rest of that step
// against it, instead of scoring all 8.  The fused and unfused paths then
// differ by the logits' write and read-back, the traffic the IO model
// counts, and by the noise work that the fused kernel hides under its MMAs.
template <typename T>
__device__ __forceinline__ void load8(const T *row, int64_t v, int64_t v_end, bool vec_ok,
                                      float (&l)[8]);

template <>
__device__ __forceinline__ void load8<float>(const float *row, int64_t v, int64_t v_end,
                                             bool vec_ok, float (&l)[8]) {
    if (vec_ok && v + 8 <= v_end) {
        const float4 a = __ldcs(reinterpret_cast<const float4 *>(row + v));
        const float4 b = __ldcs(reinterpret_cast<const float4 *>(row + v + 4));
        l[0] = a.x; l[1] = a.y; l[2] = a.z; l[3] = a.w;
        l[4] = b.x; l[5] = b.y; l[6] = b.z; l[7] = b.w;
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) l[e] = (v + e < v_end) ? row[v + e] : 0.0f;
    }
}

template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16 *row, int64_t v,
                                                     int64_t v_end, bool vec_ok, float (&l)[8]) {
    if (vec_ok && v + 8 <= v_end) {
        const uint4 a = __ldcs(reinterpret_cast<const uint4 *>(row + v));
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            l[2 * j] = __uint_as_float(w[j] << 16);
            l[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            l[e] = (v + e < v_end) ? __bfloat162float(row[v + e]) : 0.0f;
    }
}

template <typename T>
__global__ void __launch_bounds__(kLogitsThreads)
    logits_sample_kernel(const T *__restrict__ Y, int64_t B, int64_t V,
                         const float *__restrict__ temps, float temp_scalar, uint64_t seed,
                         uint64_t offset, uint32_t flags, float *__restrict__ cand_score,
                         int32_t *__restrict__ cand_idx, int chunk_len, bool vec_ok) {
    __shared__ float red_s[kLogitsThreads / 32];
    __shared__ uint32_t red_i[kLogitsThreads / 32];
    const int chunk = blockIdx.x;
    const bool no_noise = (flags & 1u) != 0;
    for (int64_t b = blockIdx.y; b < B; b += gridDim.y) {
        const float Tb = temps ? temps[b] : temp_scalar;
        const bool t_ok = temperature_ok(Tb);
        const float invT = __frcp_rn(Tb);
        const int64_t v_begin = static_cast<int64_t>(chunk) * chunk_len;
        const int64_t v_end = min(V, v_begin + chunk_len);
        const T *row = Y + b * V;
        const PhiloxRow prow = philox_row(seed, offset, static_cast<uint64_t>(b));
        float best = -INFINITY;
        uint32_t bi = 0xFFFFFFFFu;
        if (t_ok) {
            for (int64_t v = v_begin + threadIdx.x * 8; v < v_end; v += kLogitsStep) {
                float l[8];
                load8<T>(row, v, v_end, vec_ok, l);
                if (no_noise) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float s = __fmul_rn(l[e], invT);
                        if (v + e < v_end && s > best) {
                            best = s;
                            bi = static_cast<uint32_t>(v + e);
                        }
                    }
                    continue;
                }
                uint32_t x[8];
                noise_words8(prow, static_cast<uint64_t>(v) >> 3, x);
                float lt[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) lt[e] = __fmul_rn(l[e], invT);
                // the thread's first element (v < v_end here) is scored
                // exactly; the others are screened against the best so far
                int first = 0;
                if (best == -INFINITY) {
                    const float s0 = __fadd_rn(lt[0], gumbel_from_word(x[0]));
                    if (s0 > best) {
                        best = s0;
                        bi = static_cast<uint32_t>(v);
                    }
                    first = 1;
                }
                const float best0 = best;
                uint32_t pass = 0;
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (e >= first && v + e < v_end &&
                        screen_lg2_tail(x[e]) < screen_bound(lt[e], best0))
                        pass |= 1u << e;
                while (pass) {
                    const int e = __ffs(pass) - 1;
                    pass &= pass - 1;
                    float lte = lt[0];
                    uint32_t xe = x[0];
#pragma unroll
                    for (int k = 1; k < 8; ++k) {
                        lte = (e == k) ? lt[k] : lte;
                        xe = (e == k) ? x[k] : xe;
                    }
                    const float s = __fadd_rn(lte, gumbel_from_word(xe));
                    if (s > best) {
                        best = s;
                        bi = static_cast<uint32_t>(v + e);
                    }
                }
            }
        }
        warp_argmax(best, bi);
        const int w = threadIdx.x >> 5;
        if ((threadIdx.x & 31) == 0) {
            red_s[w] = best;
            red_i[w] = bi;
        }
        __syncthreads();
        if (w == 0) {
            best = (threadIdx.x < kLogitsThreads / 32) ? red_s[threadIdx.x] : -INFINITY;
            bi = (threadIdx.x < kLogitsThreads / 32) ? red_i[threadIdx.x] : 0xFFFFFFFFu;
            warp_argmax(best, bi);
            if (threadIdx.x == 0) {
                cand_score[static_cast<int64_t>(chunk) * B + b] = best;
                cand_idx[static_cast<int64_t>(chunk) * B + b] = static_cast<int32_t>(bi);
            }
        }
        __syncthreads();
    }
}

cudaError_t launch_logits_sample(const void *Y, int y_dtype, int64_t B, int64_t V,
                                 const float *temps, float temp_scalar, uint64_t seed,
                                 uint64_t offset, uint32_t flags, float *cand_score,
                                 int32_t *cand_idx, int nChunks, int chunk,
                                 cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>(nChunks), static_cast<unsigned>(B < 65535 ? B : 65535));
    const uintptr_t base = reinterpret_cast<uintptr_t>(Y);
    if (y_dtype == 1) {
        const bool vec_ok = (base % 16 == 0) && (V % 4 == 0);
        logits_sample_kernel<float><<<grid, kLogitsThreads, 0, stream>>>(
            static_cast<const float *>(Y), B, V, temps, temp_scalar, seed, offset, flags,
            cand_score, cand_idx, chunk, vec_ok);
    } else {
        const bool vec_ok = (base % 16 == 0) && (V % 8 == 0);
        logits_sample_kernel<__nv_bfloat16><<<grid, kLogitsThreads, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(Y), B, V, temps, temp_scalar, seed, offset, flags,
            cand_score, cand_idx, chunk, vec_ok);
    }
    return cudaGetLastError();
}

// ------------------------------------------------------------------ debug gumbel
__global__ void debug_gumbel_kernel(const uint32_t *__restrict__ words, int64_t n,
                                    float *__restrict__ out_g) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        out_g[i] = gumbel_from_word(words[i]);
}

cudaError_t launch_debug_gumbel(const uint32_t *words, int64_t n, float *out_g,
                                cudaStream_t stream) {
    int64_t blocks = (n + 255) / 256;
    if (blocks > 65535) blocks = 65535;
    if (blocks < 1) blocks = 1;
    debug_gumbel_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(words, n, out_g);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ debug noise
__global__ void debug_noise_kernel(uint64_t seed, uint64_t offset, int64_t b0, int64_t nb,
                                   int64_t V, uint32_t *__restrict__ out_words,
                                   float *__restrict__ out_g) {
    const int64_t groups = (V + 7) / 8;
    const int64_t total = nb * groups;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t rb = i / groups;
        const int64_t v8 = i % groups;
        uint32_t x[8];
        noise_words8(philox_row(seed, offset, static_cast<uint64_t>(b0 + rb)),
                     static_cast<uint64_t>(v8), x);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int64_t v = v8 * 8 + e;
            if (v < V) {
                if (out_words) out_words[rb * V + v] = x[e];
                if (out_g) out_g[rb * V + v] = gumbel_from_word(x[e]);
            }
        }
    }
}

cudaError_t launch_debug_noise(uint64_t seed, uint64_t offset, int64_t b0, int64_t nb,
                               int64_t V, uint32_t *out_words, float *out_g,
                               cudaStream_t stream) {
    const int64_t total = nb * ((V + 7) / 8);
    int64_t blocks = (total + 255) / 256;
    if (blocks > 65535) blocks = 65535;
    if (blocks < 1) blocks = 1;
    debug_noise_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(seed, offset, b0, nb, V,
                                                                          out_words, out_g);
    return cudaGetLastError();
}

}  // namespace fs

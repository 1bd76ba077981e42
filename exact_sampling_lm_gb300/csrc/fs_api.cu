// fs_api.cu -- host side of the C ABI declared in include/fs_sample.h:
// argument validation, the Stage 1 schedule, TMA tensor-map encoding, the
// cached workspace of fs_sample, and the launches.  All compute runs in the
// kernels of fs_stage1.cu and fs_small.cu; nothing here computes on the host.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>

#include <map>
#include <mutex>
#include <string>
#include <utility>

#include "../../include/fs_sample.h"
#include "fs_internal.h"

namespace fs {

// ------------------------------------------------------------------ errors
static thread_local std::string t_last_error = "no error";

static fs_status fail(fs_status st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return st;
}

// Records the thread-local error text for entry points defined in other
// translation units.
fs_status set_error(fs_status st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return st;
}

static fs_status cuda_fail(cudaError_t e, const char *what) {
    return fail(FS_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// ------------------------------------------------------------------ schedule
// Stage 1 schedule.  nM batch tiles of 128 rows; the vocabulary is cut into P
// contiguous partitions, balanced in 16-row units, with P * nM <= SM count so
// that each CTA streams a 1/P share of W once.  CTA c takes batch tile c % nM
// and partition c / nM: the nM CTAs that share a partition run side by side
// and read the same W tiles, so W comes from HBM about once.
constexpr int kWorkspaceRegions = 5;

bool make_plan(int64_t B, int64_t V, int64_t D, int num_sms, Plan *p) {
    if (B < 1 || V < 1 || D < 1 || num_sms < 1) return false;
    p->B = B;
    p->V = V;
    p->D = D;
    const int64_t nM = (B + kBM - 1) / kBM;
    const int64_t U = (V + kUnitRows - 1) / kUnitRows;
    int64_t P = num_sms / nM;
    if (P < 1) P = 1;
    if (P > U) P = U;
    p->nM = static_cast<int>(nM);
    p->U = U;
    p->P = static_cast<int>(P);
    p->G = static_cast<int>(P * nM);
    p->nCand = static_cast<int>(P);
    // Tiles of the largest partition: balanced tiles of at most 256 rows, then
    // a final 128-row tile (a partition of at most 256 rows is one tile); CTAs
    // paired in clusters (an even nM) use plain 256-row tiles.
    const int64_t max_units = (U + P - 1) / P;
    const int64_t main_units = max_units - kFinalTileUnits;
    if (nM % 2 == 0)
        p->maxTiles = static_cast<int>((max_units * kUnitRows + kBN - 1) / kBN);
    else
        p->maxTiles = max_units <= kBN / kUnitRows
                          ? 1
                          : static_cast<int>((main_units + kBN / kUnitRows - 1) / (kBN / kUnitRows) + 1);
    // materialised-logits sampler: about 4 blocks per SM over all B x V
    // entries, each block a chunk of 2 K .. 64 K entries of one row
    {
        const int64_t want = (B * V) / (4 * static_cast<int64_t>(num_sms));
        int64_t chunk = (want + kLogitsStep - 1) / kLogitsStep * kLogitsStep;
        const int64_t vmax = (V + kLogitsStep - 1) / kLogitsStep * kLogitsStep;
        if (chunk > kLogitsMaxChunk) chunk = kLogitsMaxChunk;
        if (chunk > vmax) chunk = vmax;
        if (chunk < kLogitsStep) chunk = kLogitsStep;
        p->logitsChunk = static_cast<int>(chunk);
        p->nChunks = static_cast<int>((V + chunk - 1) / chunk);
    }
    auto region = [&](int64_t slots) { return ((slots * B * 4) + 255) / 256 * 256; };
    const int64_t slots = p->nCand > p->nChunks ? p->nCand : p->nChunks;
    p->wsBytes = static_cast<size_t>(kWorkspaceRegions * region(slots));
    p->wsSampleBytes = static_cast<size_t>(2 * region(p->nCand));
    p->wsLogprobBytes = static_cast<size_t>(kWorkspaceRegions * region(p->nCand));
    p->wsLogitsBytes = static_cast<size_t>(2 * region(p->nChunks));
    return true;
}

// Candidate buffers inside a workspace, each [slots][B] of 4-byte values:
// score, index, and (log-probability calls only) the winner's l~ and the
// log-mass pair (max, sum).  slots: p.nCand for the fused calls, p.nChunks
// for the materialised-logits sampler.
struct Candidates {
    float *score;
    int32_t *idx;
    float *lt, *m, *s;
};

static Candidates split_workspace(const Plan &p, void *ws, int64_t slots) {
    const int64_t region = ((slots * p.B * 4) + 255) / 256 * 256;
    char *base = static_cast<char *>(ws);
    Candidates c;
    c.score = reinterpret_cast<float *>(base);
    c.idx = reinterpret_cast<int32_t *>(base + region);
    c.lt = reinterpret_cast<float *>(base + 2 * region);
    c.m = reinterpret_cast<float *>(base + 3 * region);
    c.s = reinterpret_cast<float *>(base + 4 * region);
    return c;
}

// ------------------------------------------------------------------ device info
struct DeviceInfo {
    bool known = false;
    int sms = 0;
    int major = 0, minor = 0;
};
static std::mutex g_dev_mu;
static DeviceInfo g_dev[64];

static fs_status device_info(int *dev_out, DeviceInfo *info) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(FS_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.known) {
        if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
        if ((e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute(major)");
        if ((e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute(minor)");
        d.known = true;
    }
    if (d.major != 10 || d.minor != 3)
        return fail(FS_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                    dev, d.major, d.minor);
    *dev_out = dev;
    *info = d;
    return FS_OK;
}

// ------------------------------------------------------------------ tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

bool current_context_id(unsigned long long *id) {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
        cudaGetLastError();
    });
    if (!get_current || !get_id) return false;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

// Row-major bf16 matrix [rows, cols] read in boxes of 64 columns x box_rows
// rows, 128-byte swizzled in shared memory; out-of-range elements read as 0.
// A tensor map depends only on (address, shape, box), and a decode loop keeps
// passing the same few buffers, so each host thread keeps its most recent
// encodings and copies a match instead of calling the driver again.
struct TmapEntry {
    const void *base = nullptr;
    int64_t rows = 0, cols = 0;
    uint32_t box_rows = 0;
    CUtensorMap map;
};
constexpr int kTmapCacheSize = 16;
static thread_local TmapEntry t_tmap_cache[kTmapCacheSize];
static thread_local int t_tmap_next = 0;

static fs_status make_tmap(CUtensorMap *map, const void *base, int64_t rows, int64_t cols,
                           uint32_t box_rows) {
    for (int i = 0; i < kTmapCacheSize; ++i) {
        const TmapEntry &e = t_tmap_cache[i];
        if (e.base == base && e.base != nullptr && e.rows == rows && e.cols == cols &&
            e.box_rows == box_rows) {
            *map = e.map;
            return FS_OK;
        }
    }
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(FS_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(FS_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for [%lld x %lld] box %u",
                    static_cast<int>(r), static_cast<long long>(rows),
                    static_cast<long long>(cols), box_rows);
    TmapEntry &e = t_tmap_cache[t_tmap_next];
    t_tmap_next = (t_tmap_next + 1) % kTmapCacheSize;
    e.base = base;
    e.rows = rows;
    e.cols = cols;
    e.box_rows = box_rows;
    e.map = *map;
    return FS_OK;
}

// ------------------------------------------------------------------ validation
static bool temperature_ok(float T) { return isfinite(T) && T > 0.0f; }

static fs_status validate_shape(int64_t B, int64_t V, int64_t D) {
    if (B < 1 || V < 1 || D < 1)
        return fail(FS_ERR_INVALID_ARG, "B, V and D must be >= 1 (got %lld, %lld, %lld)",
                    static_cast<long long>(B), static_cast<long long>(V),
                    static_cast<long long>(D));
    if (V > FS_MAX_VOCAB) return fail(FS_ERR_UNSUPPORTED, "V=%lld exceeds 2^31-1", static_cast<long long>(V));
    if (B > FS_MAX_BATCH) return fail(FS_ERR_UNSUPPORTED, "B=%lld exceeds 2^24", static_cast<long long>(B));
    if (D % 8 != 0)
        return fail(FS_ERR_UNSUPPORTED, "D=%lld must be a multiple of 8 (16-byte rows)",
                    static_cast<long long>(D));
    if (D > (1 << 20)) return fail(FS_ERR_UNSUPPORTED, "D=%lld exceeds 2^20", static_cast<long long>(D));
    return FS_OK;
}

static fs_status validate_gemm_inputs(const void *H, const void *W, int64_t B, int64_t V,
                                      int64_t D) {
    if (!H || !W) return fail(FS_ERR_INVALID_ARG, "H and W must be non-null device pointers");
    fs_status st = validate_shape(B, V, D);
    if (st != FS_OK) return st;
    if (reinterpret_cast<uintptr_t>(H) % 16 || reinterpret_cast<uintptr_t>(W) % 16)
        return fail(FS_ERR_UNSUPPORTED, "H and W must be 16-byte aligned");
    return FS_OK;
}

// Device outputs must be aligned to their element size (a misaligned store
// would fault inside the kernel instead of failing here).
static fs_status validate_out(const void *p, size_t align, const char *name) {
    if (p && reinterpret_cast<uintptr_t>(p) % align)
        return fail(FS_ERR_UNSUPPORTED, "%s must be %zu-byte aligned", name, align);
    return FS_OK;
}

static fs_status validate_outputs(const int64_t *out_idx, const float *out_score,
                                  const float *temperatures) {
    fs_status st;
    if ((st = validate_out(out_idx, 8, "out_idx")) != FS_OK) return st;
    if ((st = validate_out(out_score, 4, "out_score")) != FS_OK) return st;
    return validate_out(temperatures, 4, "temperatures");
}

static fs_status validate_temperature(float temperature, const float *temperatures) {
    if (!temperatures && !temperature_ok(temperature))
        return fail(FS_ERR_INVALID_ARG,
                    "temperature must be finite and > 0 (got %g); greedy decoding is not "
                    "supported",
                    static_cast<double>(temperature));
    return FS_OK;
}

// need: p.wsSampleBytes for the calls that keep only (score, index)
// candidates, p.wsBytes for the ones that also keep log-masses.
static fs_status validate_workspace(const void *ws, size_t bytes, size_t need) {
    if (!ws) return fail(FS_ERR_INVALID_ARG, "workspace must be non-null");
    if (reinterpret_cast<uintptr_t>(ws) % 16)
        return fail(FS_ERR_UNSUPPORTED, "workspace must be 16-byte aligned");
    if (bytes < need)
        return fail(FS_ERR_NO_MEMORY, "workspace of %zu bytes is smaller than the %zu needed",
                    bytes, need);
    return FS_OK;
}

static const char *memory_type_name(cudaMemoryType t) {
    switch (t) {
        case cudaMemoryTypeHost: return "page-locked host memory";
        case cudaMemoryTypeDevice: return "device memory";
        case cudaMemoryTypeManaged: return "managed memory";
        default: return "memory the CUDA runtime does not know";
    }
}

// The TMA tensor maps of Stage 1 are encoded on the caller's H and W, and in
// the paired forms the two CTAs of a cluster either multicast W boxes to
// each other or feed one MMA from both CTAs' shared memory, their loads
// completing on one CTA's barrier.  Those loads
// must read this GPU's own memory: not host memory reached through a
// mapping, not another GPU's memory reached through peer access, not managed
// memory that may migrate.  Anything else is refused before a launch.
static fs_status require_local_device_memory(const void *p, const char *name) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    cudaPointerAttributes a;
    e = cudaPointerGetAttributes(&a, p);
    if (e != cudaSuccess) {
        cudaGetLastError();  // an unknown pointer leaves no sticky error
        return fail(FS_ERR_UNSUPPORTED, "%s is not memory the CUDA runtime knows (%s)", name,
                    cudaGetErrorString(e));
    }
    if (a.type != cudaMemoryTypeDevice)
        return fail(FS_ERR_UNSUPPORTED,
                    "%s must be device memory of the current GPU; it is %s", name,
                    memory_type_name(a.type));
    if (a.device != dev)
        return fail(FS_ERR_UNSUPPORTED,
                    "%s is memory of GPU %d, but the current GPU is %d: Stage 1 reads its "
                    "operands from the calling GPU's own memory only",
                    name, a.device, dev);
    return FS_OK;
}

static uint64_t wait_timeout_ns() {
    static uint64_t ns = [] {
        const char *s = getenv("FS_WAIT_TIMEOUT_MS");
        const long long ms = s ? atoll(s) : 0;
        return ms > 0 ? static_cast<uint64_t>(ms) * 1000000ull : 4000000000ull;
    }();
    return ns;
}

// ------------------------------------------------------------------ Stage 1 launch
static fs_status run_stage1(int mode, const void *H, const void *W, const Plan &p,
                            float temperature, const float *temperatures, uint64_t seed,
                            uint64_t offset, uint32_t flags, float *out_logits, void *out_y,
                            int y_dtype, const Candidates *cand, cudaStream_t stream,
                            const fs_transforms *tf = nullptr, int64_t vocab_offset = 0) {
    CUtensorMap tmH;
    WMaps wm;
    fs_status st;
    if ((st = require_local_device_memory(H, "H")) != FS_OK) return st;
    if ((st = require_local_device_memory(W, "W")) != FS_OK) return st;
    // With one batch tile, load only the live rows of H (rounded up to the
    // 8-row swizzle atom); the MMA's other A rows feed TMEM lanes that the
    // epilogue never reads.
    const int h_box_rows = p.nM == 1 ? static_cast<int>((p.B + 7) / 8 * 8) : kBM;
    if ((st = make_tmap(&tmH, H, p.B, p.D, static_cast<uint32_t>(h_box_rows))) != FS_OK) return st;
    if ((st = make_tmap(&wm.w16, W, p.V, p.D, 16)) != FS_OK) return st;
    if ((st = make_tmap(&wm.w64, W, p.V, p.D, 64)) != FS_OK) return st;
    if ((st = make_tmap(&wm.w128, W, p.V, p.D, 128)) != FS_OK) return st;
    if ((st = make_tmap(&wm.w256, W, p.V, p.D, 256)) != FS_OK) return st;
    Stage1Args a;
    a.B = static_cast<int32_t>(p.B);
    a.V = static_cast<int32_t>(p.V);
    a.D = static_cast<int32_t>(p.D);
    a.nM = p.nM;
    a.P = p.P;
    a.U = p.U;
    a.temps = temperatures;
    a.temp_scalar = temperature;
    a.seed = seed;
    a.offset = offset;
    a.flags = flags;
    a.cand_score = cand ? cand->score : nullptr;
    a.cand_idx = cand ? cand->idx : nullptr;
    a.cand_lt = cand ? cand->lt : nullptr;
    a.cand_m = cand ? cand->m : nullptr;
    a.cand_s = cand ? cand->s : nullptr;
    a.out_logits = out_logits;
    a.out_y = out_y;
    const void *dst = out_logits ? static_cast<const void *>(out_logits) : out_y;
    const bool f32 = (mode == kModeSampleStore) || (mode == kModeGemmF32 && y_dtype == FS_DTYPE_F32);
    a.y_vec_ok = dst && (reinterpret_cast<uintptr_t>(dst) % 16 == 0) &&
                 (f32 ? (p.V % 4 == 0) : (p.V % 8 == 0));
    a.h_box_rows = h_box_rows;
    a.vocab_offset = vocab_offset;
    a.bias = tf ? tf->bias : nullptr;
    a.softcap = tf ? tf->softcap : 0.0f;
    a.allow_mask = tf ? tf->allow_mask : nullptr;
    a.mask_words = tf ? tf->mask_words : 0;
    a.timeout_ns = wait_timeout_ns();
    cudaError_t e = launch_stage1(mode, tmH, wm, a, p.G, stream);
    if (e != cudaSuccess) return cuda_fail(e, "Stage 1 launch");
    return FS_OK;
}

// ------------------------------------------------------------------ workspace cache
struct CachedWs {
    void *ptr = nullptr;
    size_t bytes = 0;
};
static std::mutex g_ws_mu;
static std::map<std::pair<int, void *>, CachedWs> g_ws;

// True while `stream` is being captured into a CUDA graph.  Device memory
// allocated then would belong to the graph, so the caches below never grow
// during a capture.
static bool stream_capturing(cudaStream_t stream) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return cap != cudaStreamCaptureStatusNone;
}

static fs_status cached_workspace(int dev, cudaStream_t stream, size_t need, void **out) {
    std::lock_guard<std::mutex> lock(g_ws_mu);
    CachedWs &c = g_ws[std::make_pair(dev, static_cast<void *>(stream))];
    if (c.bytes < need) {
        if (stream_capturing(stream))
            return fail(FS_ERR_UNSUPPORTED,
                        "the cached workspace of this stream (%zu bytes) cannot grow to %zu "
                        "during stream capture: make one call of the same size on this stream "
                        "before capturing, or pass a workspace to fs_sample_ex",
                        c.bytes, need);
        size_t grow = 65536;
        while (grow < need) grow <<= 1;
        if (c.ptr) {
            cudaError_t e = cudaFreeAsync(c.ptr, stream);
            c.ptr = nullptr;
            c.bytes = 0;
            if (e != cudaSuccess) return cuda_fail(e, "cudaFreeAsync(workspace)");
        }
        cudaError_t e = cudaMallocAsync(&c.ptr, grow, stream);
        if (e != cudaSuccess) {
            c.ptr = nullptr;
            return fail(FS_ERR_NO_MEMORY, "cudaMallocAsync(%zu) failed: %s", grow,
                        cudaGetErrorString(e));
        }
        c.bytes = grow;
    }
    *out = c.ptr;
    return FS_OK;
}

}  // namespace fs

using namespace fs;

// ====================================================================== C ABI
extern "C" {

const char *fs_version(void) { return "fs_sample 0.1.0 (sm_103a: TMA + tcgen05 + TMEM)"; }

const char *fs_last_error_string(void) { return t_last_error.c_str(); }

fs_status fs_plan_info(int64_t B, int64_t V, int64_t D, int num_sms, int64_t out[6]) {
    if (!out) return fail(FS_ERR_INVALID_ARG, "out must be non-null");
    fs_status st = validate_shape(B, V, D);
    if (st != FS_OK) return st;
    if (num_sms < 1) return fail(FS_ERR_INVALID_ARG, "num_sms must be >= 1");
    Plan p;
    make_plan(B, V, D, num_sms, &p);
    out[0] = p.nM;
    out[1] = p.P;
    out[2] = p.G;
    out[3] = p.nCand;
    out[4] = static_cast<int64_t>(p.wsBytes);
    out[5] = p.maxTiles;
    return FS_OK;
}

fs_status fs_stage1_form(int64_t B, int64_t V, int64_t D, int *out_form) {
    if (!out_form) return fail(FS_ERR_INVALID_ARG, "out_form must be non-null");
    fs_status st = validate_shape(B, V, D);
    if (st != FS_OK) return st;
    int dev = 0;
    DeviceInfo info;
    if ((st = device_info(&dev, &info)) != FS_OK) return st;
    Plan p;
    make_plan(B, V, D, info.sms, &p);
    *out_form = stage1_form(static_cast<int>(p.nM), static_cast<int>(D), static_cast<int>(p.G));
    return FS_OK;
}

}  // extern "C"

namespace fs {
size_t sample_workspace_bytes(int64_t B, int64_t V, int64_t D) {
    if (validate_shape(B, V, D) != FS_OK) return 0;
    int dev;
    DeviceInfo info;
    if (device_info(&dev, &info) != FS_OK) return 0;
    Plan p;
    make_plan(B, V, D, info.sms, &p);
    return p.wsSampleBytes;
}
}  // namespace fs

extern "C" {

size_t fs_workspace_size(int64_t B, int64_t V, int64_t D) {
    if (validate_shape(B, V, D) != FS_OK) return 0;
    int dev;
    DeviceInfo info;
    if (device_info(&dev, &info) != FS_OK) return 0;
    Plan p;
    make_plan(B, V, D, info.sms, &p);
    return p.wsBytes;
}

fs_status fs_stage1(const void *H, const void *W, int64_t B, int64_t V, int64_t D,
                    float temperature, const float *temperatures, uint64_t seed,
                    uint64_t offset, uint32_t flags, float *out_logits, void *workspace,
                    size_t ws_bytes, void *stream) {
    fs_status st;
    if ((st = validate_gemm_inputs(H, W, B, V, D)) != FS_OK) return st;
    if ((st = validate_temperature(temperature, temperatures)) != FS_OK) return st;
    if (flags & ~(FS_FLAG_NO_NOISE | FS_FLAG_STORE_LOGITS | FS_FLAG_TEST_NO_LOADS))
        return fail(FS_ERR_INVALID_ARG, "unknown flag bits 0x%x", flags);
    if ((flags & FS_FLAG_STORE_LOGITS) && !out_logits)
        return fail(FS_ERR_INVALID_ARG, "FS_FLAG_STORE_LOGITS needs out_logits");
    if ((st = validate_out(out_logits, 4, "out_logits")) != FS_OK) return st;
    if ((st = validate_out(temperatures, 4, "temperatures")) != FS_OK) return st;
    int dev;
    DeviceInfo info;
    if ((st = device_info(&dev, &info)) != FS_OK) return st;
    Plan p;
    make_plan(B, V, D, info.sms, &p);
    if ((st = validate_workspace(workspace, ws_bytes, p.wsSampleBytes)) != FS_OK) return st;
    const Candidates cand = split_workspace(p, workspace, p.nCand);
    const int mode = (flags & FS_FLAG_STORE_LOGITS) ? kModeSampleStore : kModeSample;
    return run_stage1(mode, H, W, p, temperature, temperatures, seed, offset, flags,
                      (flags & FS_FLAG_STORE_LOGITS) ? out_logits : nullptr, nullptr, 0, &cand,
                      static_cast<cudaStream_t>(stream));
}

fs_status fs_stage2(int64_t B, int64_t V, int64_t D, float temperature,
                    const float *temperatures, int64_t *out_idx, float *out_score,
                    const void *workspace, size_t ws_bytes, void *stream) {
    fs_status st;
    if ((st = validate_shape(B, V, D)) != FS_OK) return st;
    if ((st = validate_temperature(temperature, temperatures)) != FS_OK) return st;
    if (!out_idx) return fail(FS_ERR_INVALID_ARG, "out_idx must be non-null");
    if ((st = validate_outputs(out_idx, out_score, temperatures)) != FS_OK) return st;
    int dev;
    DeviceInfo info;
    if ((st = device_info(&dev, &info)) != FS_OK) return st;
    Plan p;
    make_plan(B, V, D, info.sms, &p);
    if ((st = validate_workspace(workspace, ws_bytes, p.wsSampleBytes)) != FS_OK) return st;
    const Candidates cand = split_workspace(p, const_cast<void *>(workspace), p.nCand);
    cudaError_t e = launch_stage2(cand.score, cand.idx, p.nCand, B, temperatures, temperature,
                                  out_idx, out_score, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "Stage 2 launch");
    return FS_OK;
}

fs_status fs_sample_ex(const void *H, const void *W, int64_t B, int64_t V, int64_t D,
                       float temperature, const float *temperatures, uint64_t seed,
                       uint64_t offset, uint32_t flags, int64_t *out_idx, float *out_score,
                       float *out_logits, void *workspace, size_t ws_bytes, void *stream) {
    if (!out_idx) return fail(FS_ERR_INVALID_ARG, "out_idx must be non-null");
    // Stage 2's own arguments are checked before Stage 1 launches, so that a
    // bad output pointer launches nothing.
    fs_status st = validate_outputs(out_idx, out_score, temperatures);
    if (st != FS_OK) return st;
    st = fs_stage1(H, W, B, V, D, temperature, temperatures, seed, offset, flags, out_logits,
                   workspace, ws_bytes, stream);
    if (st != FS_OK) return st;
    return fs_stage2(B, V, D, temperature, temperatures, out_idx, out_score, workspace, ws_bytes,
                     stream);
}

fs_status fs_sample(const void *H, const void *W, int64_t B, int64_t V, int64_t D,
                    float temperature, const float *temperatures, uint64_t seed,
                    uint64_t offset, int64_t *out_idx, float *out_score, void *stream) {
    fs_status st;
    if ((st = validate_gemm_inputs(H, W, B, V, D)) != FS_OK) return st;
    if ((st = validate_temperature(temperature, temperatures)) != FS_OK) return st;
    if (!out_idx) return fail(FS_ERR_INVALID_ARG, "out_idx must be non-null");
    if ((st = validate_outputs(out_idx, out_score, temperatures)) != FS_OK) return st;
    int dev;
    DeviceInfo info;
    if ((st = device_info(&dev, &info)) != FS_OK) return st;
    Plan p;
    make_plan(B, V, D, info.sms, &p);
    void *ws = nullptr;
    if ((st = cached_workspace(dev, static_cast<cudaStream_t>(stream), p.wsBytes, &ws)) != FS_OK)
        return st;
    return fs_sample_ex(H, W, B, V, D, temperature, temperatures, seed, offset, 0, out_idx,
                        out_score, nullptr, ws, p.wsBytes, stream);
}

static size_t round256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

// The device address of a page-locked host buffer, or nullptr when the buffer
// is pageable (or not host memory at all).
static void *mapped_host_alias(void *p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();  // an unknown pointer is not an error here
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// Per (device, stream) state of fs_sample_host: an internal upload stream,
// two H / temperature slots used alternately, events that order a slot's
// upload after the previous reader of that slot, and output staging for
// pageable host outputs.
struct HostPath {
    std::mutex mu;  // serialises calls on this (device, stream)
    cudaStream_t copy = nullptr;
    cudaEvent_t uploaded[2] = {nullptr, nullptr};
    cudaEvent_t consumed[2] = {nullptr, nullptr};
    cudaEvent_t all_prior = nullptr;      // everything queued on the caller's stream so far
    bool kernel_upload[2] = {false, false};  // slot last filled by the upload kernel
    int next = 0;
    char *block = nullptr;
    size_t bytes = 0;
};
static std::mutex g_host_mu;
static std::map<std::pair<int, void *>, HostPath> g_host;

static fs_status host_path_ready(HostPath &h, size_t need, bool capturing) {
    cudaError_t e;
    if (capturing && (!h.copy || h.bytes < need))
        return fail(FS_ERR_UNSUPPORTED,
                    "fs_sample_host cannot set up or grow its device staging during stream "
                    "capture: make one call of the same size on this stream before capturing");
    if (!h.copy) {
        if ((e = cudaStreamCreateWithFlags(&h.copy, cudaStreamNonBlocking)) != cudaSuccess)
            return cuda_fail(e, "cudaStreamCreate(upload stream)");
        for (int j = 0; j < 2; ++j) {
            if ((e = cudaEventCreateWithFlags(&h.uploaded[j], cudaEventDisableTiming)) !=
                    cudaSuccess ||
                (e = cudaEventCreateWithFlags(&h.consumed[j], cudaEventDisableTiming)) !=
                    cudaSuccess)
                return cuda_fail(e, "cudaEventCreate(upload events)");
        }
        if ((e = cudaEventCreateWithFlags(&h.all_prior, cudaEventDisableTiming)) != cudaSuccess)
            return cuda_fail(e, "cudaEventCreate(upload events)");
    }
    if (h.bytes < need) {
        // cudaFree waits for all work on the device, including reads of the
        // old block still queued on either stream.
        if (h.block && (e = cudaFree(h.block)) != cudaSuccess)
            return cuda_fail(e, "cudaFree(host-path staging)");
        h.block = nullptr;
        h.bytes = 0;
        size_t grow = 65536;
        while (grow < need) grow <<= 1;
        if (cudaMalloc(reinterpret_cast<void **>(&h.block), grow) != cudaSuccess) {
            cudaGetLastError();
            h.block = nullptr;
            return fail(FS_ERR_NO_MEMORY, "cudaMalloc(%zu) for host-path staging failed", grow);
        }
        h.bytes = grow;
    }
    return FS_OK;
}

fs_status fs_sample_host(const void *H_host, const void *W, int64_t B, int64_t V, int64_t D,
                         float temperature, const float *temperatures_host, uint64_t seed,
                         uint64_t offset, int64_t *out_idx_host, float *out_score_host,
                         void *stream) {
    fs_status st;
    if (!H_host || !W) return fail(FS_ERR_INVALID_ARG, "H_host and W must be non-null");
    if ((st = validate_shape(B, V, D)) != FS_OK) return st;
    if (reinterpret_cast<uintptr_t>(W) % 16)
        return fail(FS_ERR_UNSUPPORTED, "W must be 16-byte aligned");
    if ((st = validate_temperature(temperature, temperatures_host)) != FS_OK) return st;
    if (!out_idx_host) return fail(FS_ERR_INVALID_ARG, "out_idx_host must be non-null");
    int dev;
    DeviceInfo info;
    if ((st = device_info(&dev, &info)) != FS_OK) return st;
    // W is checked before the upload of H launches (H's device slot is the
    // library's own memory).
    if ((st = require_local_device_memory(W, "W")) != FS_OK) return st;
    Plan p;
    make_plan(B, V, D, info.sms, &p);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *ws = nullptr;
    if ((st = cached_workspace(dev, s, p.wsBytes, &ws)) != FS_OK) return st;

    // Outputs: page-locked host buffers are written by Stage 2 directly;
    // pageable ones go through device staging and a copy back.
    int64_t *idx_dev = static_cast<int64_t *>(mapped_host_alias(out_idx_host));
    float *score_dev = out_score_host ? static_cast<float *>(mapped_host_alias(out_score_host))
                                      : nullptr;
    const bool stage_idx = !idx_dev;
    const bool stage_score = out_score_host && !score_dev;

    const size_t ub = static_cast<size_t>(B);
    const size_t h_bytes = ub * static_cast<size_t>(D) * 2;
    const size_t h_b = round256(h_bytes);
    const size_t t_b = temperatures_host ? round256(ub * 4) : 0;
    const size_t i_b = round256(ub * 8);
    const size_t s_b = round256(ub * 4);

    // Page-locked inputs are uploaded by a kernel on the caller's stream
    // (upload_kernel): launched with programmatic serialization, it keeps the
    // chain of back-to-back calls overlapping.  Pageable inputs are copied by
    // the CUDA runtime: under stream capture on the caller's stream (a graph
    // cannot wait on events recorded outside it), otherwise on the internal
    // upload stream, overlapping the previous call's kernels.
    const void *H_src = mapped_host_alias(const_cast<void *>(H_host));
    const void *T_src =
        temperatures_host ? mapped_host_alias(const_cast<float *>(temperatures_host)) : nullptr;
    const bool by_kernel = H_src != nullptr && reinterpret_cast<uintptr_t>(H_src) % 16 == 0 &&
                           (!temperatures_host ||
                            (T_src != nullptr && reinterpret_cast<uintptr_t>(T_src) % 4 == 0));
    const bool capturing = stream_capturing(s);
    const bool overlap = !by_kernel && !capturing;

    HostPath *hp;
    {
        // std::map never moves its nodes: the entry outlives this lookup.
        std::lock_guard<std::mutex> map_lock(g_host_mu);
        hp = &g_host[std::make_pair(dev, static_cast<void *>(s))];
    }
    HostPath &h = *hp;
    std::lock_guard<std::mutex> lock(h.mu);
    if ((st = host_path_ready(h, 2 * (h_b + t_b) + i_b + s_b, capturing)) != FS_OK) return st;
    cudaError_t e;
    const int j = h.next;
    h.next ^= 1;
    char *slot = h.block + j * (h_b + t_b);
    void *H = slot;
    float *T = temperatures_host ? reinterpret_cast<float *>(slot + h_b) : nullptr;
    if (stage_idx) idx_dev = reinterpret_cast<int64_t *>(h.block + 2 * (h_b + t_b));
    if (stage_score) score_dev = reinterpret_cast<float *>(h.block + 2 * (h_b + t_b) + i_b);

    if (by_kernel) {
        // Slot j was last read by the Stage 1 two calls back.  This kernel can
        // start only once the previous call's Stage 2 has started, i.e. once
        // every CTA of the previous Stage 1 has triggered its dependents --
        // after its last load and after its own wait for the Stage 1 before.
        if ((e = launch_upload(H_src, H, static_cast<int64_t>(h_bytes),
                               static_cast<const float *>(T_src), T, T ? B : 0, s)) !=
            cudaSuccess)
            return cuda_fail(e, "upload kernel launch");
        h.kernel_upload[j] = true;
    } else {
        cudaStream_t up = overlap ? h.copy : s;
        if (overlap) {
            // A slot last filled by the upload kernel recorded no release
            // event: wait for everything queued so far instead.
            cudaEvent_t ready = h.consumed[j];
            if (h.kernel_upload[j]) {
                if ((e = cudaEventRecord(h.all_prior, s)) != cudaSuccess)
                    return cuda_fail(e, "upload ordering");
                ready = h.all_prior;
            }
            if ((e = cudaStreamWaitEvent(up, ready, 0)) != cudaSuccess)
                return cuda_fail(e, "upload stream wait");
        }
        if ((e = cudaMemcpyAsync(H, H_host, h_bytes, cudaMemcpyDefault, up)) != cudaSuccess)
            return cuda_fail(e, "upload of H");
        if (T && (e = cudaMemcpyAsync(T, temperatures_host, ub * 4, cudaMemcpyDefault, up)) !=
                     cudaSuccess)
            return cuda_fail(e, "upload of the temperatures");
        if (overlap) {
            if ((e = cudaEventRecord(h.uploaded[j], up)) != cudaSuccess ||
                (e = cudaStreamWaitEvent(s, h.uploaded[j], 0)) != cudaSuccess)
                return cuda_fail(e, "upload ordering");
        }
        h.kernel_upload[j] = false;
    }
    if ((st = fs_sample_ex(H, W, B, V, D, temperature, T, seed, offset, 0, idx_dev, score_dev,
                           nullptr, ws, p.wsBytes, stream)) != FS_OK)
        return st;
    if (overlap && (e = cudaEventRecord(h.consumed[j], s)) != cudaSuccess)
        return cuda_fail(e, "slot release");
    if (stage_idx &&
        (e = cudaMemcpyAsync(out_idx_host, idx_dev, ub * 8, cudaMemcpyDefault, s)) != cudaSuccess)
        return cuda_fail(e, "read-back of out_idx");
    if (stage_score && (e = cudaMemcpyAsync(out_score_host, score_dev, ub * 4,
                                            cudaMemcpyDefault, s)) != cudaSuccess)
        return cuda_fail(e, "read-back of out_score");
    return FS_OK;
}

fs_status fs_sample_logprob(const void *H, const void *W, int64_t B, int64_t V, int64_t D,
                            float temperature, const float *temperatures, uint64_t seed,
                            uint64_t offset, int64_t *out_idx, float *out_score,
                            float *out_logprob, void *workspace, size_t ws_bytes,
                            void *stream) {
    fs_status st;
    if ((st = validate_gemm_inputs(H, W, B, V, D)) != FS_OK) return st;
    if ((st = validate_temperature(temperature, temperatures)) != FS_OK) return st;
    if (!out_idx || !out_logprob)
        return fail(FS_ERR_INVALID_ARG, "out_idx and out_logprob must be non-null");
    if ((st = validate_outputs(out_idx, out_score, temperatures)) != FS_OK) return st;
    if ((st = validate_out(out_logprob, 4, "out_logprob")) != FS_OK) return st;
    int dev;
    DeviceInfo info;
    if ((st = device_info(&dev, &info)) != FS_OK) return st;
    Plan p;
    make_plan(B, V, D, info.sms, &p);
    if ((st = validate_workspace(workspace, ws_bytes, p.wsLogprobBytes)) != FS_OK) return st;
    const Candidates cand = split_workspace(p, workspace, p.nCand);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((st = run_stage1(kModeSampleLogprob, H, W, p, temperature, temperatures, seed, offset, 0,
                         nullptr, nullptr, 0, &cand, s)) != FS_OK)
        return st;
    cudaError_t e = launch_stage2_logprob(cand.score, cand.idx, cand.lt, cand.m, cand.s, p.nCand,
                                          B, temperatures, temperature, out_idx, out_score,
                                          out_logprob, s);
    if (e != cudaSuccess) return cuda_fail(e, "Stage 2 (log-probability) launch");
    return FS_OK;
}

fs_status fs_sample_transformed(const void *H, const void *W, int64_t B, int64_t V, int64_t D,
                                const fs_transforms *tf, float temperature,
                                const float *temperatures, uint64_t seed, uint64_t offset,
                                uint32_t flags, int64_t *out_idx, float *out_score,
                                float *out_logprob, void *workspace, size_t ws_bytes,
                                void *stream) {
    fs_status st;
    if ((st = validate_gemm_inputs(H, W, B, V, D)) != FS_OK) return st;
    if ((st = validate_temperature(temperature, temperatures)) != FS_OK) return st;
    if (!tf) return fail(FS_ERR_INVALID_ARG, "tf must be non-null (zero it for no transform)");
    if (!out_idx) return fail(FS_ERR_INVALID_ARG, "out_idx must be non-null");
    if ((st = validate_outputs(out_idx, out_score, temperatures)) != FS_OK) return st;
    if ((st = validate_out(out_logprob, 4, "out_logprob")) != FS_OK) return st;
    if (flags & ~FS_FLAG_NO_NOISE)
        return fail(FS_ERR_INVALID_ARG, "only FS_FLAG_NO_NOISE applies to fs_sample_transformed");
    if (!isfinite(tf->softcap) || tf->softcap < 0.0f)
        return fail(FS_ERR_INVALID_ARG, "softcap must be finite and >= 0 (got %g)",
                    static_cast<double>(tf->softcap));
    if (tf->bias && reinterpret_cast<uintptr_t>(tf->bias) % 16)
        return fail(FS_ERR_UNSUPPORTED, "bias must be 16-byte aligned");
    if (tf->allow_mask) {
        if (tf->mask_words < (V + 31) / 32)
            return fail(FS_ERR_INVALID_ARG, "mask_words=%lld < ceil(V/32)=%lld",
                        static_cast<long long>(tf->mask_words),
                        static_cast<long long>((V + 31) / 32));
        if (reinterpret_cast<uintptr_t>(tf->allow_mask) % 4)
            return fail(FS_ERR_UNSUPPORTED, "allow_mask must be 4-byte aligned");
    }
    int dev;
    DeviceInfo info;
    if ((st = device_info(&dev, &info)) != FS_OK) return st;
    Plan p;
    make_plan(B, V, D, info.sms, &p);
    if ((st = validate_workspace(workspace, ws_bytes, out_logprob ? p.wsLogprobBytes : p.wsSampleBytes)) !=
        FS_OK)
        return st;
    const Candidates cand = split_workspace(p, workspace, p.nCand);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int mode = out_logprob ? kModeSampleXformLogprob : kModeSampleXform;
    if ((st = run_stage1(mode, H, W, p, temperature, temperatures, seed, offset, flags, nullptr,
                         nullptr, 0, &cand, s, tf)) != FS_OK)
        return st;
    cudaError_t e;
    if (out_logprob)
        e = launch_stage2_logprob(cand.score, cand.idx, cand.lt, cand.m, cand.s, p.nCand, B,
                                  temperatures, temperature, out_idx, out_score, out_logprob, s);
    else
        e = launch_stage2(cand.score, cand.idx, p.nCand, B, temperatures, temperature, out_idx,
                          out_score, s);
    if (e != cudaSuccess) return cuda_fail(e, "Stage 2 launch");
    return FS_OK;
}

fs_status fs_sample_shard(const void *H, const void *W_shard, int64_t B, int64_t V_shard,
                          int64_t D, int64_t vocab_offset, float temperature,
                          const float *temperatures, uint64_t seed, uint64_t offset,
                          int64_t *out_idx, float *out_score, float *out_logmass,
                          void *workspace, size_t ws_bytes, void *stream) {
    fs_status st;
    if ((st = validate_gemm_inputs(H, W_shard, B, V_shard, D)) != FS_OK) return st;
    if ((st = validate_temperature(temperature, temperatures)) != FS_OK) return st;
    if (!out_idx || !out_logmass)
        return fail(FS_ERR_INVALID_ARG, "out_idx and out_logmass must be non-null");
    if ((st = validate_outputs(out_idx, out_score, temperatures)) != FS_OK) return st;
    if ((st = validate_out(out_logmass, 4, "out_logmass")) != FS_OK) return st;
    if (vocab_offset < 0 || vocab_offset % 16 != 0)
        return fail(FS_ERR_INVALID_ARG, "vocab_offset=%lld must be >= 0 and a multiple of 16",
                    static_cast<long long>(vocab_offset));
    if (vocab_offset + V_shard > FS_MAX_VOCAB)
        return fail(FS_ERR_UNSUPPORTED, "vocab_offset + V_shard exceeds 2^31-1");
    int dev;
    DeviceInfo info;
    if ((st = device_info(&dev, &info)) != FS_OK) return st;
    Plan p;
    make_plan(B, V_shard, D, info.sms, &p);
    if ((st = validate_workspace(workspace, ws_bytes, p.wsLogprobBytes)) != FS_OK) return st;
    const Candidates cand = split_workspace(p, workspace, p.nCand);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((st = run_stage1(kModeSampleLogprob, H, W_shard, p, temperature, temperatures, seed,
                         offset, 0, nullptr, nullptr, 0, &cand, s, nullptr, vocab_offset)) !=
        FS_OK)
        return st;
    cudaError_t e = launch_stage2_logprob(cand.score, cand.idx, cand.lt, cand.m, cand.s, p.nCand,
                                          B, temperatures, temperature, out_idx, out_score,
                                          nullptr, s, out_logmass);
    if (e != cudaSuccess) return cuda_fail(e, "Stage 2 (shard) launch");
    return FS_OK;
}

fs_status fs_combine_groups(int64_t n_groups, int64_t B, const int64_t *group_idx,
                            const float *group_logmass, uint64_t seed, uint64_t offset,
                            int64_t *out_idx, int64_t *out_group, void *stream) {
    if (n_groups < 1 || B < 1)
        return fail(FS_ERR_INVALID_ARG, "n_groups and B must be >= 1");
    if (B > FS_MAX_BATCH) return fail(FS_ERR_UNSUPPORTED, "B exceeds 2^24");
    if (!group_idx || !group_logmass || !out_idx)
        return fail(FS_ERR_INVALID_ARG, "group_idx, group_logmass and out_idx must be non-null");
    fs_status st0;
    if ((st0 = validate_out(group_idx, 8, "group_idx")) != FS_OK ||
        (st0 = validate_out(group_logmass, 4, "group_logmass")) != FS_OK ||
        (st0 = validate_out(out_idx, 8, "out_idx")) != FS_OK ||
        (st0 = validate_out(out_group, 8, "out_group")) != FS_OK)
        return st0;
    int dev;
    DeviceInfo info;
    fs_status st = device_info(&dev, &info);
    if (st != FS_OK) return st;
    cudaError_t e = launch_combine_groups(n_groups, B, group_idx, group_logmass, seed, offset,
                                          out_idx, out_group, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "group combine launch");
    return FS_OK;
}

fs_status fs_logits_gemm(const void *H, const void *W, int64_t B, int64_t V, int64_t D,
                         void *Y, int y_dtype, void *stream) {
    fs_status st;
    if ((st = validate_gemm_inputs(H, W, B, V, D)) != FS_OK) return st;
    if (!Y) return fail(FS_ERR_INVALID_ARG, "Y must be non-null");
    if (y_dtype != FS_DTYPE_BF16 && y_dtype != FS_DTYPE_F32)
        return fail(FS_ERR_INVALID_ARG, "y_dtype must be FS_DTYPE_BF16 or FS_DTYPE_F32");
    int dev;
    DeviceInfo info;
    if ((st = device_info(&dev, &info)) != FS_OK) return st;
    Plan p;
    make_plan(B, V, D, info.sms, &p);
    return run_stage1(y_dtype == FS_DTYPE_F32 ? kModeGemmF32 : kModeGemmBf16, H, W, p, 1.0f,
                      nullptr, 0, 0, 0, nullptr, Y, y_dtype, nullptr,
                      static_cast<cudaStream_t>(stream));
}

fs_status fs_sample_from_logits(const void *Y, int y_dtype, int64_t B, int64_t V,
                                float temperature, const float *temperatures, uint64_t seed,
                                uint64_t offset, uint32_t flags, int64_t *out_idx,
                                float *out_score, void *workspace, size_t ws_bytes,
                                void *stream) {
    fs_status st;
    if (!Y) return fail(FS_ERR_INVALID_ARG, "Y must be non-null");
    if (y_dtype != FS_DTYPE_BF16 && y_dtype != FS_DTYPE_F32)
        return fail(FS_ERR_INVALID_ARG, "y_dtype must be FS_DTYPE_BF16 or FS_DTYPE_F32");
    if ((st = validate_shape(B, V, 8)) != FS_OK) return st;
    if ((st = validate_temperature(temperature, temperatures)) != FS_OK) return st;
    if (flags & ~FS_FLAG_NO_NOISE)
        return fail(FS_ERR_INVALID_ARG, "only FS_FLAG_NO_NOISE applies to materialised logits");
    if (!out_idx) return fail(FS_ERR_INVALID_ARG, "out_idx must be non-null");
    if ((st = validate_outputs(out_idx, out_score, temperatures)) != FS_OK) return st;
    if ((st = validate_out(Y, y_dtype == FS_DTYPE_F32 ? 4 : 2, "Y")) != FS_OK) return st;
    int dev;
    DeviceInfo info;
    if ((st = device_info(&dev, &info)) != FS_OK) return st;
    Plan p;
    make_plan(B, V, 8, info.sms, &p);
    if ((st = validate_workspace(workspace, ws_bytes, p.wsLogitsBytes)) != FS_OK) return st;
    const Candidates cand = split_workspace(p, workspace, p.nChunks);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_logits_sample(Y, y_dtype, B, V, temperatures, temperature, seed,
                                         offset, flags, cand.score, cand.idx, p.nChunks,
                                         p.logitsChunk, s);
    if (e != cudaSuccess) return cuda_fail(e, "logits sampling launch");
    e = launch_stage2(cand.score, cand.idx, p.nChunks, B, temperatures, temperature, out_idx,
                      out_score, s);
    if (e != cudaSuccess) return cuda_fail(e, "Stage 2 launch");
    return FS_OK;
}

fs_status fs_sample_unfused(const void *H, const void *W, int64_t B, int64_t V, int64_t D,
                            float temperature, const float *temperatures, uint64_t seed,
                            uint64_t offset, void *Y, int y_dtype, int64_t *out_idx,
                            float *out_score, void *workspace, size_t ws_bytes, void *stream) {
    fs_status st;
    if ((st = validate_temperature(temperature, temperatures)) != FS_OK) return st;
    if (!out_idx) return fail(FS_ERR_INVALID_ARG, "out_idx must be non-null");
    if ((st = fs_logits_gemm(H, W, B, V, D, Y, y_dtype, stream)) != FS_OK) return st;
    return fs_sample_from_logits(Y, y_dtype, B, V, temperature, temperatures, seed, offset, 0,
                                 out_idx, out_score, workspace, ws_bytes, stream);
}

fs_status fs_debug_noise(uint64_t seed, uint64_t offset, int64_t b0, int64_t nb, int64_t V,
                         uint32_t *out_words, float *out_g, void *stream) {
    if (b0 < 0 || nb < 1 || V < 1)
        return fail(FS_ERR_INVALID_ARG, "need b0 >= 0, nb >= 1, V >= 1");
    if (!out_words && !out_g) return fail(FS_ERR_INVALID_ARG, "no output requested");
    int dev;
    DeviceInfo info;
    fs_status st = device_info(&dev, &info);
    if (st != FS_OK) return st;
    cudaError_t e = launch_debug_noise(seed, offset, b0, nb, V, out_words, out_g,
                                       static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "debug noise launch");
    return FS_OK;
}

fs_status fs_debug_gumbel(const uint32_t *words, int64_t n, float *out_g, void *stream) {
    if (!words || !out_g || n < 1)
        return fail(FS_ERR_INVALID_ARG, "need words, out_g and n >= 1");
    fs_status st;
    if ((st = validate_out(words, 4, "words")) != FS_OK) return st;
    if ((st = validate_out(out_g, 4, "out_g")) != FS_OK) return st;
    int dev;
    DeviceInfo info;
    if ((st = device_info(&dev, &info)) != FS_OK) return st;
    cudaError_t e = launch_debug_gumbel(words, n, out_g, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "debug gumbel launch");
    return FS_OK;
}

fs_status fs_get_device_status(void *stream, uint32_t *out_word) {
    int dev;
    DeviceInfo info;
    fs_status st = device_info(&dev, &info);
    if (st != FS_OK) return st;
    uint32_t w = 0;
    cudaError_t e = read_and_clear_status(static_cast<cudaStream_t>(stream), &w);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
    if (out_word) *out_word = w;
    if (w) return fail(FS_ERR_TIMEOUT, "a bounded wait inside Stage 1 expired (word 0x%x)", w);
    return FS_OK;
}

fs_status fs_release_workspaces(void) {
    std::lock_guard<std::mutex> lock(g_ws_mu);
    int cur = 0;
    cudaGetDevice(&cur);
    fs_status st = FS_OK;
    for (auto &kv : g_ws) {
        if (!kv.second.ptr) continue;
        cudaSetDevice(kv.first.first);
        cudaError_t e = cudaFree(kv.second.ptr);
        if (e != cudaSuccess && st == FS_OK) st = cuda_fail(e, "cudaFree(workspace)");
    }
    g_ws.clear();
    std::lock_guard<std::mutex> lock2(g_host_mu);
    for (auto &kv : g_host) {
        HostPath &h = kv.second;
        cudaSetDevice(kv.first.first);
        if (h.block) {
            cudaError_t e = cudaFree(h.block);
            if (e != cudaSuccess && st == FS_OK) st = cuda_fail(e, "cudaFree(host-path staging)");
        }
        for (int j = 0; j < 2; ++j) {
            if (h.uploaded[j]) cudaEventDestroy(h.uploaded[j]);
            if (h.consumed[j]) cudaEventDestroy(h.consumed[j]);
        }
        if (h.all_prior) cudaEventDestroy(h.all_prior);
        if (h.copy) cudaStreamDestroy(h.copy);
    }
    g_host.clear();
    cudaSetDevice(cur);
    return st;
}

}  // extern "C"

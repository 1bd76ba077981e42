// fs_noalloc.cu -- fs_sample_noalloc: the fused sampling call for callers
// that must not allocate device memory.
//
// Who needs it: applications that own all of the GPU's memory themselves, for
// example an inference server that reserves its memory pool at start-up and
// forbids any allocation afterwards, or a plug-in whose host process controls
// the allocator; and latency-critical decode loops that cannot pay for
// cudaMalloc, which may synchronise the device.  fs_sample grows a cached
// workspace with cudaMallocAsync and fs_sample_ex needs a caller buffer; this
// entry point needs neither.
//
// The Stage 1 candidate buffers (score and index arrays) live in
// g_noalloc_scratch, a static array in the library's own device memory
// (FS_NOALLOC_SCRATCH_BYTES on every GPU that loads the library, held until
// the process exits).  Host code cannot use the array's name as a device
// address, so the first call in each CUDA context looks the address up with
// cudaGetSymbolAddress (with that context's device current) and caches it;
// that first call should therefore come before any stream capture.  The
// cache is keyed by context, not by device ordinal: a context created again
// after cudaDeviceReset loads the module anew, possibly at another address.
// Every call shares the one array: calls whose kernels overlap on the GPU
// (different streams, or different host threads) race on it.  Nothing in it
// needs to start at zero: Stage 1 writes every candidate slot that Stage 2
// reads, and Stage 2 ignores the candidates of a call whose Stage 1 gave up a
// bounded wait (the device error word is set; every row then reads -1).
#include <cuda_runtime.h>

#include <map>
#include <mutex>

#include "../../include/fs_sample.h"
#include "fs_internal.h"

namespace fs {
fs_status set_error(fs_status st, const char *fmt, ...);  // fs_api.cu
}

static __device__ __align__(256) unsigned char g_noalloc_scratch[FS_NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_mu;
std::map<unsigned long long, void *> g_scratch_addr;  // device address, per CUDA context

// The device address of g_noalloc_scratch in the current context.
cudaError_t scratch_address(void **out) {
    unsigned long long ctx = 0;
    const bool have_ctx = fs::current_context_id(&ctx);
    std::lock_guard<std::mutex> lock(g_mu);
    if (have_ctx) {
        auto it = g_scratch_addr.find(ctx);
        if (it != g_scratch_addr.end()) {
            *out = it->second;
            return cudaSuccess;
        }
    }
    void *ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (ptr == nullptr) return cudaErrorInvalidSymbol;
    // the lookup makes the device's primary context current if none was
    if (have_ctx || fs::current_context_id(&ctx)) g_scratch_addr[ctx] = ptr;
    *out = ptr;
    return cudaSuccess;
}

}  // namespace

extern "C" fs_status fs_sample_noalloc(const void *H, const void *W, int64_t B, int64_t V,
                                       int64_t D, float temperature, const float *temperatures,
                                       uint64_t seed, uint64_t offset, int64_t *out_idx,
                                       float *out_score, void *stream) {
    // Plain sampling keeps two candidate arrays (score, index), each of
    // partitions x B four-byte values rounded up to 256 B.
    const size_t need = fs::sample_workspace_bytes(B, V, D);
    if (need == 0) {
        // bad arguments or no usable device: let the regular entry point
        // validate and report the reason (it launches nothing on error)
        return fs_sample_ex(H, W, B, V, D, temperature, temperatures, seed, offset, 0, out_idx,
                            out_score, nullptr, nullptr, 0, stream);
    }
    if (need > FS_NOALLOC_SCRATCH_BYTES)
        return fs::set_error(FS_ERR_UNSUPPORTED,
                             "fs_sample_noalloc: B=%lld, V=%lld needs %zu bytes of candidate "
                             "scratch, more than its static %d-byte array; use fs_sample_ex",
                             static_cast<long long>(B), static_cast<long long>(V), need,
                             FS_NOALLOC_SCRATCH_BYTES);
    void *scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess)
        return fs::set_error(FS_ERR_CUDA, "fs_sample_noalloc: cudaGetSymbolAddress: %s",
                             cudaGetErrorString(e));
    return fs_sample_ex(H, W, B, V, D, temperature, temperatures, seed, offset, 0, out_idx,
                        out_score, nullptr, scratch, FS_NOALLOC_SCRATCH_BYTES, stream);
}

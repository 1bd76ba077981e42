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
// The Stage 1 candidate buffers live in g_noalloc_scratch, a static array in
// the library's own device memory (FS_NOALLOC_SCRATCH_BYTES on every GPU that
// loads the library, held until the process exits).  Host code cannot use the
// array's name as a device address, so the first call on each device looks the
// address up with cudaGetSymbolAddress (with that device current) and caches
// it; that first call should therefore come before any stream capture.  Every
// call shares the one array: calls whose kernels overlap on the GPU (different
// streams, or different host threads) race on it.  Nothing in it needs to
// start at zero: Stage 1 writes every candidate slot that Stage 2 reads.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/fs_sample.h"

namespace fs {
fs_status set_error(fs_status st, const char *fmt, ...);  // fs_api.cu
}

static __device__ __align__(256) unsigned char g_noalloc_scratch[FS_NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_mu;
void *g_scratch_addr[64];  // device address of g_noalloc_scratch, per device ordinal

}  // namespace

extern "C" fs_status fs_sample_noalloc(const void *H, const void *W, int64_t B, int64_t V,
                                       int64_t D, float temperature, const float *temperatures,
                                       uint64_t seed, uint64_t offset, int64_t *out_idx,
                                       float *out_score, void *stream) {
    const size_t need = fs_workspace_size(B, V, D);
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
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fs::set_error(FS_ERR_CUDA, "fs_sample_noalloc: cudaGetDevice: %s",
                             cudaGetErrorString(e));
    if (dev < 0 || dev >= 64)
        return fs::set_error(FS_ERR_UNSUPPORTED, "fs_sample_noalloc: device ordinal %d", dev);
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_scratch_addr[dev]) {
            void *ptr = nullptr;
            e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
            if (e != cudaSuccess || ptr == nullptr)
                return fs::set_error(FS_ERR_CUDA,
                                     "fs_sample_noalloc: cudaGetSymbolAddress: %s",
                                     cudaGetErrorString(e));
            g_scratch_addr[dev] = ptr;
        }
        scratch = g_scratch_addr[dev];
    }
    return fs_sample_ex(H, W, B, V, D, temperature, temperatures, seed, offset, 0, out_idx,
                        out_score, nullptr, scratch, FS_NOALLOC_SCRATCH_BYTES, stream);
}

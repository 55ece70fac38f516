// noalloc.cu -- pkv_paged_decode_noalloc: paged decode whose split-K
// scratch lives in a fixed device array owned by the library, for callers
// that cannot allocate device memory at call time.
//
// Who needs it: code that enqueues work where cudaMalloc is not allowed or
// not affordable -- plugin / custom-op hooks of inference engines that hand
// the op only its inputs and outputs and forbid allocation while
// enqueueing, runtimes whose memory is owned by their own pool allocator,
// and latency-critical serving loops where cudaMalloc's implicit
// device-wide synchronisation would stall every other stream.  Such callers
// cannot provide the workspace that pkv_paged_decode asks for, so this entry
// point brings its own.
//
// The scratch is one file-scope __device__ array of kNoAllocScratchBytes.
// Every GPU that loads the library's device code reserves it until the
// process exits.  Host code must not hand the array's name to a kernel (on
// the host it is only a stand-in symbol), so the device address is looked
// up with cudaGetSymbolAddress once per device and cached.  The cache is
// keyed by device ordinal and so assumes the device's primary context (the
// one the runtime API uses) for the life of the process: after a
// cudaDeviceReset the cached address is stale.
#include <cstdio>
#include <mutex>

#include "pkv_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;   // 8 MiB

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device (looked up on
// the first call for that device, with that device current).
cudaError_t scratch_address(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

thread_local char g_msg[256];

}  // namespace

extern "C" {

size_t pkv_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

int pkv_paged_decode_noalloc(const pkv_tensor *q, const pkv_cache *cache,
                             const pkv_tensor *block_tables, const pkv_tensor *context_lens,
                             float sm_scale, const pkv_tensor *out, int num_splits,
                             int32_t *err_flag, void *stream)
{
    size_t need = 0;
    int rc = pkv_paged_decode_workspace(q, cache, block_tables, num_splits, &need);
    if (rc != PKV_OK) return rc;
    if (need > kNoAllocScratchBytes && num_splits == 0) {
        // The automatic plan does not fit: take the largest explicit split
        // count that does.  One split needs no scratch at all, so this
        // always ends with a plan.
        for (int s = 16; s >= 1; --s) {
            rc = pkv_paged_decode_workspace(q, cache, block_tables, s, &need);
            if (rc != PKV_OK) return rc;
            if (need <= kNoAllocScratchBytes) {
                num_splits = s;
                break;
            }
        }
    }
    if (need > kNoAllocScratchBytes) {
        // Report through the same per-thread message as every other call.
        snprintf(g_msg, sizeof(g_msg),
                 "paged_decode_noalloc: num_splits %d needs %zu bytes of scratch, more than the "
                 "library's fixed %zu-byte array; pass num_splits 0 (a plan that fits) or 1 "
                 "(no scratch)",
                 num_splits, need, kNoAllocScratchBytes);
        return pkv::set_last_error(PKV_ERR_WORKSPACE, g_msg);
    }
    void *scratch = nullptr;
    if (need > 0) {
        cudaError_t e = scratch_address(&scratch);
        if (e != cudaSuccess) {
            snprintf(g_msg, sizeof(g_msg), "paged_decode_noalloc: cudaGetSymbolAddress: %s",
                     cudaGetErrorString(e));
            return pkv::set_last_error(PKV_ERR_CUDA, g_msg);
        }
    }
    return pkv_paged_decode(q, cache, block_tables, context_lens, sm_scale, out, num_splits,
                            scratch, need > 0 ? kNoAllocScratchBytes : 0, err_flag, stream);
}

}  // extern "C"

// kda_noalloc.cu -- forward pass for callers that must not allocate device
// memory during the call.
//
// kda_fwd takes its per-chunk scratch from the stream-ordered allocator and
// kda_fwd_ws needs the caller to hand in a buffer.  Some callers can do
// neither: a serving runtime that reserves all device memory at start-up and
// forbids allocation on the request path, a plug-in that runs inside a host
// whose memory pools it does not own, or real-time code that cannot afford an
// allocator call (and the synchronisation it may imply) per request.  For
// them this file holds a fixed scratch area compiled into the library: every
// GPU that loads the library reserves it (kNoAllocScratchBytes) until the
// process exits, and kda_fwd_noalloc runs the usual kernels on it.
//
// Set-up: the first kda_fwd_noalloc call on a device, with that device
// current, asks the runtime for the area's device address
// (cudaGetSymbolAddress) and caches it; make that first call before any
// stream capture.  Later calls only read the cached address.
//
// Sharing: every call uses the same area, which keeps the previous call's
// contents.  Nothing in it has to start at zero (the schedule pass rewrites
// every byte the later kernels read before they read it), but two calls whose
// work overlaps on the GPU (different streams, or different host threads)
// race on the area and corrupt each other's results: serialise them.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "kda.h"
#include "kda_internal.h"

namespace {

// 64 MiB: room for about 800 (chunk, head) records, e.g. a 4096-token prefill
// with 12 heads, or decode-sized batches.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;

static __device__ __align__(256) unsigned char g_kda_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[128] = {nullptr};

// Device address of the scratch area on the current device (looked up once).
kda_status_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return kda::cuda_error(e, "kda_fwd_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= 128)
        return kda::set_error(KDA_ERR_UNSUPPORTED, "kda_fwd_noalloc: device index above 127");
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_kda_noalloc_scratch);
        if (e != cudaSuccess)
            return kda::cuda_error(e, "kda_fwd_noalloc: cudaGetSymbolAddress(scratch)");
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return KDA_OK;
}

}  // namespace

extern "C" size_t kda_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" kda_status_t kda_fwd_noalloc(const void* q, const void* k, const void* v, const void* g,
                                        const void* beta, float scale, void* out,
                                        const float* A_log, const float* dt_bias,
                                        float lower_bound, const void* initial_state,
                                        kda_dtype_t initial_dtype, void* final_state,
                                        kda_dtype_t final_dtype, const int32_t* cu_seqlens,
                                        int32_t num_seqs, int32_t B, int32_t T, int32_t H,
                                        int32_t K, int32_t V, void* stream) {
    kda::clear_error();
    const size_t need = kda_workspace_size(B, T, H, num_seqs, cu_seqlens != nullptr ? 1 : 0);
    if (need == 0) return KDA_ERR_INVALID_ARGUMENT;  // message set by kda_workspace_size
    if (need > kNoAllocScratchBytes) {
        char msg[256];
        std::snprintf(msg, sizeof msg,
                      "kda_fwd_noalloc: this problem needs %zu bytes of scratch but the built-in "
                      "area holds %zu (64 MiB); use kda_fwd or kda_fwd_ws",
                      need, kNoAllocScratchBytes);
        return kda::set_error(KDA_ERR_UNSUPPORTED, msg);
    }
    void* ws = nullptr;
    const kda_status_t rc = scratch_address(&ws);
    if (rc != KDA_OK) return rc;
    return kda_fwd_ws(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state,
                      initial_dtype, final_state, final_dtype, cu_seqlens, num_seqs, B, T, H, K, V,
                      ws, kNoAllocScratchBytes, stream);
}

// ssd_scan_varlen_noalloc: the same scan for callers that cannot allocate
// device memory.
//
// Some callers have no way to hand the library a workspace: a serving engine
// that gives all free HBM to its state and KV pools at start-up and forbids
// later cudaMalloc calls (they would fail, or fragment the pool); a plug-in
// or foreign-language runtime whose ABI only passes in the tensors it already
// owns; a latency-critical path where cudaMalloc's implicit device-wide
// synchronisation is not acceptable.  For them this entry point takes its
// scratch -- the longest-first sequence order the chunked kernel needs --
// from a fixed array in the library's own device memory instead of
// `params->workspace`.
//
// Costs and limits:
//  * every GPU that loads the library holds the array (kNoallocMaxSeqs
//    int32 = 256 KiB) until the process exits;
//  * batches of more than kNoallocMaxSeqs sequences are rejected with
//    SSD_ERR_SCRATCH_LIMIT before anything is enqueued;
//  * the first call on a device looks up the array's device address (with
//    that device current) -- make that first call before any stream capture;
//  * all calls share the one array: two calls whose kernels overlap on the
//    GPU (different streams, no ordering between them) race on it.  The
//    kernels rewrite every entry they read, so nothing has to start at zero.
#include <mutex>

#include "ssd_internal.h"

namespace {

constexpr int kNoallocMaxSeqs = SSD_NOALLOC_MAX_SEQS;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) int32_t g_noalloc_scratch[kNoallocMaxSeqs];

std::mutex g_setup_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
cudaError_t scratch_for_current_device(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" ssd_status ssd_scan_varlen_noalloc(const ssd_scan_params *params,
                                              struct CUstream_st *stream) {
    const ssd_status v = ssd::detail::validate(params);
    if (v != SSD_OK) return v;
    if (params->num_seqs == 0) return SSD_OK;
    if (params->num_seqs > kNoallocMaxSeqs) return SSD_ERR_SCRATCH_LIMIT;
    const ssd::ScanArgs a = ssd::detail::make_args(params);
    cudaError_t err;
    if (ssd::detail::use_chunked(params)) {
        void *scratch = nullptr;
        err = scratch_for_current_device(&scratch);
        if (err == cudaSuccess) err = ssd::launch_chunked(a, params->state_dtype, scratch, sizeof(g_noalloc_scratch), stream);
    } else {
        err = ssd::launch_recurrent(a, params->io_dtype, params->state_dtype, stream);
    }
    return err == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

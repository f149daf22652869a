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
//  * on the tensor-core path, batches of more than kNoallocMaxSeqs sequences
//    are rejected with SSD_ERR_SCRATCH_LIMIT before anything is enqueued (the
//    token-by-token path needs no scratch and takes any batch);
//  * the array has no room for the snapshot of initial states that calls
//    with crossed or shared slots need: such calls are rejected with
//    SSD_ERR_SCRATCH_LIMIT unless the caller sets slots_disjoint;
//  * every call looks the array's device address up with the call's device
//    current (a host-side lookup; the first one on a device may load the
//    library's module, so make it before any stream capture).  Not caching the
//    address keeps a call correct after the device was reset and the module
//    reloaded elsewhere;
//  * all calls share the one array: two calls whose kernels overlap on the
//    GPU (different streams, no ordering between them) race on it.  The
//    kernels rewrite every entry they read, so nothing has to start at zero.
#include "ssd_internal.h"

namespace {

constexpr int kNoallocMaxSeqs = SSD_NOALLOC_MAX_SEQS;

static __device__ __align__(256) int32_t g_noalloc_scratch[kNoallocMaxSeqs];

// Device address of the scratch array on the current device.
cudaError_t scratch_for_current_device(void **out) {
    void *ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    *out = ptr;
    return cudaSuccess;
}

}  // namespace

extern "C" ssd_status ssd_scan_varlen_noalloc(const ssd_scan_params *params,
                                              struct CUstream_st *stream) {
    const ssd_status v = ssd::detail::validate(params);
    if (v != SSD_OK) return v;
    if (params->num_seqs == 0) return SSD_OK;
    if (ssd::snapshot_needed(*params)) return SSD_ERR_SCRATCH_LIMIT;
    const bool chunked = ssd::detail::use_chunked(params);
    if (chunked && params->num_seqs > kNoallocMaxSeqs) return SSD_ERR_SCRATCH_LIMIT;
    void *scratch = nullptr;
    if (chunked) {
        const cudaError_t err = scratch_for_current_device(&scratch);
        if (err != cudaSuccess) return SSD_ERR_CUDA;
    }
    return ssd::detail::run(params, scratch, chunked ? sizeof(g_noalloc_scratch) : 0, stream);
}

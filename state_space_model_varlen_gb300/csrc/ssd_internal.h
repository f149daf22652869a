// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ssd_scan.h"

namespace ssd {

// Launch-ready copy of the public parameters (validated on the host).
struct ScanArgs {
    int64_t T;
    int32_t S, H, P, N, G;
    int32_t max_seqlen;          // host hint (0 = unknown)
    int32_t heads_per_group;
    int32_t num_slots;
    int32_t dt_softplus, write_final;
    const void *x;
    const float *dt, *dt_bias, *A, *D;
    const void *B, *C;
    const int32_t *cu_seqlens, *slot_idx;
    const uint8_t *has_init;
    void *state_cache, *out_y, *out_intermediate;
    int32_t *device_status;
};

// Token-by-token SIMT scan (any shape with N <= 256, any dtype).  One launch.
cudaError_t launch_recurrent(const ScanArgs &a, int io_dtype, int state_dtype,
                             cudaStream_t stream);

// Chunked tcgen05 scan (bf16 I/O, P = 64, N = 128).  One or two launches.  Long
// sequences are cut into segments run by different CTAs when the workspace
// holds chunked_workspace_bytes; a smaller one (at least 4 S bytes, the
// sequence order) runs every sequence on one CTA.
bool chunked_supported(const ssd_scan_params &p);
size_t chunked_workspace_bytes(const ssd_scan_params &p);
cudaError_t launch_chunked(const ScanArgs &a, int state_dtype, void *workspace,
                           size_t workspace_bytes, cudaStream_t stream);
// Launches of a chunked call with this workspace size on the current device
// (1 when the kernel sorts a small unsegmented batch itself, else 2; -1 on a
// CUDA error).
int32_t chunked_num_launches(const ssd_scan_params &p, size_t workspace_bytes);

namespace detail {
// Host-side argument checks, launch arguments and kernel-path choice shared by
// the entry points (defined in ssd_api.cu).
ssd_status validate(const ssd_scan_params *p);
ScanArgs make_args(const ssd_scan_params *p);
bool use_chunked(const ssd_scan_params *p);
}  // namespace detail

}  // namespace ssd

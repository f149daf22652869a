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
    // per-chunk (checkpoint) states
    void *out_chunk_states;
    const int32_t *cu_chunks;
    int32_t num_chunk_rows, chunk_size;
    // slots: entry s of slot_idx at s * slot_stride; final states to final_slot_idx
    const int32_t *final_slot_idx;
    int64_t slot_stride, final_slot_stride;
    const uint64_t *sr_seed;     // fp16 caches: stochastic rounding seed (device)
    // snapshot of initial states that another sequence's final slot would
    // overwrite (workspace, filled by the snapshot pass): flag and state per sequence
    const int32_t *snap_flag;
    const void *snap_states;
    // ReplaySSM verification (ring_x != nullptr)
    void *ring_x, *ring_B;
    float *ring_dt;
    int32_t ring_capacity, ring_window;
    const int32_t *ring_start, *ring_count;
    int32_t *ring_start_out, *ring_count_out;
};

// Workspace of the snapshot pass (offsets from the workspace base, 256-byte
// aligned): int32 flags [S], then S states in the cache dtype.
struct SnapLayout {
    size_t flags = 0, states = 0, total = 0;
};
SnapLayout snapshot_layout(const ssd_scan_params &p, size_t base);
bool snapshot_needed(const ssd_scan_params &p);
// The snapshot pass: one launch that copies, for every sequence whose initial
// slot is another sequence's final slot, its initial state into the workspace.
// The chunked path folds it into its prep launch instead (prep_snapshot below).
cudaError_t launch_snapshot(const ScanArgs &a, int state_dtype, int32_t *flags, void *states,
                            cudaStream_t stream);
struct SnapshotArgs;
SnapshotArgs make_snapshot_args(const ScanArgs &a, int state_dtype, int32_t *flags, void *states);

// Token-by-token SIMT scan (any shape with N <= 256, any dtype).  One launch.
cudaError_t launch_recurrent(const ScanArgs &a, int io_dtype, int state_dtype,
                             cudaStream_t stream);
// Bytes of one sequence's state in the cache dtype.
size_t state_bytes(const ssd_scan_params &p);

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
// Failure-detection test hooks of the chunked kernel (ssd_testing_set_hooks).
void set_test_hooks(int64_t wait_cycles, int32_t withhold, int32_t force_unsegmented);

namespace detail {
// Host-side argument checks, launch arguments and kernel-path choice shared by
// the entry points (defined in ssd_api.cu).
ssd_status validate(const ssd_scan_params *p);
ScanArgs make_args(const ssd_scan_params *p);
bool use_chunked(const ssd_scan_params *p);
SnapLayout workspace_layout(const ssd_scan_params *p);
ssd_status run(const ssd_scan_params *params, void *workspace, size_t workspace_bytes, cudaStream_t stream);
}  // namespace detail

}  // namespace ssd

// C ABI entry points: host-side validation and kernel-path selection.
// See include/ssd_scan.h for the contract.
#include <string.h>

#include "ssd_internal.h"

namespace ssd {
namespace detail {

namespace {
bool dtype_ok(int d) { return d == SSD_F32 || d == SSD_BF16 || d == SSD_F16; }
}  // namespace

// Host-side argument validation; no device memory is read.
ssd_status validate(const ssd_scan_params *p) {
    if (p == nullptr) return SSD_ERR_INVALID_ARG;
    if (p->total_tokens < 0 || p->num_seqs < 0 || p->max_seqlen < 0) return SSD_ERR_INVALID_ARG;
    if (p->nheads <= 0 || p->headdim <= 0 || p->dstate <= 0 || p->ngroups <= 0)
        return SSD_ERR_INVALID_ARG;
    if (p->nheads % p->ngroups != 0 || p->chunk_size <= 0) return SSD_ERR_INVALID_ARG;
    if (!(p->io_dtype == SSD_F32 || p->io_dtype == SSD_BF16)) return SSD_ERR_INVALID_ARG;
    if (!dtype_ok(p->state_dtype)) return SSD_ERR_INVALID_ARG;
    if (p->num_seqs > 0) {
        if (p->cu_seqlens == nullptr || p->dt == nullptr || p->A == nullptr)
            return SSD_ERR_INVALID_ARG;
        if (p->total_tokens > 0 &&
            (p->x == nullptr || p->B == nullptr || p->C == nullptr || p->out_y == nullptr))
            return SSD_ERR_INVALID_ARG;
        const bool uses_slots = p->write_final || p->has_init != nullptr;
        if (uses_slots && (p->state_cache == nullptr || p->slot_idx == nullptr || p->num_slots <= 0))
            return SSD_ERR_INVALID_ARG;
    }
    if (p->slot_idx_stride < 0 || p->final_slot_idx_stride < 0) return SSD_ERR_INVALID_ARG;
    if (p->out_chunk_states != nullptr && (p->cu_chunks == nullptr || p->num_chunk_rows < 0))
        return SSD_ERR_INVALID_ARG;
    if (p->final_slot_idx != nullptr && !p->write_final) return SSD_ERR_INVALID_ARG;
    if (p->dstate > 256) return SSD_ERR_UNSUPPORTED;
    // index arithmetic is 64-bit; keep per-token strides in range
    if ((int64_t)p->nheads * p->headdim * p->dstate > (1LL << 31)) return SSD_ERR_UNSUPPORTED;
    return SSD_OK;
}

ssd::ScanArgs make_args(const ssd_scan_params *p) {
    ssd::ScanArgs a;
    a.T = p->total_tokens;
    a.S = p->num_seqs;
    a.max_seqlen = p->max_seqlen;
    a.H = p->nheads;
    a.P = p->headdim;
    a.N = p->dstate;
    a.G = p->ngroups;
    a.heads_per_group = p->nheads / p->ngroups;
    a.num_slots = p->num_slots;
    a.dt_softplus = p->dt_softplus ? 1 : 0;
    a.write_final = p->write_final ? 1 : 0;
    a.x = p->x;
    a.dt = p->dt;
    a.dt_bias = p->dt_bias;
    a.A = p->A;
    a.D = p->D;
    a.B = p->B;
    a.C = p->C;
    a.cu_seqlens = p->cu_seqlens;
    a.slot_idx = p->slot_idx;
    a.has_init = p->has_init;
    a.state_cache = p->state_cache;
    a.out_y = p->out_y;
    a.out_intermediate = p->out_intermediate;
    a.device_status = p->device_status;
    a.out_chunk_states = p->out_chunk_states;
    a.cu_chunks = p->cu_chunks;
    a.num_chunk_rows = p->num_chunk_rows;
    a.chunk_size = p->chunk_size;
    a.final_slot_idx = p->final_slot_idx;
    a.slot_stride = p->slot_idx_stride;
    a.final_slot_stride = p->final_slot_idx_stride;
    a.sr_seed = p->state_dtype == SSD_F16 ? p->sr_seed : nullptr;
    a.snap_flag = nullptr;
    a.snap_states = nullptr;
    a.ring_x = a.ring_B = nullptr;
    a.ring_dt = nullptr;
    a.ring_capacity = a.ring_window = 0;
    a.ring_start = a.ring_count = nullptr;
    a.ring_start_out = a.ring_count_out = nullptr;
    return a;
}

// The tensor-core chunked kernel covers bf16 prefill shapes; continuations of
// at most three tokens and everything else go token by token.
bool use_chunked(const ssd_scan_params *p) {
    if (p->out_intermediate != nullptr) return false;
    if (p->max_seqlen > 0 && p->max_seqlen <= 3) return false;
    return ssd::chunked_supported(*p);
}

// Workspace of a call: the chunked kernel's part first, then the snapshot's.
SnapLayout workspace_layout(const ssd_scan_params *p) {
    const size_t base = use_chunked(p) ? ssd::chunked_workspace_bytes(*p) : 0;
    return snapshot_layout(*p, base);
}

// Run the scan with `workspace` (already checked to hold the layout).
ssd_status run(const ssd_scan_params *params, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    ssd::ScanArgs a = make_args(params);
    if (snapshot_needed(*params)) {
        const SnapLayout L = workspace_layout(params);
        uint8_t *ws = static_cast<uint8_t *>(workspace);
        a.snap_flag = reinterpret_cast<const int32_t *>(ws + L.flags);
        a.snap_states = ws + L.states;
    }
    cudaError_t err;
    if (use_chunked(params)) {
        err = ssd::launch_chunked(a, params->state_dtype, workspace, workspace_bytes, stream);
    } else {
        err = cudaSuccess;
        if (a.snap_flag != nullptr)
            err = ssd::launch_snapshot(a, params->state_dtype, const_cast<int32_t *>(a.snap_flag),
                                       const_cast<void *>(a.snap_states), stream);
        if (err == cudaSuccess) err = ssd::launch_recurrent(a, params->io_dtype, params->state_dtype, stream);
    }
    return err == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace detail
}  // namespace ssd

using ssd::detail::make_args;
using ssd::detail::use_chunked;
using ssd::detail::validate;

extern "C" {

size_t ssd_scan_varlen_workspace_size(const ssd_scan_params *params) {
    if (validate(params) != SSD_OK) return 0;
    if (params->num_seqs == 0) return 0;
    return ssd::detail::workspace_layout(params).total;
}

int32_t ssd_scan_varlen_num_launches(const ssd_scan_params *params) {
    if (validate(params) != SSD_OK) return -1;
    if (params->num_seqs == 0) return 0;
    if (use_chunked(params)) return ssd::chunked_num_launches(*params, params->workspace_bytes);
    return ssd::snapshot_needed(*params) ? 2 : 1;
}

const char *ssd_scan_varlen_path(const ssd_scan_params *params) {
    if (validate(params) != SSD_OK) return "invalid";
    return use_chunked(params) ? "chunked_tc" : "recurrent";
}

ssd_status ssd_scan_varlen(const ssd_scan_params *params, struct CUstream_st *stream) {
    const ssd_status v = validate(params);
    if (v != SSD_OK) return v;
    if (params->num_seqs == 0) return SSD_OK;
    const size_t need = ssd::detail::workspace_layout(params).total;
    if (need > 0 && (params->workspace == nullptr || params->workspace_bytes < need ||
                     (reinterpret_cast<uintptr_t>(params->workspace) & 255u) != 0))
        return SSD_ERR_WORKSPACE;
    return ssd::detail::run(params, params->workspace, params->workspace_bytes, stream);
}

ssd_status ssd_replay_mtp(const ssd_replay_params *rp, struct CUstream_st *stream) {
    if (rp == nullptr) return SSD_ERR_INVALID_ARG;
    const ssd_scan_params *params = &rp->scan;
    const ssd_status v = validate(params);
    if (v != SSD_OK) return v;
    if (params->write_final || params->out_intermediate != nullptr || params->out_chunk_states != nullptr ||
        params->final_slot_idx != nullptr || params->state_cache == nullptr || params->slot_idx == nullptr ||
        params->num_slots <= 0)
        return SSD_ERR_INVALID_ARG;
    if (rp->ring_x == nullptr || rp->ring_dt == nullptr || rp->ring_B == nullptr || rp->ring_start == nullptr ||
        rp->ring_count == nullptr || rp->ring_start_out == nullptr || rp->ring_count_out == nullptr)
        return SSD_ERR_INVALID_ARG;
    if (rp->ring_window < 0 || rp->ring_capacity <= rp->ring_window) return SSD_ERR_INVALID_ARG;
    if (params->max_seqlen > 0 && params->max_seqlen > rp->ring_capacity - rp->ring_window)
        return SSD_ERR_INVALID_ARG;
    if (rp->ring_start_out == rp->ring_start || rp->ring_count_out == rp->ring_count) return SSD_ERR_INVALID_ARG;
    if (params->num_seqs == 0) return SSD_OK;
    ssd::ScanArgs a = make_args(params);
    a.has_init = nullptr;
    a.ring_x = rp->ring_x;
    a.ring_dt = rp->ring_dt;
    a.ring_B = rp->ring_B;
    a.ring_capacity = rp->ring_capacity;
    a.ring_window = rp->ring_window;
    a.ring_start = rp->ring_start;
    a.ring_count = rp->ring_count;
    a.ring_start_out = rp->ring_start_out;
    a.ring_count_out = rp->ring_count_out;
    const cudaError_t err = ssd::launch_recurrent(a, params->io_dtype, params->state_dtype, stream);
    return err == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

void ssd_testing_set_hooks(int64_t wait_cycles, int32_t withhold_handover, int32_t force_unsegmented) {
    ssd::set_test_hooks(wait_cycles, withhold_handover, force_unsegmented);
}

const char *ssd_status_string(ssd_status status) {
    switch (status) {
        case SSD_OK: return "ok";
        case SSD_ERR_INVALID_ARG: return "invalid argument";
        case SSD_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case SSD_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case SSD_ERR_CUDA: return "CUDA error while enqueueing";
        case SSD_ERR_SCRATCH_LIMIT: return "batch exceeds the fixed scratch of the no-allocation entry point";
    }
    return "unknown status";
}

}  // extern "C"

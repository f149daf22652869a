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
    return a;
}

// The tensor-core chunked kernel covers bf16 prefill shapes; continuations of
// at most three tokens and everything else go token by token.
bool use_chunked(const ssd_scan_params *p) {
    if (p->out_intermediate != nullptr) return false;
    if (p->max_seqlen > 0 && p->max_seqlen <= 3) return false;
    return ssd::chunked_supported(*p);
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
    return use_chunked(params) ? ssd::chunked_workspace_bytes(*params) : 0;
}

int32_t ssd_scan_varlen_num_launches(const ssd_scan_params *params) {
    if (validate(params) != SSD_OK) return -1;
    if (params->num_seqs == 0) return 0;
    return use_chunked(params) ? ssd::chunked_num_launches(*params, params->workspace_bytes) : 1;
}

const char *ssd_scan_varlen_path(const ssd_scan_params *params) {
    if (validate(params) != SSD_OK) return "invalid";
    return use_chunked(params) ? "chunked_tc" : "recurrent";
}

ssd_status ssd_scan_varlen(const ssd_scan_params *params, struct CUstream_st *stream) {
    const ssd_status v = validate(params);
    if (v != SSD_OK) return v;
    if (params->num_seqs == 0) return SSD_OK;
    const ssd::ScanArgs a = make_args(params);
    cudaError_t err;
    if (use_chunked(params)) {
        const size_t need = ssd::chunked_workspace_bytes(*params);
        if (need > 0 && (params->workspace == nullptr || params->workspace_bytes < need ||
                         (reinterpret_cast<uintptr_t>(params->workspace) & 255u) != 0))
            return SSD_ERR_WORKSPACE;
        err = ssd::launch_chunked(a, params->state_dtype, params->workspace, params->workspace_bytes, stream);
    } else {
        err = ssd::launch_recurrent(a, params->io_dtype, params->state_dtype, stream);
    }
    return err == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
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

// The snapshot pass of calls whose sequences may read a slot that another
// sequence of the same call writes (crossed or shared slots, vLLM PR #62922
// "Details" and "Correctness"): one CTA per sequence checks whether its
// initial slot is another sequence's final slot and, if so, copies the slot
// into the workspace before the scan kernel writes any final state.
#include "ssd_common.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kSnapThreads = 256;

__global__ void __launch_bounds__(kSnapThreads) snapshot_kernel(SnapshotArgs a) {
    __shared__ int conflict;
    for (int s = blockIdx.x; s < a.S; s += gridDim.x) snapshot_sequence(a, s, &conflict);
}

size_t dtype_bytes(int d) { return d == SSD_F32 ? 4 : 2; }

}  // namespace

size_t state_bytes(const ssd_scan_params &p) {
    return (size_t)p.nheads * p.headdim * p.dstate * dtype_bytes(p.state_dtype);
}

// Needed when more than one sequence may read an initial state while final
// states are written, unless the caller promises disjoint slots.
bool snapshot_needed(const ssd_scan_params &p) {
    return p.has_init != nullptr && p.write_final && p.num_seqs > 1 && !p.slots_disjoint;
}

SnapLayout snapshot_layout(const ssd_scan_params &p, size_t base) {
    SnapLayout L;
    L.total = base;
    if (!snapshot_needed(p)) return L;
    auto r256 = [](size_t v) { return (v + 255) & ~(size_t)255; };
    L.flags = r256(base);
    L.states = r256(L.flags + (size_t)p.num_seqs * sizeof(int32_t));
    L.total = L.states + (size_t)p.num_seqs * state_bytes(p);     // states packed like cache slots
    return L;
}

SnapshotArgs make_snapshot_args(const ScanArgs &a, int state_dtype, int32_t *flags, void *states) {
    SnapshotArgs s;
    s.slot_idx = a.slot_idx;
    s.final_slot_idx = a.final_slot_idx;
    s.slot_stride = a.slot_stride ? a.slot_stride : 1;
    s.final_slot_stride = a.final_slot_stride ? a.final_slot_stride : 1;
    s.has_init = a.has_init;
    s.S = a.S;
    s.num_slots = a.num_slots;
    s.cache = static_cast<const uint8_t *>(a.state_cache);
    s.state_bytes = (size_t)a.H * a.P * a.N * dtype_bytes(state_dtype);
    s.flags = flags;
    s.states = static_cast<uint8_t *>(states);
    return s;
}

cudaError_t launch_snapshot(const ScanArgs &a, int state_dtype, int32_t *flags, void *states,
                            cudaStream_t stream) {
    const SnapshotArgs s = make_snapshot_args(a, state_dtype, flags, states);
    const int grid = a.S < 4096 ? a.S : 4096;
    if (grid <= 0) return cudaSuccess;
    snapshot_kernel<<<grid, kSnapThreads, 0, stream>>>(s);
    return cudaGetLastError();
}

}  // namespace ssd

"""ssd_scan_varlen_noalloc: the entry point for callers that cannot allocate.

Some callers cannot give the library a workspace: an engine that has handed
all free device memory to its state/KV pools and forbids later cudaMalloc, a
plug-in ABI that only passes the caller's own tensors, or a latency-critical
path that cannot take cudaMalloc's device-wide synchronisation.  This entry
point uses a fixed scratch array in the library's device memory instead.  The
GPU test checks, through the C ABI, that it returns what ssd_scan_varlen
returns, on two calls in a row (the second call sees the first call's stale
scratch); the CPU test checks the size limit.  This file is collected last so
that a failure here never hides the other tests.
"""
import ctypes

import numpy as np
import pytest

from state_space_model_varlen_gb300 import binding
from state_space_model_varlen_gb300 import workloads as W
from tests import harness as Hn


def _problems():
    # chunked tensor-core path (uses scratch), then a different batch shape
    a = W.make_problem([300, 7, 129, 0, 64], nheads=8, headdim=64, dstate=128, ngroups=2,
                       num_slots=8, has_init=[1, 0, 1, 1, 0], cache_std=0.1, seed=91)
    b = W.make_problem([5, 700, 1, 250], nheads=4, headdim=64, dstate=128, ngroups=1,
                       state_dtype="bf16", num_slots=6, has_init=[0, 1, 1, 0], cache_std=0.1,
                       seed=92)
    return [a, b]


def _run(p, noalloc):
    """Run one problem through the chosen C entry point; host copies of y and cache."""
    import torch
    d = Hn.upload(p)
    y = torch.full_like(d["x"], float("nan"))
    params = binding.make_params(
        d["x"], d["dt"], d["A"], d["B"], d["C"], d["cu_seqlens"], dt_bias=d["dt_bias"], D=d["D"],
        state_cache=d["state_cache"], slot_idx=d["slot_idx"], has_init=d["has_init"],
        write_final=p.write_final, out_y=y, dt_softplus=p.dt_softplus, chunk_size=p.chunk_size,
        max_seqlen=p.max_seqlen, slots_disjoint=True)     # distinct slots: no snapshot needed
    assert binding.kernel_path(params) == "chunked_tc"
    lib = binding.load()
    stream = torch.cuda.current_stream().cuda_stream
    if noalloc:
        rc = lib.ssd_scan_varlen_noalloc(ctypes.byref(params), ctypes.c_void_p(stream))
    else:
        need = binding.workspace_size(params)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        params.workspace, params.workspace_bytes = ws.data_ptr(), need
        rc = lib.ssd_scan_varlen(ctypes.byref(params), ctypes.c_void_p(stream))
    assert rc == binding.SSD_OK, binding.status_string(rc)
    torch.cuda.synchronize()
    y_host = Hn.oracle.widen(Hn._numpy(y, p.io_dtype), p.io_dtype)
    return y_host, Hn._numpy(d["state_cache"], p.state_dtype)


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice_in_a_row():
    for p in _problems():                       # two calls in a row, different batches
        y_ref, cache_ref = _run(p, noalloc=False)
        y_na, cache_na = _run(p, noalloc=True)
        Hn.check_y(y_na, y_ref, p.io_dtype)
        for s in range(p.num_seqs):
            slot = int(p.slot_idx[s])
            Hn.check_state(cache_na[slot], Hn.oracle.widen(cache_ref[slot], p.state_dtype),
                           p.state_dtype)
        untouched = [i for i in range(p.num_slots) if i not in set(int(v) for v in p.slot_idx)]
        np.testing.assert_array_equal(cache_na[untouched], p.cache[untouched])


def test_noalloc_rejects_batches_beyond_its_scratch():
    """More sequences than the fixed scratch holds on the tensor-core path (the
    one that uses scratch; zero tokens keep the path choice on the host): clear
    error, nothing enqueued.  A call that would need the snapshot of initial
    states is rejected the same way, unless the caller declares disjoint slots."""
    p = binding.ScanParams()
    p.total_tokens, p.num_seqs = 0, binding.SSD_NOALLOC_MAX_SEQS + 1
    p.nheads, p.headdim, p.dstate, p.ngroups, p.chunk_size = 4, 64, 128, 2, 128
    p.io_dtype, p.state_dtype, p.dt_softplus, p.write_final, p.num_slots = 1, 0, 1, 1, 4
    for name in ("x", "dt", "A", "B", "C", "cu_seqlens", "state_cache", "slot_idx", "out_y"):
        setattr(p, name, 0x1000)
    assert binding.kernel_path(p) == "chunked_tc"
    rc = binding.load().ssd_scan_varlen_noalloc(ctypes.byref(p), None)
    assert rc == binding.SSD_ERR_SCRATCH_LIMIT
    assert "scratch" in binding.status_string(rc)
    p.num_seqs, p.has_init = 3, 0x1000          # crossed slots possible: needs a snapshot
    assert binding.load().ssd_scan_varlen_noalloc(ctypes.byref(p), None) == binding.SSD_ERR_SCRATCH_LIMIT

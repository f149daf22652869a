"""Test harness: move a seeded ``workloads.Problem`` to the GPU, run the scan
through the C ABI, bring the results back and compare them with the oracle.

Tolerances (the scan's stated bounds, plus the rounding of the stored result):
  y, bf16 I/O:      |dy| <= 2e-2 * rms(y_ref) + 2^-8 |y_ref|
  y, fp32 I/O:      |dy| <= 1e-3 * rms(y_ref) + 2^-23 |y_ref|
  states, per slot: |dh| <= tol * rms(h_ref) + u |h_ref|
                    tol = 1e-3 (fp32 storage) or 1e-2 (bf16/fp16 storage),
                    u = half an ulp of the storage type relative to the value
                    (2^-24 fp32, 2^-8 bf16, 2^-11 fp16).
The ``u |ref|`` term is the unavoidable rounding of a correctly rounded
result into its storage type; without it the bf16 bound would be violated by
the exact answer wherever |y| exceeds about 5 rms.
"""
from __future__ import annotations

import numpy as np

import oracle

UNIT = {"f32": 2.0 ** -24, "bf16": 2.0 ** -8, "f16": 2.0 ** -11}


def _torch():
    import torch
    return torch


def _tensor(a: np.ndarray, dtype: str, device):
    torch = _torch()
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def _numpy(t, dtype: str) -> np.ndarray:
    torch = _torch()
    if dtype == "bf16":
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def upload(p, device="cuda"):
    torch = _torch()
    d = {
        "x": _tensor(p.x, p.io_dtype, device),
        "dt": torch.from_numpy(p.dt).to(device),
        "A": torch.from_numpy(p.A).to(device),
        "B": _tensor(p.B, p.io_dtype, device),
        "C": _tensor(p.C, p.io_dtype, device),
        "cu_seqlens": torch.from_numpy(p.cu_seqlens).to(device),
        "dt_bias": None if p.dt_bias is None else torch.from_numpy(p.dt_bias).to(device),
        "D": None if p.D is None else torch.from_numpy(p.D).to(device),
        "state_cache": _tensor(p.cache, p.state_dtype, device),
        "slot_idx": torch.from_numpy(p.slot_idx).to(device),
        "has_init": None if p.has_init is None else torch.from_numpy(p.has_init).to(device),
    }
    return d


def run_gpu(p, *, device="cuda", max_seqlen=None, status=False, chunk_size=None):
    """Run the CUDA scan on problem ``p``; returns a dict of host numpy arrays."""
    torch = _torch()
    from state_space_model_varlen_gb300 import binding
    d = upload(p, device)
    T, H, P, N = p.total_tokens, p.nheads, p.headdim, p.dstate
    y = torch.full_like(d["x"], float("nan"))
    inter = None
    if p.want_intermediate:
        st = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[p.state_dtype]
        inter = torch.full((T, H, P, N), float("nan"), dtype=st, device=device)
    dev_status = torch.zeros(1, dtype=torch.int32, device=device)
    params = binding.make_params(
        d["x"], d["dt"], d["A"], d["B"], d["C"], d["cu_seqlens"], dt_bias=d["dt_bias"], D=d["D"],
        state_cache=d["state_cache"], slot_idx=d["slot_idx"], has_init=d["has_init"],
        write_final=p.write_final, out_y=y, out_intermediate=inter, dt_softplus=p.dt_softplus,
        chunk_size=chunk_size or p.chunk_size,
        max_seqlen=p.max_seqlen if max_seqlen is None else max_seqlen, device_status=dev_status)
    need = binding.workspace_size(params)
    ws = None
    if need:
        ws = torch.empty(need, dtype=torch.uint8, device=device)
        params.workspace, params.workspace_bytes = ws.data_ptr(), need
    path = binding.kernel_path(params)
    launches = binding.num_launches(params)
    binding.call(params, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    out = {
        "y": oracle.widen(_numpy(y, p.io_dtype), p.io_dtype),
        "cache": _numpy(d["state_cache"], p.state_dtype),
        "inter": None if inter is None else _numpy(inter, p.state_dtype),
        "status": int(dev_status.item()),
        "path": path,
        "launches": launches,
    }
    return out


def max_ratio(err, tol):
    return float(np.max(err / tol)) if err.size else 0.0


def check_y(y_gpu, y_ref, io_dtype, rows=None, heads=None):
    g, r = y_gpu, y_ref
    if rows is not None:
        g, r = g[rows], r[rows]
    if heads is not None:
        g, r = g[:, heads[0]:heads[1]], r[:, heads[0]:heads[1]]
    if r.size == 0:
        return 0.0
    assert np.all(np.isfinite(g)), "non-finite y"
    rms = float(np.sqrt(np.mean(r ** 2)))
    if io_dtype == "bf16":
        tol = 2e-2 * rms + UNIT["bf16"] * np.abs(r)
    else:
        tol = 1e-3 * rms + 2.0 ** -23 * np.abs(r)
    ratio = max_ratio(np.abs(g - r), tol + 1e-30)
    assert ratio <= 1.0, "y error %.3g x tolerance (rms %.3g)" % (ratio, rms)
    return ratio


def check_state(h_gpu_storage, h_ref64, state_dtype):
    g = oracle.widen(h_gpu_storage, state_dtype)
    assert np.all(np.isfinite(g)), "non-finite state"
    rms = float(np.sqrt(np.mean(h_ref64 ** 2)))
    tol_rel = 1e-3 if state_dtype == "f32" else 1e-2
    tol = tol_rel * rms + UNIT[state_dtype] * np.abs(h_ref64) + 1e-30
    ratio = max_ratio(np.abs(g - h_ref64), tol)
    assert ratio <= 1.0, "state error %.3g x tolerance (rms %.3g)" % (ratio, rms)
    return ratio


def check_all(p, out, ref, heads=None):
    """Full comparison of one run against the oracle result ``ref``."""
    h0, h1 = (0, p.nheads) if heads is None else heads
    check_y(out["y"], ref["y"], p.io_dtype, heads=(h0, h1))
    named = set(int(s) for s in p.slot_idx) if p.write_final else set()
    untouched = [i for i in range(p.num_slots) if i not in named]
    # slots not written must be bit-identical
    np.testing.assert_array_equal(out["cache"][untouched], p.cache[untouched])
    if p.write_final:
        for s in range(p.num_seqs):
            slot = int(p.slot_idx[s])
            check_state(out["cache"][slot, h0:h1], ref["final"][s, h0:h1], p.state_dtype)
    if p.want_intermediate:
        for t in range(p.total_tokens):
            check_state(out["inter"][t, h0:h1], ref["inter"][t, h0:h1], p.state_dtype)

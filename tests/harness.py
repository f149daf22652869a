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


def _strided_view(idx, stride, device):
    """``idx`` as column 1 of a [S, stride] int32 block table (a strided view)."""
    torch = _torch()
    table = torch.full((len(idx), stride), -7, dtype=torch.int32)
    table[:, 1] = torch.from_numpy(np.asarray(idx, dtype=np.int32))
    return table.to(device)[:, 1]


def run_gpu(p, *, device="cuda", max_seqlen=None, status=False, chunk_size=None,
            slot_stride=1, slots_disjoint=False):
    """Run the CUDA scan on problem ``p``; returns a dict of host numpy arrays.
    ``slot_stride`` > 1 passes the slot indices as a column of a block table."""
    torch = _torch()
    from state_space_model_varlen_gb300 import binding
    d = upload(p, device)
    T, H, P, N = p.total_tokens, p.nheads, p.headdim, p.dstate
    st = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[p.state_dtype]
    y = torch.full_like(d["x"], float("nan"))
    inter = None
    if p.want_intermediate:
        inter = torch.full((T, H, P, N), float("nan"), dtype=st, device=device)
    chunks, cu_chunks = None, None
    if p.want_chunk_states:
        cuc = p.cu_chunks
        chunks = torch.full((int(cuc[-1]), H, P, N), float("nan"), dtype=st, device=device)
        cu_chunks = torch.from_numpy(cuc).to(device)
    slot_idx = d["slot_idx"] if slot_stride == 1 else _strided_view(p.slot_idx, slot_stride, device)
    final_idx = None
    if p.final_slot_idx is not None:
        final_idx = torch.from_numpy(np.asarray(p.final_slot_idx, np.int32)).to(device) \
            if slot_stride == 1 else _strided_view(p.final_slot_idx, slot_stride + 1, device)
    seed = None
    if p.sr_seed is not None:
        seed = torch.tensor([np.int64(np.uint64(p.sr_seed).astype(np.int64))], dtype=torch.int64,
                            device=device)
    dev_status = torch.zeros(1, dtype=torch.int32, device=device)
    params = binding.make_params(
        d["x"], d["dt"], d["A"], d["B"], d["C"], d["cu_seqlens"], dt_bias=d["dt_bias"], D=d["D"],
        state_cache=d["state_cache"], slot_idx=slot_idx, has_init=d["has_init"],
        write_final=p.write_final, out_y=y, out_intermediate=inter, dt_softplus=p.dt_softplus,
        chunk_size=chunk_size or p.chunk_size,
        max_seqlen=p.max_seqlen if max_seqlen is None else max_seqlen, device_status=dev_status,
        final_slot_idx=final_idx, out_chunk_states=chunks, cu_chunks=cu_chunks, sr_seed=seed,
        slots_disjoint=slots_disjoint)
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
        "chunks": None if chunks is None else _numpy(chunks, p.state_dtype),
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


def check_all(p, out, ref, heads=None, sr_err_rel=1e-4):
    """Full comparison of one run against the oracle result ``ref``."""
    h0, h1 = (0, p.nheads) if heads is None else heads
    check_y(out["y"], ref["y"], p.io_dtype, heads=(h0, h1))
    named = set(int(s) for s in p.final_slots) if p.write_final else set()
    untouched = [i for i in range(p.num_slots) if i not in named]
    # slots not written must be bit-identical
    np.testing.assert_array_equal(out["cache"][untouched], p.cache[untouched])
    if p.write_final:
        for s in range(p.num_seqs):
            slot = int(p.final_slots[s])
            if p.sr_seed is not None and p.state_dtype == "f16":
                words = oracle.sr_words(p.sr_seed, slot, (h0, h1), p.nheads, p.headdim, p.dstate)
                share = check_sr(out["cache"][slot, h0:h1], ref["final"][s, h0:h1], words,
                                 err_rel=sr_err_rel)
                print("stochastic rounding, slot %d: %.2f of the elements compared exactly"
                      % (slot, share))
            else:
                check_state(out["cache"][slot, h0:h1], ref["final"][s, h0:h1], p.state_dtype)
    if p.want_intermediate:
        for t in range(p.total_tokens):
            check_state(out["inter"][t, h0:h1], ref["inter"][t, h0:h1], p.state_dtype)
    if p.want_chunk_states:
        assert out["chunks"].shape[0] == ref["chunks"].shape[0]
        for r in range(ref["chunks"].shape[0]):
            check_state(out["chunks"][r, h0:h1], ref["chunks"][r, h0:h1], p.state_dtype)


def check_sr(g16, ref64, words, err_rel=1e-4, min_clear=0.2):
    """fp16 stochastic rounding of one written state (all elements of one slot
    row set), against the exact state ``ref64`` and the Philox words the oracle
    assigns to those elements.

    The GPU's fp32 state differs from the exact one by at most err = err_rel *
    rms(ref) (well above the scan's measured state error).  Where the exact
    value is more than err away from both fp16 grid points around it and from
    its rounding threshold lo + (word / 2^32) * spacing, the GPU must make the
    oracle's choice exactly; elsewhere it must lie within one spacing (+ err)
    of the exact value.  At least ``min_clear`` of the elements must be of the
    first kind, so the exact comparison covers most of the state."""
    g = np.asarray(g16).astype(np.float64)
    v = ref64.astype(np.float32).astype(np.float64)
    err = err_rel * float(np.sqrt(np.mean(ref64 ** 2)))
    want = oracle.sr_round_f16(v.astype(np.float32), words).astype(np.float64)
    a = np.abs(v)
    _, k = np.frexp(np.where(a > 0, a, 1.0))
    spacing = np.ldexp(1.0, np.clip(k - 1, -14, 15) - 10)
    lo = np.floor(a / spacing) * spacing
    thr = lo + (np.asarray(words, dtype=np.float64) / 2.0 ** 32) * spacing
    clear = (np.abs(a - thr) > err) & (a - lo > err) & (lo + spacing - a > err)
    assert np.all(np.isfinite(g)), "non-finite state"
    np.testing.assert_array_equal(g[clear], want[clear])
    assert np.all(np.abs(g - v) <= spacing + err), "stochastic rounding left the two neighbours"
    share = float(np.mean(clear))
    assert share >= min_clear, "only %.2f of the elements had a clear rounding decision" % share
    return share


def run_replay(p, ring, *, device="cuda"):
    """One ReplaySSM verification step on the GPU through ``ssd_replay_mtp``.
    ``ring`` as for ``oracle.replay_reference``; returns host arrays."""
    torch = _torch()
    from state_space_model_varlen_gb300 import binding
    d = upload(p, device)
    y = torch.full_like(d["x"], float("nan"))
    rx = _tensor(ring["x"], p.io_dtype, device)
    rdt = torch.from_numpy(np.ascontiguousarray(ring["dt"], dtype=np.float32)).to(device)
    rB = _tensor(ring["B"], p.io_dtype, device)
    start = torch.from_numpy(np.asarray(ring["start"], np.int32)).to(device)
    count = torch.from_numpy(np.asarray(ring["count"], np.int32)).to(device)
    start_out = torch.full_like(start, -1)
    count_out = torch.full_like(count, -1)
    seed = None
    if p.sr_seed is not None:
        seed = torch.tensor([np.int64(np.uint64(p.sr_seed).astype(np.int64))], dtype=torch.int64,
                            device=device)
    dev_status = torch.zeros(1, dtype=torch.int32, device=device)
    scan = binding.make_params(
        d["x"], d["dt"], d["A"], d["B"], d["C"], d["cu_seqlens"], dt_bias=d["dt_bias"], D=d["D"],
        state_cache=d["state_cache"], slot_idx=d["slot_idx"], write_final=False, out_y=y,
        dt_softplus=p.dt_softplus, chunk_size=p.chunk_size, max_seqlen=p.max_seqlen,
        device_status=dev_status, sr_seed=seed)
    rp = binding.make_replay_params(scan, rx, rdt, rB, ring["window"], start, count, start_out,
                                    count_out)
    binding.call_replay(rp, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return {"y": oracle.widen(_numpy(y, p.io_dtype), p.io_dtype),
            "cache": _numpy(d["state_cache"], p.state_dtype),
            "ring_x": _numpy(rx, p.io_dtype), "ring_dt": rdt.cpu().numpy(),
            "ring_B": _numpy(rB, p.io_dtype), "start": start_out.cpu().numpy(),
            "count": count_out.cpu().numpy(), "status": int(dev_status.item())}

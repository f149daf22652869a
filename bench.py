#!/usr/bin/env python3
"""Benchmark of the SSD varlen scan: tokens/s on one GB300 and the fraction of
the HBM roofline, with the fp64 CPU oracle timed beside it.

One "step" is one ``ssd_scan_varlen`` call over the whole batch of the
workload (every row of the hot path: dt softplus + chunk cumsum, chunk
states, state passing from the cache slot, chunk output, final-state
writeback).  Inputs are resident in HBM when the timed region starts; the L2
is flushed (256 MiB write) between timed steps and each step is timed with
CUDA events on the launching stream.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-per-config]

The headline workload defaults to ``varlen_prefill`` (32 packed sequences,
about 62 K tokens, the largest configuration); the same run then times every
other named configuration (dense prefill, both continued prefills, MTP, the
tiny fp32 case) with the same method and reports each under ``per_config``.

Under torchrun every rank runs its own copy of the workload (the scan shards
by sequence and head with no exchange: weak scaling, no collective on the
data path); value = tokens of all ranks / max-over-ranks time.  ``--gpus``
must equal the launcher's WORLD_SIZE.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SSD scan tokens/s (1 GB300) and % of roofline; vs CPU oracle tokens/s"
DEFAULT_WORKLOAD = "varlen_prefill"
L2_FLUSH_BYTES = 256 << 20


# ---------------------------------------------------------------------------
# algorithmic bytes / flops of one call (the roofline counts only these)
# ---------------------------------------------------------------------------
def algorithmic_bytes(p) -> int:
    io = 2 if p.io_dtype == "bf16" else 4
    st = 4 if p.state_dtype == "f32" else 2
    T, H, P, N, G, S = p.total_tokens, p.nheads, p.headdim, p.dstate, p.ngroups, p.num_seqs
    b = T * H * P * io * 2            # x read, y written
    b += T * G * N * io * 2           # B, C read
    b += T * H * 4                    # dt read
    b += H * 4 * 3 + (S + 1) * 4 + S * 4
    state = H * P * N * st
    if p.has_init is not None:
        b += int(sum(1 for v in p.has_init if v)) * state
    if p.write_final:
        b += S * state
    if p.want_intermediate:
        b += T * state
    return int(b)


def replay_bytes(p, ring) -> int:
    """Algorithmic bytes of one ReplaySSM verification step: checkpoints read,
    pending ring inputs read, window inputs read and y written, window inputs
    appended to the ring, and the checkpoints of requests that fold written."""
    io = 2 if p.io_dtype == "bf16" else 4
    st = 4 if p.state_dtype == "f32" else 2
    H, P, N, G, S = p.nheads, p.headdim, p.dstate, p.ngroups, p.num_seqs
    tok_in = H * P * io + H * 4 + G * N * io          # one token's x, dt, B
    state = H * P * N * st
    K = p.seqlens
    b = S * state                                       # checkpoints
    b += int(sum(int(c) for c in ring["count"])) * tok_in
    b += p.total_tokens * (tok_in + G * N * io + H * P * io)   # window x, dt, B, C in; y out
    b += p.total_tokens * tok_in                        # appended to the ring
    b += int(sum(1 for c, k in zip(ring["count"], K) if c + k > ring["window"])) * state
    return int(b)


TC_BLOCK = 128   # tokens per block of the tensor-core kernel, whatever chunk_size is


def algorithmic_flops(p) -> int:
    """Chunked-SSD contraction work with causal halves counted (per block and
    head: 2lNP block state + 2lNP C.h_prev + P l(l+1) masked scores.X; per
    block and group: N l(l+1) for C.B^T), for the 128-token blocks the
    tensor-core kernel runs (chunk_size only sets where checkpoint states are
    written; the scan's result does not depend on it beyond rounding)."""
    L, H, P, N, G = TC_BLOCK, p.nheads, p.headdim, p.dstate, p.ngroups
    f = 0
    for l_seq in p.seqlens:
        l_seq = int(l_seq)
        for c0 in range(0, l_seq, L):
            l = min(L, l_seq - c0)
            f += H * (4 * l * N * P + P * l * (l + 1)) + G * N * l * (l + 1)
    return int(f)


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# The sources the tensor-core scan kernel is compiled from (its translation unit
# and the headers it includes): a DRAM-traffic capture stays valid while they do.
_SCAN_KERNEL_SOURCES = ("state_space_model_varlen_gb300/csrc/sm100.cuh",
                        "state_space_model_varlen_gb300/csrc/ssd_common.cuh",
                        "state_space_model_varlen_gb300/csrc/ssd_chunked.cu",
                        "state_space_model_varlen_gb300/csrc/ssd_internal.h",
                        "include/ssd_scan.h")


def _strip_comments(text: str) -> str:
    """C/C++ source without comments and with whitespace runs collapsed (string
    and character literals kept), so that editing a comment keeps the digest."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def _kernel_source_digest() -> str:
    h = hashlib.sha256()
    for name in _SCAN_KERNEL_SOURCES:
        with open(os.path.join(ROOT, name), encoding="utf-8") as f:
            h.update(name.encode() + _strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def _traffic_per_launch(workload: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    digest = _kernel_source_digest()
    with open(path) as f:
        for line in f:
            parts = line.split("#", 1)[0].split()
            if len(parts) == 3 and parts[0] == workload and parts[1] == digest:
                return int(parts[2])
    return None


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [v.strip() for v in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        sm.sort()
        med = sm[len(sm) // 2] if sm else None
        return {"sm_mhz": med, "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# multi-rank aggregation (weak scaling: every rank runs its own batch)
# ---------------------------------------------------------------------------
def max_over_ranks(values, device=None):
    """Element-wise max of per-rank timings (identity on one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def whole_job_rate(units_per_rank, world, ms_per_step_max):
    """Units processed by all ranks per second, timed by the slowest rank."""
    return units_per_rank * world / (ms_per_step_max / 1e3)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
PER_CONFIG = ("dense_prefill", "varlen_prefill", "continued_a", "continued_b", "mtp", "mtp_replay",
              "tiny")


def _dev_tensor(a, dtype_name, dev):
    import numpy as np
    import torch
    if dtype_name == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


class _Resident:
    """One workload's inputs and outputs resident on the device, with the
    C-ABI parameter block that points at them."""

    def __init__(self, ssd, p, dev):
        import torch
        self.p = p
        T, H, P, N = p.total_tokens, p.nheads, p.headdim, p.dstate
        self.x = _dev_tensor(p.x, p.io_dtype, dev)
        self.B = _dev_tensor(p.B, p.io_dtype, dev)
        self.C = _dev_tensor(p.C, p.io_dtype, dev)
        self.dt = torch.from_numpy(p.dt).to(dev)
        A = torch.from_numpy(p.A).to(dev)
        D = None if p.D is None else torch.from_numpy(p.D).to(dev)
        bias = None if p.dt_bias is None else torch.from_numpy(p.dt_bias).to(dev)
        cu = torch.from_numpy(p.cu_seqlens).to(dev)
        self.slots = torch.from_numpy(p.slot_idx).to(dev)
        has_init = None if p.has_init is None else torch.from_numpy(p.has_init).to(dev)
        self.cache = _dev_tensor(p.cache, p.state_dtype, dev)
        self.y = torch.empty_like(self.x)
        st_t = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[p.state_dtype]
        self.inter = torch.empty((T, H, P, N), dtype=st_t, device=dev) if p.want_intermediate else None
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self._keep = (A, D, bias, cu, has_init)
        self.params = ssd.make_params(
            self.x, self.dt, A, self.B, self.C, cu, dt_bias=bias, D=D, state_cache=self.cache,
            slot_idx=self.slots, has_init=has_init, write_final=p.write_final, out_y=self.y,
            out_intermediate=self.inter, dt_softplus=p.dt_softplus, chunk_size=p.chunk_size,
            max_seqlen=p.max_seqlen, device_status=self.status,
            # each sequence owns its slot (the serving case): the caller says so,
            # which spares the snapshot of initial states
            slots_disjoint=p.final_slot_idx is None and len(set(p.slot_idx.tolist())) == p.num_seqs)
        need = ssd.workspace_size(self.params)
        self.ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        self.params.workspace, self.params.workspace_bytes = self.ws.data_ptr(), self.ws.numel()
        self.launches = ssd.num_launches(self.params)
        self.path = ssd.kernel_path(self.params)

    def twin(self, ssd):
        """A second set of per-step buffers (x, B, C, dt, y, intermediate
        states, workspace, status) over the same state cache and parameters,
        for pipelined end-to-end steps."""
        import copy
        import torch
        t = copy.copy(self)
        t.x, t.B, t.C = torch.empty_like(self.x), torch.empty_like(self.B), torch.empty_like(self.C)
        t.dt, t.y = torch.empty_like(self.dt), torch.empty_like(self.y)
        t.inter = None if self.inter is None else torch.empty_like(self.inter)
        t.status = torch.zeros_like(self.status)
        t.ws = torch.empty_like(self.ws)
        q = type(self.params).from_buffer_copy(self.params)
        q.x, q.B, q.C, q.dt, q.out_y = (t.x.data_ptr(), t.B.data_ptr(), t.C.data_ptr(), t.dt.data_ptr(),
                                        t.y.data_ptr())
        q.out_intermediate = None if t.inter is None else t.inter.data_ptr()
        q.workspace, q.device_status = t.ws.data_ptr(), t.status.data_ptr()
        t.params = q
        return t


class _ResidentReplay(_Resident):
    """The MTP windows plus rings on the device, verified with ssd_replay_mtp."""

    def __init__(self, ssd, p, dev):
        import torch
        from state_space_model_varlen_gb300 import workloads as W
        super().__init__(ssd, p, dev)
        self.ring = W.replay_ring(p, seed=40)
        self.rx = _dev_tensor(self.ring["x"], p.io_dtype, dev)
        self.rdt = torch.from_numpy(self.ring["dt"]).to(dev)
        self.rB = _dev_tensor(self.ring["B"], p.io_dtype, dev)
        self.rstart = torch.from_numpy(self.ring["start"]).to(dev)
        self.rcount = torch.from_numpy(self.ring["count"]).to(dev)
        self.rstart_out = torch.empty_like(self.rstart)
        self.rcount_out = torch.empty_like(self.rcount)
        self.params.write_final = 0
        self.params.has_init = None
        self.replay = ssd.make_replay_params(self.params, self.rx, self.rdt, self.rB,
                                             self.ring["window"], self.rstart, self.rcount,
                                             self.rstart_out, self.rcount_out)
        self.launches, self.path = 1, "replay"
        self._ssd = ssd

    def twin(self, ssd):
        t = super().twin(ssd)
        t.replay = ssd.make_replay_params(t.params, self.rx, self.rdt, self.rB, self.ring["window"],
                                          self.rstart, self.rcount, self.rstart_out, self.rcount_out)
        return t

    def call(self, sptr):
        self._ssd.call_replay(self.replay, sptr)


def _call(ssd, r, sptr):
    if isinstance(r, _ResidentReplay):
        r.call(sptr)
    else:
        ssd.call(r.params, sptr)


def _capture(ssd, r):
    """The call captured once in a CUDA graph (the library enqueues kernels only,
    so a call can be captured); None if capture is not possible here."""
    import torch
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            _call(ssd, r, torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        return g
    except Exception:                       # noqa: BLE001 -- fall back to direct calls
        torch.cuda.synchronize()
        return None


def _time_device(ssd, r, stream, steps, warmup, flush, local_rank, world):
    """Device time of ``steps`` calls (CUDA events on the launching stream, L2
    flushed between calls), with the SM clocks sampled meanwhile.  Each call is
    a replay of one C-ABI call captured in a CUDA graph, so the host's argument
    marshalling and launch latency (tens of microseconds) do not leave the GPU
    idle inside the timed region of a short call; direct calls if capture fails.
    Returns (total ms, clocks, wall s, how the calls were launched)."""
    import torch
    sptr = stream.cuda_stream
    for _ in range(warmup):
        _call(ssd, r, sptr)
    torch.cuda.synchronize()
    if int(r.status.item()) != 0:
        raise RuntimeError("device status %d after warm-up" % int(r.status.item()))
    graph = _capture(ssd, r)
    if graph is not None:
        graph.replay()
        torch.cuda.synchronize()
        if int(r.status.item()) != 0:
            raise RuntimeError("device status %d after a graph replay" % int(r.status.item()))
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    sampler = ClockSampler(local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.25)                      # let the sampler take its first reading
    t_wall = time.perf_counter()
    for i in range(steps):
        flush.fill_(i)                    # L2 flush (outside the events)
        starts[i].record(stream)
        if graph is not None:
            graph.replay()
        else:
            _call(ssd, r, sptr)
        ends[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    clocks = sampler.stop()
    if world > 1:
        torch.distributed.barrier()
    total_ms = float(sum(s.elapsed_time(e) for s, e in zip(starts, ends)))
    return total_ms, clocks, wall, ("cuda graph replay" if graph is not None else "direct C-ABI call")


def _roofline_entry(p, ms_per_step, b=None):
    hbm_peak, _, peak_kind = _peaks()
    b = algorithmic_bytes(p) if b is None else b
    achieved = b / (ms_per_step / 1e3) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
            "frac": achieved / hbm_peak, "peak_kind": peak_kind + " (burst copy)",
            "algorithmic_bytes_per_launch": b}


def run_ours(args, rank, world, local_rank):
    import torch
    import state_space_model_varlen_gb300 as ssd
    from state_space_model_varlen_gb300 import workloads as W

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    ssd.load()
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    p = W.workload(args.workload)
    T = p.total_tokens
    replay = args.workload == "mtp_replay"
    r = _ResidentReplay(ssd, p, dev) if replay else _Resident(ssd, p, dev)
    launches, path = r.launches, r.path
    replay_b = replay_bytes(p, r.ring) if replay else None
    total_ms, clocks, wall, how = _time_device(ssd, r, stream, args.steps, args.warmup, flush,
                                               local_rank, world)

    # ---- end to end through the C ABI with host buffers --------------------
    # Every step copies its inputs from pinned host memory, makes the C-ABI
    # call and reads its results back (y, and the final states gathered from
    # the cache, or the per-token states).  Steps are pipelined as a serving
    # loop would: two sets of device buffers over one state cache, the inputs
    # of step i+1 going up on an upload stream while step i computes and its
    # results come down on a third stream (the host link carries both
    # directions at once); every step's copies are inside the timed region.
    sets = [r, r.twin(ssd)]
    params, sptr = r.params, stream.cuda_stream
    pin = lambda t: t.cpu().pin_memory()
    hx, hB, hC, hdt = pin(r.x), pin(r.B), pin(r.C), pin(r.dt)
    hy = torch.empty(r.y.shape, dtype=r.y.dtype, pin_memory=True)
    write_final = p.write_final and not replay
    slots64 = r.slots.long()
    if write_final:
        hfinal = torch.empty((p.num_seqs,) + tuple(r.cache.shape[1:]), dtype=r.cache.dtype, pin_memory=True)
        finals = [torch.empty(hfinal.shape, dtype=r.cache.dtype, device=dev) for _ in sets]
    h2d = sum(t.numel() * t.element_size() for t in (hx, hB, hC, hdt))
    d2h = hy.numel() * hy.element_size() + (hfinal.numel() * hfinal.element_size() if write_final else 0)
    if r.inter is not None:
        hinter = torch.empty(r.inter.shape, dtype=r.inter.dtype, pin_memory=True)
        d2h += hinter.numel() * hinter.element_size()
    e2e_steps = max(3, min(args.steps, 20))
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    uploaded = [torch.cuda.Event() for _ in sets]
    computed = [torch.cuda.Event() for _ in sets]
    read = [None for _ in sets]

    def e2e_step(i):
        k = i % len(sets)
        b = sets[k]
        with torch.cuda.stream(up):
            if read[k] is not None:
                up.wait_event(read[k])             # set k's step of two steps ago is computed and down
            b.x.copy_(hx, non_blocking=True)
            b.B.copy_(hB, non_blocking=True)
            b.C.copy_(hC, non_blocking=True)
            b.dt.copy_(hdt, non_blocking=True)
            uploaded[k].record(up)
        stream.wait_event(uploaded[k])
        _call(ssd, b, sptr)
        if write_final:
            torch.index_select(b.cache, 0, slots64, out=finals[k])
        computed[k].record(stream)
        down.wait_event(computed[k])
        with torch.cuda.stream(down):
            hy.copy_(b.y, non_blocking=True)
            if write_final:
                hfinal.copy_(finals[k], non_blocking=True)
            if b.inter is not None:
                hinter.copy_(b.inter, non_blocking=True)
            read[k] = torch.cuda.Event()
            read[k].record(down)

    for i in range(2):                    # untimed: first-use costs of the copy path
        e2e_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    up.wait_stream(stream)                    # the timed uploads start after e0
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_stream(down)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    for b in sets:
        if int(b.status.item()) != 0:
            raise RuntimeError("device status %d in the end-to-end steps" % int(b.status.item()))
    del r, sets, hx, hB, hC, hdt, hy, params
    torch.cuda.empty_cache()

    # ---- every other config of the task, same method ------------------------
    per_config = {}
    if not args.no_per_config:
        pc_steps = max(3, min(args.steps, args.per_config_steps))
        for name in PER_CONFIG:
            if name == args.workload:
                continue
            q = W.workload(name)
            rq = _ResidentReplay(ssd, q, dev) if name == "mtp_replay" else _Resident(ssd, q, dev)
            ms, ck, _, pc_how = _time_device(ssd, rq, stream, pc_steps, args.warmup, flush, local_rank, world)
            per_config[name] = {"ms": ms, "steps": pc_steps, "clocks": ck, "problem": q,
                                "launches": rq.launches, "path": rq.path, "how": pc_how,
                                "bytes": replay_bytes(q, rq.ring) if name == "mtp_replay" else None}
            del rq
            torch.cuda.empty_cache()

    # ---- max over ranks ------------------------------------------------------
    names = sorted(per_config)
    vals = max_over_ranks([total_ms, e2e_ms] + [per_config[n]["ms"] for n in names], dev)
    total_ms, e2e_ms = vals[0], vals[1]
    for n, v in zip(names, vals[2:]):
        per_config[n]["ms"] = v
    if rank != 0:
        return None

    ms_per_step = total_ms / args.steps
    tokens_all = T * world
    value = whole_job_rate(T, world, ms_per_step)
    _, tc_peak, _ = _peaks()
    bytes_per_call = replay_b if replay else algorithmic_bytes(p)
    roof = _roofline_entry(p, ms_per_step, bytes_per_call)
    roof.update({
        "traffic": None if replay else _traffic_per_launch(args.workload),
        "algorithmic_flops_per_launch": algorithmic_flops(p),
        "tensor_time_at_peak_us": algorithmic_flops(p) / (tc_peak * 1e12) * 1e6,
        "hbm_time_at_peak_us": bytes_per_call / (roof["peak"] * 1e9) * 1e6,
        "note": "achieved = algorithmic bytes / device time of the whole call "
                "(%d launch(es)); a lower bound for the dominant kernel" % launches,
    })
    pc_out = {}
    for n in names:
        e = per_config[n]
        q, ms = e["problem"], e["ms"] / e["steps"]
        pc_out[n] = {"value": whole_job_rate(q.total_tokens, world, ms), "unit": "tokens/s",
                     "ms_per_step": ms, "steps": e["steps"], "kernel_path": e["path"],
                     "launches_per_call": e["launches"], "tokens": q.total_tokens,
                     "launched_as": e["how"],
                     "roofline": _roofline_entry(q, ms, e["bytes"]), "clocks": e["clocks"]}
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if path == "chunked_tc" else "f32",
        "data": "synthetic (seeded, distributions of the workload recipe)",
        "config": {
            "workload": args.workload, "tokens": T, "seqs": p.num_seqs, "nheads": p.nheads,
            "headdim": p.headdim, "dstate": p.dstate, "ngroups": p.ngroups,
            "chunk_size": p.chunk_size, "io_dtype": p.io_dtype, "state_dtype": p.state_dtype,
            "kernel_path": path,
            "parallelism": "replicas x%d (independent batches, no collective)" % world,
            "l2": "flushed between timed steps (256 MiB write); working set %.0f MB"
                  % (bytes_per_call / 1e6),
            "timed_call": how,
        },
        "roofline": roof,
        "e2e": {
            "value": tokens_all / (e2e_ms / 1e3),
            "unit": "tokens/s",
            "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h),
            "how": "C-ABI call per step with its inputs copied up from pinned host memory and its "
                   "results read back; steps pipelined over two device buffer sets and one state "
                   "cache (step i+1's upload overlaps step i's call and readback)",
        },
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
        "wall_s_timed_region": wall,
        "per_config": pc_out,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(p, args.cpu_seconds)
    return line


# ---------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------
def _oracle_calibrate(p):
    """Seconds per token and head of the fp64 oracle on this host, from a head
    slice of the first non-empty sequence of ``p``."""
    import oracle
    from state_space_model_varlen_gb300 import workloads as W
    threads = oracle.max_threads()
    first = next(s for s in range(p.num_seqs) if p.seqlens[s] > 0)
    q = W.select_sequences(p, [first], compact=True)
    h1 = max(1, min(p.nheads, threads))
    t = time.perf_counter()
    oracle.ssd_scan_reference(q, heads=(0, h1))
    return (time.perf_counter() - t) / (int(p.seqlens[first]) * h1)


def _oracle_sample(p, target_s, per_tok_head=None):
    """Time the fp64 oracle on a bounded sample of ``p`` sized to ~target_s
    seconds: the first sequences, or, where even one sequence would take
    longer, a prefix of the first; all heads.  Returns (tokens, seconds,
    threads, sequences, passes, heads)."""
    import oracle
    from state_space_model_varlen_gb300 import workloads as W
    threads = oracle.max_threads()
    if per_tok_head is None:
        per_tok_head = _oracle_calibrate(p)
    budget = target_s / max(per_tok_head, 1e-12)          # token-heads
    first = next(s for s in range(p.num_seqs) if p.seqlens[s] > 0)
    if budget < int(p.seqlens[first]) * p.nheads:
        # all heads of as long a prefix of the first sequence as the budget
        # holds (the oracle converts every head's inputs whatever slice it
        # scans, so a head slice would count less work than it does)
        ntok = int(min(int(p.seqlens[first]), max(16, budget // p.nheads)))
        q = W.sequence_prefix(p, first, ntok)
        t = time.perf_counter()
        oracle.ssd_scan_reference(q)
        el = time.perf_counter() - t
        return q.total_tokens, el, threads, 1, 1, p.nheads
    chosen, tok = [], 0
    for s in range(p.num_seqs):
        if tok * p.nheads >= budget and chosen:
            break
        chosen.append(s)
        tok += int(p.seqlens[s])
    q = W.select_sequences(p, chosen, compact=True)
    # the whole workload may take well under target_s: repeat it until the
    # sample spans most of the budget, so the rate is not a single short run
    passes, el = 0, 0.0
    while passes == 0 or (len(chosen) == p.num_seqs and el < 0.7 * target_s):
        t = time.perf_counter()
        oracle.ssd_scan_reference(q)
        el += time.perf_counter() - t
        passes += 1
    return q.total_tokens * passes, el, threads, len(chosen), passes, p.nheads


def cpu_baseline(p, target_s):
    tok, el, threads, nseq, passes, _ = _oracle_sample(p, target_s)
    return {"value": tok / el, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": "%d of %d sequences (all %d heads) of workload %s, %d pass(es), %d tokens, fp64, %.1f s"
                      % (nseq, p.num_seqs, p.nheads, p.name, passes, tok, el)}


def run_reference(args, rank):
    from state_space_model_varlen_gb300 import workloads as W
    if rank != 0:
        return None
    p = W.workload(args.workload)
    # the whole run (warm-up and timed steps) takes about four times
    # --cpu-seconds of host time, or 0.1 s a step where that is longer (so that
    # the oracle's per-call overhead stays a small part of each step)
    rate = _oracle_calibrate(p)
    per_step = max(0.1, 4.0 * args.cpu_seconds / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        _oracle_sample(p, per_step, rate)
    tok_total, el_total, threads, nseq, heads = 0.0, 0.0, 0, 0, 0
    for _ in range(args.steps):
        tok, el, threads, nseq, _, heads = _oracle_sample(p, per_step, rate)
        tok_total += tok
        el_total += el
    value = tok_total / el_total
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el_total / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, distributions of the workload recipe)",
        "config": {"workload": args.workload, "tokens": p.total_tokens, "nheads": p.nheads,
                   "headdim": p.headdim, "dstate": p.dstate, "ngroups": p.ngroups,
                   "chunk_size": p.chunk_size, "io_dtype": p.io_dtype,
                   "state_dtype": p.state_dtype},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": "%d of %d sequences (or a prefix of the first) per step, "
                                   "all %d heads, fp64" % (nseq, p.num_seqs, heads)},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only --workload, not the other configs")
    ap.add_argument("--per-config-steps", type=int, default=20)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        raise SystemExit("--gpus %d but WORLD_SIZE=%d: launch N>1 under torch.distributed.run "
                         "with --nproc-per-node N" % (args.gpus, world))
    if args.impl == "reference":
        line = run_reference(args, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    line = run_ours(args, rank, world, local_rank)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

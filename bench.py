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
                    [--impl ours|reference]

Under torchrun every rank runs its own copy of the workload (the scan shards
by sequence and head with no exchange: weak scaling, no collective on the
data path); value = tokens of all ranks / max-over-ranks time.
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
DEFAULT_WORKLOAD = "dense_prefill"
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


def algorithmic_flops(p) -> int:
    """Chunked-SSD contraction work with causal halves counted (per chunk and
    head: 2lNP chunk state + 2lNP C.h_prev + P l(l+1) masked scores.X; per
    chunk and group: N l(l+1) for C.B^T)."""
    L, H, P, N, G = p.chunk_size, p.nheads, p.headdim, p.dstate, p.ngroups
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
def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch
    import state_space_model_varlen_gb300 as ssd
    from state_space_model_varlen_gb300 import workloads as W

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    ssd.load()
    p = W.workload(args.workload)
    T, H, P, N = p.total_tokens, p.nheads, p.headdim, p.dstate

    def dev_t(a, dtype_name):
        if dtype_name == "bf16":
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    x = dev_t(p.x, p.io_dtype)
    B = dev_t(p.B, p.io_dtype)
    C = dev_t(p.C, p.io_dtype)
    dt = torch.from_numpy(p.dt).to(dev)
    A = torch.from_numpy(p.A).to(dev)
    D = None if p.D is None else torch.from_numpy(p.D).to(dev)
    bias = None if p.dt_bias is None else torch.from_numpy(p.dt_bias).to(dev)
    cu = torch.from_numpy(p.cu_seqlens).to(dev)
    slots = torch.from_numpy(p.slot_idx).to(dev)
    has_init = None if p.has_init is None else torch.from_numpy(p.has_init).to(dev)
    cache = dev_t(p.cache, p.state_dtype)
    y = torch.empty_like(x)
    st_t = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[p.state_dtype]
    inter = torch.empty((T, H, P, N), dtype=st_t, device=dev) if p.want_intermediate else None
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    params = ssd.make_params(x, dt, A, B, C, cu, dt_bias=bias, D=D, state_cache=cache,
                             slot_idx=slots, has_init=has_init, write_final=p.write_final,
                             out_y=y, out_intermediate=inter, dt_softplus=p.dt_softplus,
                             chunk_size=p.chunk_size, max_seqlen=p.max_seqlen,
                             device_status=status)
    need = ssd.workspace_size(params)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    params.workspace, params.workspace_bytes = ws.data_ptr(), ws.numel()
    launches = ssd.num_launches(params)
    path = ssd.kernel_path(params)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    for _ in range(args.warmup):
        ssd.call(params, sptr)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("device status %d after warm-up" % int(status.item()))

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.25)                      # let the sampler take its first reading
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i)                    # L2 flush (outside the events)
        starts[i].record(stream)
        ssd.call(params, sptr)
        ends[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    clocks = sampler.stop()
    if world > 1:
        torch.distributed.barrier()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = float(sum(step_ms))

    # ---- end to end through the C ABI with host buffers --------------------
    pin = lambda t: t.cpu().pin_memory()
    hx, hB, hC, hdt = pin(x), pin(B), pin(C), pin(dt)
    hy = torch.empty(y.shape, dtype=y.dtype, pin_memory=True)
    if p.write_final:
        hfinal = torch.empty((p.num_seqs,) + tuple(cache.shape[1:]), dtype=cache.dtype,
                             pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in (hx, hB, hC, hdt))
    d2h = hy.numel() * hy.element_size() + (hfinal.numel() * hfinal.element_size()
                                            if p.write_final else 0)
    if inter is not None:
        hinter = torch.empty(inter.shape, dtype=inter.dtype, pin_memory=True)
        d2h += hinter.numel() * hinter.element_size()
    e2e_steps = max(3, min(args.steps, 20))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    slots64 = slots.long()

    def e2e_step():
        x.copy_(hx, non_blocking=True)
        B.copy_(hB, non_blocking=True)
        C.copy_(hC, non_blocking=True)
        dt.copy_(hdt, non_blocking=True)
        ssd.call(params, sptr)
        hy.copy_(y, non_blocking=True)
        if p.write_final:
            hfinal.copy_(cache.index_select(0, slots64), non_blocking=True)
        if inter is not None:
            hinter.copy_(inter, non_blocking=True)

    for _ in range(2):                    # untimed: first-use costs of the copy path
        e2e_step()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps

    # ---- max over ranks ------------------------------------------------------
    total_ms, e2e_ms = max_over_ranks([total_ms, e2e_ms], dev)
    if rank != 0:
        return None

    ms_per_step = total_ms / args.steps
    tokens_all = T * world
    value = whole_job_rate(T, world, ms_per_step)
    hbm_peak, tc_peak, peak_kind = _peaks()
    bytes_per_call = algorithmic_bytes(p)
    achieved_gbs = bytes_per_call / (ms_per_step / 1e3) / 1e9
    traffic = _traffic_per_launch(args.workload)
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
            "workload": args.workload, "tokens": T, "seqs": p.num_seqs, "nheads": H,
            "headdim": P, "dstate": N, "ngroups": p.ngroups, "chunk_size": p.chunk_size,
            "io_dtype": p.io_dtype, "state_dtype": p.state_dtype, "kernel_path": path,
            "parallelism": "replicas x%d (independent batches, no collective)" % world,
            "l2": "flushed between timed steps (256 MiB write); working set %.0f MB"
                  % (bytes_per_call / 1e6),
        },
        "roofline": {
            "bound": "hbm",
            "achieved": achieved_gbs,
            "peak": hbm_peak,
            "unit": "GB/s",
            "frac": achieved_gbs / hbm_peak,
            "traffic": traffic,
            "peak_kind": peak_kind + " (burst copy)",
            "algorithmic_bytes_per_launch": bytes_per_call,
            "algorithmic_flops_per_launch": algorithmic_flops(p),
            "tensor_time_at_peak_us": algorithmic_flops(p) / (tc_peak * 1e12) * 1e6,
            "hbm_time_at_peak_us": bytes_per_call / (hbm_peak * 1e9) * 1e6,
            "note": "achieved = algorithmic bytes / device time of the whole call "
                    "(%d launch(es)); a lower bound for the dominant kernel" % launches,
        },
        "e2e": {
            "value": tokens_all / (e2e_ms / 1e3),
            "unit": "tokens/s",
            "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h),
        },
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
        "wall_s_timed_region": wall,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(p, args.cpu_seconds)
    return line


# ---------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------
def _oracle_sample(p, target_s):
    """Time the fp64 oracle on a bounded sample of ``p``: the first sequences,
    all heads, sized from a short calibration run to ~target_s seconds."""
    import numpy as np
    import oracle
    from state_space_model_varlen_gb300 import workloads as W
    threads = oracle.max_threads()
    order = list(range(p.num_seqs))
    # calibration: a head slice of the first non-empty sequence
    first = next(s for s in order if p.seqlens[s] > 0)
    q = W.select_sequences(p, [first])
    h1 = max(1, min(p.nheads, threads))
    t = time.perf_counter()
    oracle.ssd_scan_reference(q, heads=(0, h1))
    per_tok_head = (time.perf_counter() - t) / (int(p.seqlens[first]) * h1)
    budget_tok = target_s / max(per_tok_head, 1e-12) / p.nheads
    chosen, tok = [], 0
    for s in order:
        if tok >= budget_tok and chosen:
            break
        chosen.append(s)
        tok += int(p.seqlens[s])
    q = W.select_sequences(p, chosen)
    # the whole workload may take well under target_s: repeat it until the
    # sample spans most of the budget, so the rate is not a single short run
    passes, el = 0, 0.0
    while passes == 0 or (len(chosen) == p.num_seqs and el < 0.7 * target_s):
        t = time.perf_counter()
        oracle.ssd_scan_reference(q)
        el += time.perf_counter() - t
        passes += 1
    return q.total_tokens * passes, el, threads, len(chosen), passes


def cpu_baseline(p, target_s):
    tok, el, threads, nseq, passes = _oracle_sample(p, target_s)
    return {"value": tok / el, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": "%d of %d sequences (all %d heads) of workload %s, %d pass(es), %d tokens, fp64, %.1f s"
                      % (nseq, p.num_seqs, p.nheads, p.name, passes, tok, el)}


def run_reference(args, rank):
    from state_space_model_varlen_gb300 import workloads as W
    if rank != 0:
        return None
    p = W.workload(args.workload)
    per_step = max(2.0, args.cpu_seconds / max(1, args.steps + args.warmup) * 2)
    for _ in range(args.warmup):
        _oracle_sample(p, per_step / 4)
    tok_total, el_total, threads, nseq = 0, 0.0, 0, 0
    for _ in range(args.steps):
        tok, el, threads, nseq, _ = _oracle_sample(p, per_step)
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
                         "sample": "%d of %d sequences per step, all heads, fp64"
                                   % (nseq, p.num_seqs)},
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
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
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

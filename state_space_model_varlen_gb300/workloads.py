"""Seeded synthetic inputs for the Mamba2 SSD varlen scan.

This module only draws numbers.  It holds none of the scan's arithmetic, so
both the fp64 oracle (under ``oracle/``) and the CUDA path can consume the
very same values without sharing any code of the method itself.

Input recipe (the pages give no dataset or weights; these distributions stand
in for the Nemotron/Granite prefill and MTP workloads they describe):

* ``x ~ N(0, 1)``
* ``dt_raw ~ N(0, 1)`` clipped to [-2.3, 2.3]; ``dt_bias_h = ln(expm1(0.01))``
  for every head, so ``softplus(dt_raw + dt_bias)`` lies in [1.0e-3, 0.0956]
* ``A_h = -exp(U(ln 1, ln 16))``  (so A in [-16, -1])
* ``B, C ~ N(0, 1) / sqrt(d_state)``
* ``D ~ N(0, 1)``
* state-cache slots: ``N(0, cache_std)``

Draw order for one problem: lengths -> slots -> A -> dt_bias -> D -> dt_raw ->
x -> B -> C -> cache.  Values are drawn in float64, rounded once to float32
and, for bf16/fp16 tensors, rounded to nearest-even from that float32.  bf16
tensors are carried as their uint16 bit patterns.

The named workloads follow the shapes of the pages: head dim 64 / state 128
(the shapes the FlashInfer fused SSD scan compiles, vLLM PR #61501
"Details"), continued-prefill suffixes [32, 600, 1600] from a bf16 cache
(vLLM PR #62922 "Serving performance"), and 1 + 2 speculative tokens per
request for MTP verification (vLLM PR #52928 "Summary").
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

DT_BIAS = math.log(math.expm1(0.01))   # inverse softplus of 0.01
DT_CLIP = 2.3


# ----------------------------------------------------------------------------
# dtype helpers (storage only)
# ----------------------------------------------------------------------------
def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest-even); return the uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def to_storage(a64: np.ndarray, dtype: str) -> np.ndarray:
    """Store float64 draws in ``dtype`` ('f32', 'bf16' as uint16 bits, 'f16')."""
    a32 = a64 if (isinstance(a64, np.ndarray) and a64.dtype == np.float32) else \
        np.asarray(a64, dtype=np.float64).astype(np.float32)
    if dtype == "f32":
        return a32
    if dtype == "bf16":
        return f32_to_bf16_bits(a32)
    if dtype == "f16":
        return a32.astype(np.float16)
    raise ValueError(dtype)


def storage_to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16_bits_to_f32(a).astype(np.float64)
    return np.asarray(a).astype(np.float64)


# ----------------------------------------------------------------------------
# problem container
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class Problem:
    name: str
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    chunk_size: int
    io_dtype: str            # x, B, C, y
    state_dtype: str         # state cache and intermediate states
    cu_seqlens: np.ndarray   # int32 [S+1]
    x: np.ndarray            # [T, H, P]   io_dtype storage
    dt: np.ndarray           # float32 [T, H] (raw, before bias/softplus)
    dt_bias: Optional[np.ndarray]  # float32 [H]
    dt_softplus: int
    A: np.ndarray            # float32 [H]
    B: np.ndarray            # [T, G, N]   io_dtype storage
    C: np.ndarray            # [T, G, N]   io_dtype storage
    D: Optional[np.ndarray]  # float32 [H]
    cache: np.ndarray        # [num_slots, H, P, N] state_dtype storage
    slot_idx: np.ndarray     # int32 [S]
    has_init: Optional[np.ndarray]  # uint8 [S]
    write_final: int
    want_intermediate: int
    # optional parts of the call (defaults: the plain scan)
    final_slot_idx: Optional[np.ndarray] = None   # int32 [S]: where final states go (None: slot_idx)
    want_chunk_states: int = 0                    # also return the state at every chunk boundary
    sr_seed: Optional[int] = None                 # fp16 cache writes with stochastic rounding

    @property
    def num_seqs(self) -> int:
        return int(self.cu_seqlens.shape[0] - 1)

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def num_slots(self) -> int:
        return int(self.cache.shape[0])

    @property
    def seqlens(self) -> np.ndarray:
        return np.diff(self.cu_seqlens.astype(np.int64))

    @property
    def max_seqlen(self) -> int:
        return int(self.seqlens.max()) if self.num_seqs else 0

    @property
    def final_slots(self) -> np.ndarray:
        return self.slot_idx if self.final_slot_idx is None else self.final_slot_idx

    @property
    def cu_chunks(self) -> np.ndarray:
        return chunk_offsets(self.seqlens, self.chunk_size)


def chunk_offsets(seqlens, chunk_size) -> np.ndarray:
    """int32 [S+1]: first checkpoint row of each sequence, ceil(len / chunk_size)
    rows per sequence (the layout of the per-chunk state output)."""
    lens = np.asarray(seqlens, dtype=np.int64)
    out = np.zeros(lens.shape[0] + 1, dtype=np.int64)
    out[1:] = np.cumsum((lens + chunk_size - 1) // chunk_size)
    return out.astype(np.int32)


def make_problem(seqlens, *, nheads, headdim, dstate, ngroups=1, chunk_size=128,
                 io_dtype="bf16", state_dtype="f32", num_slots=None, slots=None,
                 has_init=False, write_final=True, want_intermediate=False,
                 dt_softplus=True, with_dt_bias=True, with_D=True, cache_std=1.0,
                 seed=0, name="custom", rng=None) -> Problem:
    """Draw one problem.  ``slots`` is an explicit slot list or None (random distinct)."""
    rng = np.random.default_rng(seed) if rng is None else rng
    seqlens = np.asarray(seqlens, dtype=np.int64)
    S = int(seqlens.shape[0])
    H, P, N, G = nheads, headdim, dstate, ngroups
    cu = np.zeros(S + 1, dtype=np.int64)
    cu[1:] = np.cumsum(seqlens)
    T = int(cu[-1])
    if num_slots is None:
        num_slots = max(S, 1)
    # slots
    if slots is None:
        slot_idx = rng.permutation(num_slots)[:S].astype(np.int32)
    else:
        slot_idx = np.asarray(slots, dtype=np.int32)
    A = -np.exp(rng.uniform(math.log(1.0), math.log(16.0), size=H))
    dt_bias = np.full(H, DT_BIAS) if with_dt_bias else None
    D = rng.standard_normal(H) if with_D else None
    dt_raw = np.clip(rng.standard_normal((T, H)), -DT_CLIP, DT_CLIP)
    x = rng.standard_normal((T, H, P))
    B = rng.standard_normal((T, G, N)) / math.sqrt(N)
    C = rng.standard_normal((T, G, N)) / math.sqrt(N)
    cache = rng.standard_normal((num_slots, H, P, N), dtype=np.float64 if num_slots * H * P * N < (1 << 26) else np.float32) * cache_std
    hi = np.ones(S, dtype=np.uint8) if has_init is True else (
        None if has_init is False else np.asarray(has_init, dtype=np.uint8))
    return Problem(
        name=name, nheads=H, headdim=P, dstate=N, ngroups=G, chunk_size=chunk_size,
        io_dtype=io_dtype, state_dtype=state_dtype,
        cu_seqlens=cu.astype(np.int32),
        x=to_storage(x, io_dtype), dt=dt_raw.astype(np.float32),
        dt_bias=None if dt_bias is None else dt_bias.astype(np.float32),
        dt_softplus=int(bool(dt_softplus)), A=A.astype(np.float32),
        B=to_storage(B, io_dtype), C=to_storage(C, io_dtype),
        D=None if D is None else D.astype(np.float32),
        cache=to_storage(cache, state_dtype), slot_idx=slot_idx, has_init=hi,
        write_final=int(bool(write_final)), want_intermediate=int(bool(want_intermediate)))


# ----------------------------------------------------------------------------
# the named workloads
# ----------------------------------------------------------------------------
WORKLOADS = {
    "tiny": "1 seq x 256 tokens, H4 P16 N16 G1, chunk 64, fp32 everywhere, final state -> slot 2 of 4",
    "dense_prefill": "8 x 2048 tokens, H80 P64 N128 G1, chunk 256, bf16 x/B/C/y, fp32 dt/A/D/state, final -> 8 fp32 slots",
    "varlen_prefill": "32 seqs len U{1..4096} (2 forced < 128), H128 P64 N128 G8, chunk 128, bf16 I/O, fp32 state, final -> 32 of 512 fp32 slots",
    "continued_a": "1 seq x 32 tokens from a bf16 512-slot cache (N(0,0.1)), H128 P64 N128 G8, in-place writeback",
    "continued_b": "3 seqs [32, 600, 1600] from a bf16 512-slot cache (N(0,0.1)), H128 P64 N128 G8, in-place writeback",
    "mtp": "128 requests x 3 tokens from a 512-slot fp32 cache (N(0,0.1)), H128 P64 N128 G8, per-token states, no writeback",
    "mtp_replay": "the mtp windows verified ReplaySSM-style: checkpoints in the 512-slot fp32 cache, "
                  "rings of 11 positions (window 8) holding 0-8 pending accepted tokens per request",
}

REPLAY_CAPACITY = 11     # ring positions per slot: the logical window plus one window of 3
REPLAY_WINDOW = 8


def replay_ring(p: Problem, seed: int, capacity: int = REPLAY_CAPACITY, window: int = REPLAY_WINDOW):
    """Seeded ring contents for ``p``'s slots (draws only): raw x, dt, B of
    ``capacity`` positions per slot with the recipe's distributions, a random
    start and a pending count uniform in [0, window] per request."""
    rng = np.random.default_rng(seed)
    n = p.num_slots * capacity
    H, P, N, G = p.nheads, p.headdim, p.dstate, p.ngroups
    x = rng.standard_normal((n, H, P), dtype=np.float32)
    dt = np.clip(rng.standard_normal((n, H), dtype=np.float32), -DT_CLIP, DT_CLIP)
    B = rng.standard_normal((n, G, N), dtype=np.float32) / np.float32(math.sqrt(N))
    return {"x": to_storage(x, p.io_dtype).reshape(p.num_slots, capacity, H, P),
            "dt": dt.reshape(p.num_slots, capacity, H),
            "B": to_storage(B, p.io_dtype).reshape(p.num_slots, capacity, G, N),
            "window": window,
            "start": rng.integers(0, capacity, size=p.num_seqs).astype(np.int32),
            "count": rng.integers(0, window + 1, size=p.num_seqs).astype(np.int32)}


def workload(name: str, *, seed: Optional[int] = None, seq_subset=None) -> Problem:
    """Build a named workload.  ``seq_subset`` keeps only those sequences (same draws)."""
    if name == "tiny":
        p = make_problem([256], nheads=4, headdim=16, dstate=16, ngroups=1, chunk_size=64,
                         io_dtype="f32", state_dtype="f32", num_slots=4, slots=[2],
                         seed=0 if seed is None else seed, name=name)
    elif name == "dense_prefill":
        p = make_problem([2048] * 8, nheads=80, headdim=64, dstate=128, ngroups=1, chunk_size=256,
                         num_slots=8, slots=np.arange(8), seed=1 if seed is None else seed, name=name)
    elif name == "varlen_prefill":
        rng = np.random.default_rng(2 if seed is None else seed)
        lens = rng.integers(1, 4097, size=32)
        lens[3] = rng.integers(1, 128)
        lens[17] = rng.integers(1, 128)
        p = make_problem(lens, nheads=128, headdim=64, dstate=128, ngroups=8, chunk_size=128,
                         num_slots=512, rng=rng, name=name)
    elif name == "continued_a":
        p = make_problem([32], nheads=128, headdim=64, dstate=128, ngroups=8, chunk_size=128,
                         state_dtype="bf16", num_slots=512, has_init=True, cache_std=0.1,
                         seed=3 if seed is None else seed, name=name)
    elif name == "continued_b":
        p = make_problem([32, 600, 1600], nheads=128, headdim=64, dstate=128, ngroups=8,
                         chunk_size=128, state_dtype="bf16", num_slots=512, has_init=True,
                         cache_std=0.1, seed=3 if seed is None else seed, name=name)
    elif name in ("mtp", "mtp_replay"):
        p = make_problem([3] * 128, nheads=128, headdim=64, dstate=128, ngroups=8, chunk_size=128,
                         num_slots=512, has_init=True, write_final=False,
                         want_intermediate=(name == "mtp"), cache_std=0.1,
                         seed=4 if seed is None else seed, name=name)
    else:
        raise KeyError(name)
    if seq_subset is not None:
        p = select_sequences(p, seq_subset)
    return p


def sequence_prefix(p: Problem, s: int, ntok: int) -> Problem:
    """A one-sequence problem: the first ``ntok`` tokens of sequence ``s`` of
    ``p`` (a prefix is itself a valid sequence), with its cache slots only."""
    q = select_sequences(p, [s], compact=True)
    n = max(0, min(int(ntok), q.total_tokens))
    return dataclasses.replace(q, cu_seqlens=np.array([0, n], dtype=np.int32),
                               x=q.x[:n], dt=q.dt[:n], B=q.B[:n], C=q.C[:n])


def select_sequences(p: Problem, seqs, compact: bool = False) -> Problem:
    """A new problem made of the listed sequences of ``p`` (same values, repacked).
    compact: keep only the cache slots those sequences name (in slot order,
    indices renumbered), instead of a copy of the whole cache."""
    seqs = list(seqs)
    cu = p.cu_seqlens.astype(np.int64)
    rows = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in seqs]) if seqs else np.zeros(0, np.int64)
    lens = [int(cu[s + 1] - cu[s]) for s in seqs]
    ncu = np.zeros(len(seqs) + 1, dtype=np.int64)
    ncu[1:] = np.cumsum(lens)
    slot_idx = p.slot_idx[seqs].copy()
    final_slot_idx = None if p.final_slot_idx is None else p.final_slot_idx[seqs].copy()
    if compact:
        named = slot_idx if final_slot_idx is None else np.concatenate([slot_idx, final_slot_idx])
        used = np.unique(named.astype(np.int64))
        cache = p.cache[used]
        slot_idx = np.searchsorted(used, slot_idx).astype(np.int32)
        if final_slot_idx is not None:
            final_slot_idx = np.searchsorted(used, final_slot_idx).astype(np.int32)
    else:
        cache = p.cache.copy()
    return dataclasses.replace(
        p, cu_seqlens=ncu.astype(np.int32), x=p.x[rows], dt=p.dt[rows], B=p.B[rows], C=p.C[rows],
        slot_idx=slot_idx, final_slot_idx=final_slot_idx,
        has_init=None if p.has_init is None else p.has_init[seqs].copy(),
        cache=cache)

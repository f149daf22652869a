"""fp64 CPU oracle of the Mamba2 SSD varlen scan.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import, build
or call anything in this package.  It shares no code with the CUDA library
(``state_space_model_varlen_gb300``); the only thing both sides use is the
seeded input generator, which holds none of the scan's arithmetic.

``ssd_scan_reference(problem)`` covers the whole operation the CUDA path
implements:

* the recurrence itself (``ssd_oracle.c``, fp64, token by token);
* reading the initial state of sequence s from ``cache[slot_idx[s]]`` when
  ``has_init[s]`` is set, else a zero state without reading the slot
  ("otherwise starts from a zero state", vLLM PR #61501 "Details");
* writing the final state back into the same slot in the cache dtype, rounded
  to nearest-even ("final states come out in the cache dtype", vLLM PR #61501
  "Details"; in-place update of the slot, vLLM PR #62922 "Validation");
* optionally the state after every token (MTP verification keeps a state per
  speculative token, vLLM PR #52928 "Summary");
* optionally the state at every chunk boundary ("Prefills that store Mamba
  checkpoints need every chunk state", vLLM PR #61501 "Details");
* final states written to a slot other than the one read, with every initial
  state read from the cache as it was before the call ("Multi-sequence,
  checkpoint and returned-state calls retain snapshot semantics", vLLM PR
  #62922 "Details"; shared/crossed cache slots, same page, "Correctness");
* fp16 cache writes with stochastic rounding driven by a Philox counter-based
  generator seeded from a device buffer (vLLM PR #61501 "Details", ReplaySSM
  seed); ``philox4x32_10`` and ``sr_round_f16`` below;
* ReplaySSM-style multi-token verification: a checkpoint plus a ring of
  pending accepted inputs that is replayed instead of storing a state per
  speculative token (vLLM PR #52928 "Summary"); ``replay_reference`` below.

Every parity claim of the CUDA path is made against this module.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIBDIR = os.path.join(_HERE, "_lib")
_LIBPATH = os.path.join(_LIBDIR, "libssd_oracle.so")
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (OpenMP) into ``oracle/_lib``."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if (not force and os.path.exists(_LIBPATH)
            and os.path.getmtime(_LIBPATH) >= os.path.getmtime(_SRC)):
        return _LIBPATH
    tmp = _LIBPATH + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIBPATH)
    return _LIBPATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIBPATH)
            d = ctypes.POINTER(ctypes.c_double)
            i64p = ctypes.POINTER(ctypes.c_int64)
            lib.ssd_oracle_scan.restype = ctypes.c_int
            lib.ssd_oracle_scan.argtypes = [
                ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                d, d, d, ctypes.c_int32, d, d, d, d, i64p, d, d, d, d, ctypes.c_int32,
                ctypes.c_int32, i64p, d]
            lib.ssd_oracle_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().ssd_oracle_threads())


def _dp(a: Optional[np.ndarray]):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def scan(x, dt, A, B, C, cu_seqlens, *, dt_bias=None, dt_softplus=True, D=None,
         h_init=None, want_final=True, want_inter=False, heads=None, threads=0,
         chunk_size=None, with_chunks=False):
    """Run the fp64 recurrence.  All float inputs are widened to float64.

    Shapes: x [T,H,P], dt [T,H], A [H], B/C [T,G,N], cu_seqlens [S+1],
    h_init [S,H,P,N] or None.  ``heads=(h0, h1)`` limits the work to those
    heads (other entries of the outputs stay zero).
    Returns (y [T,H,P], h_final [S,H,P,N] or None, h_inter [T,H,P,N] or None);
    with ``with_chunks`` a fourth item, the state at the end of every
    ``chunk_size``-token chunk of every sequence [sum_s ceil(len_s/L), H,P,N].
    """
    lib = _load()
    f = lambda a: None if a is None else np.ascontiguousarray(a, dtype=np.float64)
    x, dt, A, B, C, dt_bias, D, h_init = map(f, (x, dt, A, B, C, dt_bias, D, h_init))
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    T, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    S = cu.shape[0] - 1
    h0, h1 = (0, H) if heads is None else heads
    y = np.zeros((T, H, P))
    hf = np.zeros((S, H, P, N)) if want_final else None
    hint = np.zeros((T, H, P, N)) if want_inter else None
    i64 = ctypes.POINTER(ctypes.c_int64)
    hc, cuc, L = None, None, 0
    if with_chunks:
        L = int(chunk_size)
        lens = np.diff(cu)
        cuc = np.zeros(S + 1, dtype=np.int64)
        cuc[1:] = np.cumsum((lens + L - 1) // L)
        hc = np.zeros((int(cuc[-1]), H, P, N))
    rc = lib.ssd_oracle_scan(
        T, S, H, P, N, G, h0, h1, _dp(x), _dp(dt), _dp(dt_bias), int(bool(dt_softplus)),
        _dp(A), _dp(B), _dp(C), _dp(D), cu.ctypes.data_as(i64),
        _dp(h_init), _dp(y), _dp(hf), _dp(hint), int(threads), L,
        i64() if cuc is None else cuc.ctypes.data_as(i64), _dp(hc))
    if rc != 0:
        raise ValueError("ssd_oracle_scan rejected its arguments")
    if with_chunks:
        return y, hf, hint, hc
    return y, hf, hint


# ----------------------------------------------------------------------------
# storage conversions of the oracle's own (no code shared with the CUDA path)
# ----------------------------------------------------------------------------
def widen(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact value of stored data as float64 ('f32', 'f16', 'bf16' uint16 bits)."""
    if dtype == "bf16":
        u = np.ascontiguousarray(a, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return u.view(np.float32).astype(np.float64)
    return np.asarray(a).astype(np.float64)


def round_to(a64: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values to ``dtype`` storage with round-to-nearest-even.

    bf16 is rounded straight from the float64 bits (8-bit significand), so no
    double rounding through float32 takes place.
    """
    a64 = np.ascontiguousarray(a64, dtype=np.float64)
    if dtype == "f32":
        return a64.astype(np.float32)
    if dtype == "f16":
        return a64.astype(np.float16)
    if dtype == "bf16":
        u = a64.view(np.uint64)
        # keep 8 significant bits: drop the low 45 of the 52 mantissa bits, RNE
        bias = ((u >> np.uint64(45)) & np.uint64(1)) + np.uint64((1 << 44) - 1)
        r = ((u + bias) >> np.uint64(45)) << np.uint64(45)
        f32 = r.view(np.float64).astype(np.float32)      # exact: 8-bit significand
        return (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    raise ValueError(dtype)


def ssd_scan_reference(p, *, heads=None, threads=0):
    """Oracle for a whole ``workloads.Problem`` (slot reads, writeback, dtypes).

    Every initial state is read from the cache as it was before the call
    (snapshot semantics), so a sequence may read a slot that another one
    writes.  Final states go to ``p.final_slot_idx`` (default ``p.slot_idx``)
    in batch order.  With ``p.sr_seed`` and an fp16 cache they are rounded
    stochastically (``sr_round_f16`` on the float32 value of the state, the
    random word of each element from ``sr_words``), else to nearest-even.

    Returns a dict with
      y      float64 [T,H,P]
      final  float64 [S,H,P,N]  (state after the last token, before rounding)
      inter  float64 [T,H,P,N] or None
      chunks float64 [sum ceil(len/L),H,P,N] or None (``p.want_chunk_states``)
      cache  the expected cache after the call, in storage dtype (copy)
    """
    S = p.num_seqs
    H, P, N = p.nheads, p.headdim, p.dstate
    h_init = None
    if p.has_init is not None and np.any(p.has_init):
        h_init = np.zeros((S, H, P, N))
        for s in range(S):
            if p.has_init[s]:
                h_init[s] = widen(p.cache[int(p.slot_idx[s])], p.state_dtype)
    out = scan(
        widen(p.x, p.io_dtype), p.dt, p.A, widen(p.B, p.io_dtype), widen(p.C, p.io_dtype),
        p.cu_seqlens, dt_bias=p.dt_bias, dt_softplus=p.dt_softplus, D=p.D, h_init=h_init,
        want_final=True, want_inter=bool(p.want_intermediate), heads=heads, threads=threads,
        chunk_size=p.chunk_size, with_chunks=bool(p.want_chunk_states))
    y, hf, hint = out[:3]
    chunks = out[3] if p.want_chunk_states else None
    cache = p.cache.copy()
    h0, h1 = (0, H) if heads is None else heads
    if p.write_final:
        dst = p.slot_idx if p.final_slot_idx is None else p.final_slot_idx
        for s in range(S):
            slot = int(dst[s])
            if p.sr_seed is not None and p.state_dtype == "f16":
                words = sr_words(p.sr_seed, slot, (h0, h1), H, P, N, stream=0)
                cache[slot, h0:h1] = sr_round_f16(hf[s, h0:h1].astype(np.float32), words)
            else:
                cache[slot, h0:h1] = round_to(hf[s, h0:h1], p.state_dtype)
    return {"y": y, "final": hf, "inter": hint, "chunks": chunks, "cache": cache}


# ----------------------------------------------------------------------------
# Philox4x32-10 and stochastic rounding to fp16
# ----------------------------------------------------------------------------
# Philox4x32 with ten rounds, as defined by Salmon, Moraes, Dror and Shaw,
# "Parallel random numbers: as easy as 1, 2, 3" (SC'11): a counter of four
# 32-bit words and a key of two; each round multiplies words 0 and 2 by the
# two round multipliers (keeping both halves of the 64-bit products) and mixes
# in the other words and the key; the key is bumped by the two Weyl constants
# before every round after the first.
_PH_M0, _PH_M1 = 0xD2511F53, 0xCD9E8D57
_PH_W0, _PH_W1 = 0x9E3779B9, 0xBB67AE85


def philox4x32_10(ctr, key):
    """ctr: four uint32 arrays (or ints), key: two uint32 values; returns four
    uint32 arrays."""
    c = [np.asarray(v, dtype=np.uint64) & np.uint64(0xFFFFFFFF) for v in ctr]
    k0, k1 = int(key[0]) & 0xFFFFFFFF, int(key[1]) & 0xFFFFFFFF
    mask = np.uint64(0xFFFFFFFF)
    for r in range(10):
        if r:
            k0 = (k0 + _PH_W0) & 0xFFFFFFFF
            k1 = (k1 + _PH_W1) & 0xFFFFFFFF
        p0 = np.uint64(_PH_M0) * c[0]
        p1 = np.uint64(_PH_M1) * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & mask
        hi1, lo1 = p1 >> np.uint64(32), p1 & mask
        c = [hi1 ^ c[1] ^ np.uint64(k0), lo1, hi0 ^ c[3] ^ np.uint64(k1), lo0]
    return [v.astype(np.uint32) for v in c]


def sr_words(seed, slot, heads, H, P, N, stream=0):
    """The random word of every element of one written state, rows [h0, h1) of
    slot ``slot`` of a tensor laid out [rows, H, P, N].

    Element e (its flat index in that tensor) uses word (e mod 4) of
    Philox4x32-10 with key (seed mod 2^32, seed >> 32) and counter
    (e >> 2 mod 2^32, e >> 34, stream, 0); stream 0 is the state cache, 1 the
    per-chunk state output."""
    h0, h1 = heads
    base = (int(slot) * H + h0) * P * N
    e = np.arange(base, base + (h1 - h0) * P * N, dtype=np.uint64)
    q = e >> np.uint64(2)
    w = philox4x32_10([q & np.uint64(0xFFFFFFFF), q >> np.uint64(32),
                       np.full(q.shape, stream, np.uint64), np.zeros(q.shape, np.uint64)],
                      (int(seed) & 0xFFFFFFFF, (int(seed) >> 32) & 0xFFFFFFFF))
    sel = (e & np.uint64(3)).astype(np.int64)
    words = np.choose(sel, w)
    return words.reshape(h1 - h0, P, N)


_F16_MAX = 65504.0


def sr_round_f16(v32, r):
    """Stochastic rounding of float32 values to fp16 driven by uint32 words r.

    For finite v let lo be v rounded toward zero to fp16 and hi the next fp16
    value away from zero (infinity above the largest finite value, as if the
    next value were 65536 for the fraction below); with f = (|v| - |lo|) /
    (|hi| - |lo|) in [0, 1), the result is hi when f * 2^32 > r, else lo.  So
    v rounds up with probability f: the expected result is v.  Values that
    fp16 holds exactly, infinities and NaN are returned unchanged.  All of it
    is exact in float64."""
    v = np.asarray(v32, dtype=np.float32).astype(np.float64)
    r = np.asarray(r, dtype=np.uint32).astype(np.float64)
    a = np.abs(v)
    with np.errstate(over="ignore", invalid="ignore"):
        # fp16 spacing at |v|: 2^(e - 10) with e = floor(log2 |v|) kept within
        # fp16's exponent range [-14, 15] (below: subnormal spacing 2^-24)
        _, k = np.frexp(np.where(np.isfinite(a) & (a > 0), a, 1.0))
        e = np.clip(k - 1, -14, 15)
        ulp = np.ldexp(1.0, e - 10)
        lo = np.minimum(np.floor(a / ulp) * ulp, _F16_MAX)     # toward zero
        ulp = np.where(a > _F16_MAX, 32.0, ulp)
        f = (a - lo) / ulp
        up = f * 4294967296.0 > r
        mag = np.where(up, lo + ulp, lo)
        mag = np.where(mag > _F16_MAX, np.inf, mag)
        out = np.where(np.isfinite(v), np.copysign(mag, v), v)
    return out.astype(np.float16)


# ----------------------------------------------------------------------------
# ReplaySSM-style multi-token verification
# ----------------------------------------------------------------------------
def replay_reference(p, ring, heads=None):
    """One verification step over a checkpoint and a ring of pending inputs.

    ``p`` is a ``workloads.Problem`` holding the verification windows (one
    sequence per request, ``p.slot_idx`` the request's checkpoint slot in
    ``p.cache``).  ``ring`` is a dict with
      x [slots, R, H, P] (io storage), dt [slots, R, H] (raw, float32),
      B [slots, R, G, N] (io storage), start [S], count [S] (int), window (int)
    holding, for request s, ``count[s]`` accepted inputs not yet in its
    checkpoint at ring positions (start[s] + j) mod R, and the logical window.

    Per request (vLLM PR #52928 "Summary": "each layer keeps a checkpoint and a
    ring of inputs ... the checkpoint is updated only when the next
    verification window would overflow the ring"): the state is the checkpoint
    advanced through the pending inputs; y of the window tokens follows from
    it; when count + window length > window the checkpoint becomes that state
    (the pending inputs are folded in) and the live part of the ring restarts
    after them.  The window's inputs are appended to the ring after the pending
    ones.  Returns y, the expected cache and ring, and the new (start, count)
    the ring holds before the caller adds the accepted tokens.
    """
    S, H, P, N, G = p.num_seqs, p.nheads, p.headdim, p.dstate, p.ngroups
    R = ring["x"].shape[1]
    h0, h1 = (0, H) if heads is None else heads
    cu = p.cu_seqlens
    y = np.zeros((p.total_tokens, H, P))
    cache = p.cache.copy()
    rx, rdt, rB = ring["x"].copy(), ring["dt"].copy(), ring["B"].copy()
    new_start = np.zeros(S, dtype=np.int64)
    new_count = np.zeros(S, dtype=np.int64)
    for s in range(S):
        q = int(p.slot_idx[s])
        a, b = int(cu[s]), int(cu[s + 1])
        K, r0, cnt = b - a, int(ring["start"][s]), int(ring["count"][s])
        pos = [(r0 + j) % R for j in range(cnt)]
        hx = widen(ring["x"][q, pos], p.io_dtype).reshape(cnt, H, P)
        hdt = ring["dt"][q, pos].reshape(cnt, H)
        hB = widen(ring["B"][q, pos], p.io_dtype).reshape(cnt, G, N)
        h_ck = widen(p.cache[q], p.state_dtype)[None]
        # state after the pending inputs (the checkpoint advanced; no output)
        _, h_pend, _ = scan(hx, hdt, p.A, hB, hB, [0, cnt], dt_bias=p.dt_bias,
                            dt_softplus=p.dt_softplus, h_init=h_ck, heads=(h0, h1))
        # the window from that state
        yw, _, _ = scan(widen(p.x[a:b], p.io_dtype), p.dt[a:b], p.A, widen(p.B[a:b], p.io_dtype),
                        widen(p.C[a:b], p.io_dtype), [0, K], dt_bias=p.dt_bias,
                        dt_softplus=p.dt_softplus, D=p.D, h_init=h_pend, heads=(h0, h1))
        y[a:b] = yw
        fold = cnt + K > int(ring["window"])
        if fold:
            if p.sr_seed is not None and p.state_dtype == "f16":
                words = sr_words(p.sr_seed, q, (h0, h1), H, P, N, stream=0)
                cache[q, h0:h1] = sr_round_f16(h_pend[0, h0:h1].astype(np.float32), words)
            else:
                cache[q, h0:h1] = round_to(h_pend[0, h0:h1], p.state_dtype)
            new_start[s], new_count[s] = (r0 + cnt) % R, 0
        else:
            new_start[s], new_count[s] = r0, cnt
        for i in range(K):
            w = (r0 + cnt + i) % R
            rx[q, w, h0:h1] = p.x[a + i, h0:h1]
            rdt[q, w, h0:h1] = p.dt[a + i, h0:h1]
            rB[q, w] = p.B[a + i]
    return {"y": y, "cache": cache, "ring_x": rx, "ring_dt": rdt, "ring_B": rB,
            "start": new_start, "count": new_count}

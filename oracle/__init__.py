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
  speculative token, vLLM PR #52928 "Summary").

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
                d, d, d, ctypes.c_int32, d, d, d, d, i64p, d, d, d, d, ctypes.c_int32]
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
         h_init=None, want_final=True, want_inter=False, heads=None, threads=0):
    """Run the fp64 recurrence.  All float inputs are widened to float64.

    Shapes: x [T,H,P], dt [T,H], A [H], B/C [T,G,N], cu_seqlens [S+1],
    h_init [S,H,P,N] or None.  ``heads=(h0, h1)`` limits the work to those
    heads (other entries of the outputs stay zero).
    Returns (y [T,H,P], h_final [S,H,P,N] or None, h_inter [T,H,P,N] or None).
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
    rc = lib.ssd_oracle_scan(
        T, S, H, P, N, G, h0, h1, _dp(x), _dp(dt), _dp(dt_bias), int(bool(dt_softplus)),
        _dp(A), _dp(B), _dp(C), _dp(D), cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
        _dp(h_init), _dp(y), _dp(hf), _dp(hint), int(threads))
    if rc != 0:
        raise ValueError("ssd_oracle_scan rejected its arguments")
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

    Returns a dict with
      y      float64 [T,H,P]
      final  float64 [S,H,P,N]  (state after the last token, before rounding)
      inter  float64 [T,H,P,N] or None
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
    y, hf, hint = scan(
        widen(p.x, p.io_dtype), p.dt, p.A, widen(p.B, p.io_dtype), widen(p.C, p.io_dtype),
        p.cu_seqlens, dt_bias=p.dt_bias, dt_softplus=p.dt_softplus, D=p.D, h_init=h_init,
        want_final=True, want_inter=bool(p.want_intermediate), heads=heads, threads=threads)
    cache = p.cache.copy()
    h0, h1 = (0, H) if heads is None else heads
    if p.write_final:
        for s in range(S):
            cache[int(p.slot_idx[s]), h0:h1] = round_to(hf[s, h0:h1], p.state_dtype)
    return {"y": y, "final": hf, "inter": hint, "cache": cache}

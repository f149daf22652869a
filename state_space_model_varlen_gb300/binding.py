"""ctypes binding of the C ABI in ``include/ssd_scan.h``.

Argument marshalling only: every step of the scan runs in the library's CUDA
kernels.  torch supplies device memory and streams.  If the library cannot be
loaded the calls raise; there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

from . import _build

(SSD_OK, SSD_ERR_INVALID_ARG, SSD_ERR_UNSUPPORTED, SSD_ERR_WORKSPACE, SSD_ERR_CUDA,
 SSD_ERR_SCRATCH_LIMIT) = range(6)
SSD_NOALLOC_MAX_SEQS = 65536
SSD_F32, SSD_BF16, SSD_F16 = 0, 1, 2
SSD_DEV_BAD_SLOT, SSD_DEV_BAD_SEQLENS, SSD_DEV_TIMEOUT = 1, 2, 4
SSD_DEV_BAD_CHUNKS, SSD_DEV_BAD_RING = 8, 16

# every exported entry point declared in include/ssd_scan.h
EXPORTED = ("ssd_replay_mtp", "ssd_scan_varlen", "ssd_scan_varlen_noalloc",
            "ssd_scan_varlen_num_launches", "ssd_scan_varlen_path",
            "ssd_scan_varlen_workspace_size", "ssd_status_string", "ssd_testing_set_hooks")


class ScanParams(ctypes.Structure):
    """Mirror of ``ssd_scan_params``."""
    _fields_ = [
        ("total_tokens", ctypes.c_int64),
        ("num_seqs", ctypes.c_int32),
        ("max_seqlen", ctypes.c_int32),
        ("nheads", ctypes.c_int32),
        ("headdim", ctypes.c_int32),
        ("dstate", ctypes.c_int32),
        ("ngroups", ctypes.c_int32),
        ("chunk_size", ctypes.c_int32),
        ("io_dtype", ctypes.c_int32),
        ("state_dtype", ctypes.c_int32),
        ("dt_softplus", ctypes.c_int32),
        ("write_final", ctypes.c_int32),
        ("num_slots", ctypes.c_int32),
        ("reserved0", ctypes.c_int32),
        ("x", ctypes.c_void_p),
        ("dt", ctypes.c_void_p),
        ("dt_bias", ctypes.c_void_p),
        ("A", ctypes.c_void_p),
        ("B", ctypes.c_void_p),
        ("C", ctypes.c_void_p),
        ("D", ctypes.c_void_p),
        ("cu_seqlens", ctypes.c_void_p),
        ("state_cache", ctypes.c_void_p),
        ("slot_idx", ctypes.c_void_p),
        ("has_init", ctypes.c_void_p),
        ("out_y", ctypes.c_void_p),
        ("out_intermediate", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("device_status", ctypes.c_void_p),
        ("out_chunk_states", ctypes.c_void_p),
        ("cu_chunks", ctypes.c_void_p),
        ("num_chunk_rows", ctypes.c_int32),
        ("slots_disjoint", ctypes.c_int32),
        ("final_slot_idx", ctypes.c_void_p),
        ("slot_idx_stride", ctypes.c_int64),
        ("final_slot_idx_stride", ctypes.c_int64),
        ("sr_seed", ctypes.c_void_p),
    ]


class ReplayParams(ctypes.Structure):
    """Mirror of ``ssd_replay_params``."""
    _fields_ = [
        ("scan", ScanParams),
        ("ring_x", ctypes.c_void_p),
        ("ring_dt", ctypes.c_void_p),
        ("ring_B", ctypes.c_void_p),
        ("ring_capacity", ctypes.c_int32),
        ("ring_window", ctypes.c_int32),
        ("ring_start", ctypes.c_void_p),
        ("ring_count", ctypes.c_void_p),
        ("ring_start_out", ctypes.c_void_p),
        ("ring_count_out", ctypes.c_void_p),
    ]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIBPATH


def load(build_if_missing: bool = True):
    """Load the CUDA library (building it in-tree first if needed)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIBPATH
            if build_if_missing and not _build.up_to_date():
                _build.build()
            if not os.path.exists(path):
                raise RuntimeError("libssd_scan.so is missing; run __graft_entry__.build()")
            lib = ctypes.CDLL(path)
            P = ctypes.POINTER(ScanParams)
            lib.ssd_scan_varlen.restype = ctypes.c_int
            lib.ssd_scan_varlen.argtypes = [P, ctypes.c_void_p]
            lib.ssd_scan_varlen_workspace_size.restype = ctypes.c_size_t
            lib.ssd_scan_varlen_workspace_size.argtypes = [P]
            lib.ssd_scan_varlen_num_launches.restype = ctypes.c_int32
            lib.ssd_scan_varlen_num_launches.argtypes = [P]
            lib.ssd_scan_varlen_path.restype = ctypes.c_char_p
            lib.ssd_scan_varlen_path.argtypes = [P]
            lib.ssd_scan_varlen_noalloc.restype = ctypes.c_int
            lib.ssd_scan_varlen_noalloc.argtypes = [P, ctypes.c_void_p]
            lib.ssd_testing_set_hooks.restype = None
            lib.ssd_testing_set_hooks.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32]
            lib.ssd_replay_mtp.restype = ctypes.c_int
            lib.ssd_replay_mtp.argtypes = [ctypes.POINTER(ReplayParams), ctypes.c_void_p]
            lib.ssd_status_string.restype = ctypes.c_char_p
            lib.ssd_status_string.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def status_string(code: int) -> str:
    return load().ssd_status_string(int(code)).decode()


class SSDError(RuntimeError):
    def __init__(self, code: int):
        super().__init__("ssd_scan_varlen failed: %s (%d)" % (status_string(code), code))
        self.code = code


# ---------------------------------------------------------------------------
# torch-facing helpers (marshalling only)
# ---------------------------------------------------------------------------
def _torch():
    import torch
    return torch


def _dtype_code(t, allowed):
    torch = _torch()
    m = {torch.float32: SSD_F32, torch.bfloat16: SSD_BF16, torch.float16: SSD_F16}
    if t.dtype not in m or m[t.dtype] not in allowed:
        raise TypeError("unsupported dtype %s" % t.dtype)
    return m[t.dtype]


def _ptr(t, dtype=None):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the SSD scan must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError("expected %s, got %s" % (dtype, t.dtype))
    return t.data_ptr()


def _index_ptr(t):
    """A 1-D int32 index tensor, possibly a strided view (a block-table column):
    (pointer, stride in elements)."""
    torch = _torch()
    if t is None:
        return None, 0
    if t.dtype != torch.int32 or t.dim() != 1:
        raise TypeError("slot indices must be a 1-D int32 tensor")
    return t.data_ptr(), int(t.stride(0))


def make_params(x, dt, A, B, C, cu_seqlens, *, dt_bias=None, D=None, state_cache=None,
                slot_idx=None, has_init=None, write_final=True, out_y=None,
                out_intermediate=None, dt_softplus=True, chunk_size=128, max_seqlen=0,
                workspace=None, device_status=None, final_slot_idx=None,
                out_chunk_states=None, cu_chunks=None, sr_seed=None,
                slots_disjoint=False) -> ScanParams:
    """Fill ``ssd_scan_params`` from torch tensors (no copies, no device reads).

    ``slot_idx`` / ``final_slot_idx`` may be strided int32 views; ``sr_seed``
    is a one-element int64 device tensor (its bits are the 64-bit seed)."""
    torch = _torch()
    T, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    S = cu_seqlens.shape[0] - 1
    p = ScanParams()
    p.total_tokens, p.num_seqs, p.max_seqlen = T, S, int(max_seqlen)
    p.nheads, p.headdim, p.dstate, p.ngroups, p.chunk_size = H, P, N, G, int(chunk_size)
    p.io_dtype = _dtype_code(x, (SSD_F32, SSD_BF16))
    if B.dtype != x.dtype or C.dtype != x.dtype or (out_y is not None and out_y.dtype != x.dtype):
        raise TypeError("x, B, C and out_y must share one dtype")
    p.state_dtype = _dtype_code(state_cache, (SSD_F32, SSD_BF16, SSD_F16)) \
        if state_cache is not None else (
            _dtype_code(out_intermediate, (SSD_F32, SSD_BF16, SSD_F16))
            if out_intermediate is not None else SSD_F32)
    if out_intermediate is not None and state_cache is not None and \
            out_intermediate.dtype != state_cache.dtype:
        raise TypeError("out_intermediate must have the state cache dtype")
    p.dt_softplus, p.write_final = int(bool(dt_softplus)), int(bool(write_final))
    p.num_slots = 0 if state_cache is None else state_cache.shape[0]
    p.x, p.B, p.C = _ptr(x), _ptr(B), _ptr(C)
    p.dt, p.A = _ptr(dt, torch.float32), _ptr(A, torch.float32)
    p.dt_bias, p.D = _ptr(dt_bias, torch.float32), _ptr(D, torch.float32)
    p.cu_seqlens = _ptr(cu_seqlens, torch.int32)
    p.state_cache = _ptr(state_cache)
    p.slot_idx, p.slot_idx_stride = _index_ptr(slot_idx)
    p.final_slot_idx, p.final_slot_idx_stride = _index_ptr(final_slot_idx)
    if out_chunk_states is not None:
        if cu_chunks is None:
            raise ValueError("out_chunk_states needs cu_chunks")
        if state_cache is not None and out_chunk_states.dtype != state_cache.dtype:
            raise TypeError("out_chunk_states must have the state cache dtype")
        p.out_chunk_states = _ptr(out_chunk_states)
        p.num_chunk_rows = out_chunk_states.shape[0]
    p.cu_chunks = _ptr(cu_chunks, torch.int32)
    if sr_seed is not None and sr_seed.dtype not in (torch.int64, torch.uint64):
        raise TypeError("sr_seed must be a 64-bit integer tensor")
    p.sr_seed = None if sr_seed is None else sr_seed.data_ptr()
    p.slots_disjoint = int(bool(slots_disjoint))
    if has_init is not None and has_init.dtype == torch.bool:
        has_init = has_init.view(torch.uint8)
    p.has_init = _ptr(has_init, torch.uint8)
    p.out_y = _ptr(out_y)
    p.out_intermediate = _ptr(out_intermediate)
    p.workspace = _ptr(workspace)
    p.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    p.device_status = _ptr(device_status, torch.int32)
    return p


def workspace_size(params: ScanParams) -> int:
    return int(load().ssd_scan_varlen_workspace_size(ctypes.byref(params)))


def num_launches(params: ScanParams) -> int:
    return int(load().ssd_scan_varlen_num_launches(ctypes.byref(params)))


def kernel_path(params: ScanParams) -> str:
    return load().ssd_scan_varlen_path(ctypes.byref(params)).decode()


def call(params: ScanParams, stream_ptr: int = 0) -> None:
    rc = load().ssd_scan_varlen(ctypes.byref(params), ctypes.c_void_p(stream_ptr or None))
    if rc != SSD_OK:
        raise SSDError(rc)


def make_replay_params(scan: ScanParams, ring_x, ring_dt, ring_B, ring_window, ring_start,
                       ring_count, ring_start_out, ring_count_out) -> ReplayParams:
    """Fill ``ssd_replay_params`` (the scan part from ``make_params`` with
    ``write_final=False``)."""
    torch = _torch()
    r = ReplayParams()
    r.scan = scan
    r.ring_x, r.ring_B = _ptr(ring_x), _ptr(ring_B)
    r.ring_dt = _ptr(ring_dt, torch.float32)
    r.ring_capacity = ring_x.shape[1]
    r.ring_window = int(ring_window)
    r.ring_start, r.ring_count = _ptr(ring_start, torch.int32), _ptr(ring_count, torch.int32)
    r.ring_start_out = _ptr(ring_start_out, torch.int32)
    r.ring_count_out = _ptr(ring_count_out, torch.int32)
    return r


def call_replay(params: ReplayParams, stream_ptr: int = 0) -> None:
    rc = load().ssd_replay_mtp(ctypes.byref(params), ctypes.c_void_p(stream_ptr or None))
    if rc != SSD_OK:
        raise SSDError(rc)


def set_test_hooks(wait_cycles: int = 0, withhold_handover: int = -1,
                   force_unsegmented: bool = False) -> None:
    """``ssd_testing_set_hooks`` (tests of the failure detection only)."""
    load().ssd_testing_set_hooks(int(wait_cycles), int(withhold_handover), int(bool(force_unsegmented)))


def call_noalloc(params: ScanParams, stream_ptr: int = 0) -> None:
    """``ssd_scan_varlen_noalloc``: the scan with the library's fixed scratch
    instead of ``params.workspace`` (for callers that cannot allocate)."""
    rc = load().ssd_scan_varlen_noalloc(ctypes.byref(params), ctypes.c_void_p(stream_ptr or None))
    if rc != SSD_OK:
        raise SSDError(rc)


def ssd_scan_varlen(x, dt, A, B, C, cu_seqlens, *, dt_bias=None, D=None, state_cache=None,
                    slot_idx=None, has_init=None, write_final=True, out_y=None,
                    out_intermediate=None, dt_softplus=True, chunk_size=128, max_seqlen=0,
                    workspace=None, device_status=None, stream=None):
    """Run the scan on torch CUDA tensors; returns ``out_y`` (allocated if None).

    ``state_cache`` is updated in place when ``write_final``.  ``workspace`` is
    allocated here when the selected kernel needs one and none is given.
    """
    torch = _torch()
    if out_y is None:
        out_y = torch.empty_like(x)
    p = make_params(x, dt, A, B, C, cu_seqlens, dt_bias=dt_bias, D=D, state_cache=state_cache,
                    slot_idx=slot_idx, has_init=has_init, write_final=write_final, out_y=out_y,
                    out_intermediate=out_intermediate, dt_softplus=dt_softplus,
                    chunk_size=chunk_size, max_seqlen=max_seqlen, workspace=workspace,
                    device_status=device_status)
    if workspace is None:
        need = workspace_size(p)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
            p.workspace, p.workspace_bytes = workspace.data_ptr(), need
    s = torch.cuda.current_stream(x.device) if stream is None else stream
    call(p, s.cuda_stream)
    return out_y

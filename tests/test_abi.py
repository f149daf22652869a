"""C-ABI checks that need no GPU: the library builds for sm_103a, loads, exports
every entry point declared in include/ssd_scan.h, the ctypes mirror of
``ssd_scan_params`` has the C layout, and host-side validation rejects bad
arguments before anything is enqueued (those calls touch no CUDA API)."""
import ctypes
import os
import re
import subprocess

import pytest

from state_space_model_varlen_gb300 import binding, _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssd_scan.h")


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ssd_\w+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = binding.load()
    declared = _declared_functions()
    assert declared, "no declarations parsed"
    assert sorted(binding.EXPORTED) == declared
    for name in declared:
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIBPATH], capture_output=True,
                         text=True, check=True).stdout
    for name in declared:
        assert re.search(r"\bT %s$" % name, out, re.M), name


@pytest.mark.parametrize("cls,cname", [(binding.ScanParams, "ssd_scan_params"),
                                       (binding.ReplayParams, "ssd_replay_params")])
def test_params_struct_layout_matches_c(tmp_path, cls, cname):
    fields = [f[0] for f in cls._fields_]
    prog = ["#include <stdio.h>", "#include <stddef.h>", '#include "%s"' % HEADER,
            "int main(void){", 'printf("%%zu\\n", sizeof(%s));' % cname]
    for f in fields:
        prog.append('printf("%%zu\\n", offsetof(%s, %s));' % (cname, f))
    prog.append("return 0;}")
    c = tmp_path / "layout.c"
    c.write_text("\n".join(prog))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", str(c), "-o", str(exe)], check=True)
    vals = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True,
                                           check=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(cls)
    for f, off in zip(fields, vals[1:]):
        assert getattr(cls, f).offset == off, f


def _params(**kw):
    p = binding.ScanParams()
    p.total_tokens, p.num_seqs, p.max_seqlen = 10, 2, 0
    p.nheads, p.headdim, p.dstate, p.ngroups, p.chunk_size = 4, 64, 128, 2, 128
    p.io_dtype, p.state_dtype = binding.SSD_BF16, binding.SSD_F32
    p.dt_softplus, p.write_final, p.num_slots = 1, 1, 4
    for name in ("x", "dt", "A", "B", "C", "cu_seqlens", "state_cache", "slot_idx", "out_y"):
        setattr(p, name, 0x1000)
    for k, v in kw.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("field,value", [
    ("nheads", 0), ("headdim", -1), ("ngroups", 3), ("chunk_size", 0), ("io_dtype", 2),
    ("io_dtype", 7), ("state_dtype", 5), ("total_tokens", -1), ("x", None),
    ("cu_seqlens", None), ("state_cache", None), ("slot_idx", None), ("num_slots", 0),
])
def test_invalid_arguments_rejected_without_launch(field, value):
    p = _params(**{field: value})
    lib = binding.load()
    rc = lib.ssd_scan_varlen(ctypes.byref(p), None)
    assert rc == binding.SSD_ERR_INVALID_ARG
    assert binding.num_launches(p) == -1
    assert binding.kernel_path(p) == "invalid"
    assert binding.workspace_size(p) == 0


def test_unsupported_state_size():
    p = _params(dstate=512)
    assert binding.load().ssd_scan_varlen(ctypes.byref(p), None) == binding.SSD_ERR_UNSUPPORTED


def test_empty_batch_launches_nothing():
    p = _params(num_seqs=0, total_tokens=0)
    assert binding.num_launches(p) == 0
    assert binding.load().ssd_scan_varlen(ctypes.byref(p), None) == binding.SSD_OK


def test_kernel_path_selection():
    assert binding.kernel_path(_params(io_dtype=binding.SSD_F32)) == "recurrent"
    assert binding.kernel_path(_params(out_intermediate=0x2000)) == "recurrent"
    assert binding.kernel_path(_params(max_seqlen=3)) == "recurrent"
    assert binding.num_launches(_params(io_dtype=binding.SSD_F32)) == 1


def test_status_strings():
    for code in range(5):
        assert binding.status_string(code) and binding.status_string(code) != "unknown status"
    assert binding.status_string(99) == "unknown status"


@pytest.mark.parametrize("S,H,expect", [
    (2, 4, 256),                  # no hand-over possible: the sequence order only
    (40, 2, 394240),              # 6 hand-over states (6-block segments bound them)
    (600, 80, 67130624),          # 1024 hand-over states at most
    (8193, 80, 33024),            # beyond the sort: the sequence order only
])
def test_workspace_layout(S, H, expect):
    """Workspace of the tensor-core path (T = 0 keeps the query on the host):
    int32 order[S], then for segments a 64-int level table, int32 bstart[S],
    four flags and one 64 KiB fp32 state per hand-over, each part 256-byte
    aligned."""
    p = _params(total_tokens=0, num_seqs=S, nheads=H, ngroups=1)
    assert binding.kernel_path(p) == "chunked_tc"
    r256 = lambda v: (v + 255) // 256 * 256
    size = binding.workspace_size(p)
    assert size == expect
    cap = min(1024, S * (H // 2) // 6)
    if S <= 8192 and cap > 0:
        assert size == r256(4 * S) + 256 + r256(4 * S) + r256(16 * cap) + cap * 65536
    else:
        assert size == r256(4 * S)
    assert size <= r256(4 * S) * 2 + 256 + 16384 + (64 << 20)


def test_snapshot_workspace_and_launch_count():
    """Several sequences with initial states and final writeback may cross slots:
    the workspace grows by int32 flags [S] and S states (cache dtype), 256-byte
    aligned after the tensor-core part, and the call takes the prep launch; a
    caller promise of disjoint slots drops both."""
    base = _params(total_tokens=0, num_seqs=3)
    with_init = _params(total_tokens=0, num_seqs=3, has_init=0x1000)
    disjoint = _params(total_tokens=0, num_seqs=3, has_init=0x1000, slots_disjoint=1)
    r256 = lambda v: (v + 255) // 256 * 256
    state = 4 * 64 * 128 * 4
    w0 = binding.workspace_size(base)                  # the tensor-core path's own part
    assert w0 % 256 == 0
    assert binding.workspace_size(with_init) == w0 + r256(4 * 3) + 3 * state
    assert binding.workspace_size(disjoint) == w0
    one = _params(total_tokens=0, num_seqs=1, has_init=0x1000)
    assert binding.workspace_size(one) == binding.workspace_size(_params(total_tokens=0, num_seqs=1))
    rec = _params(total_tokens=0, num_seqs=3, has_init=0x1000, io_dtype=binding.SSD_F32)
    assert binding.kernel_path(rec) == "recurrent"
    assert binding.workspace_size(rec) == r256(4 * 3) + 3 * state
    assert binding.num_launches(rec) == 2


def test_option_argument_checks():
    assert binding.load().ssd_scan_varlen(ctypes.byref(_params(slot_idx_stride=-1)), None) == \
        binding.SSD_ERR_INVALID_ARG
    assert binding.load().ssd_scan_varlen(ctypes.byref(_params(out_chunk_states=0x2000)), None) == \
        binding.SSD_ERR_INVALID_ARG                    # no cu_chunks
    assert binding.load().ssd_scan_varlen(
        ctypes.byref(_params(final_slot_idx=0x2000, write_final=0)), None) == binding.SSD_ERR_INVALID_ARG
    # per-chunk states on the tensor-core path need 128-token multiples
    p = _params(total_tokens=0, out_chunk_states=0x2000, cu_chunks=0x3000, num_chunk_rows=4,
                chunk_size=64)
    assert binding.kernel_path(p) == "recurrent"
    p.chunk_size = 256
    assert binding.kernel_path(p) == "chunked_tc"


def test_replay_argument_checks():
    lib = binding.load()
    r = binding.ReplayParams()
    r.scan = _params(write_final=0)
    for name in ("ring_x", "ring_dt", "ring_B", "ring_start", "ring_count"):
        setattr(r, name, 0x4000)
    r.ring_start_out, r.ring_count_out = 0x5000, 0x6000
    r.ring_capacity, r.ring_window = 8, 5
    r.scan.max_seqlen = 4                               # 5 + 4 > 8: the window does not fit
    assert lib.ssd_replay_mtp(ctypes.byref(r), None) == binding.SSD_ERR_INVALID_ARG
    r.scan.max_seqlen = 3
    r.scan.write_final = 1                              # replay never writes final states
    assert lib.ssd_replay_mtp(ctypes.byref(r), None) == binding.SSD_ERR_INVALID_ARG
    r.scan.write_final = 0
    r.ring_start_out = 0x4000                           # aliases ring_start
    assert lib.ssd_replay_mtp(ctypes.byref(r), None) == binding.SSD_ERR_INVALID_ARG

"""Failure detection of the tensor-core kernel, made on the host, with no GPU
fault: a segment hand-over that is never published (a flag nothing sets) makes
the waiting segment's bounded wait run out; the kernel reports SSD_DEV_TIMEOUT,
returns, and the same context computes the next call correctly.  Also the
fallback that runs a segmented batch whole (taken when a cooperative launch is
refused), forced through the test hook."""
import numpy as np
import pytest

import oracle
from state_space_model_varlen_gb300 import binding
from state_space_model_varlen_gb300 import workloads as W
from tests import harness as Hn

pytestmark = pytest.mark.gpu


def _segmented(seed):
    rng = np.random.default_rng(seed)
    lens = rng.integers(2900, 5200, size=8)
    return W.make_problem(lens, nheads=80, headdim=64, dstate=128, ngroups=1, num_slots=12,
                          has_init=[1, 0, 1, 0, 0, 1, 1, 0], cache_std=0.1, seed=seed)


def _sampled_ok(p, out, seqs=(0, 3, 6), heads=(8, 24)):
    q = W.select_sequences(p, list(seqs))
    ref = oracle.ssd_scan_reference(q, heads=heads)
    rows = np.concatenate([np.arange(p.cu_seqlens[s], p.cu_seqlens[s + 1]) for s in seqs])
    Hn.check_y(out["y"][rows][:, heads[0]:heads[1]], ref["y"][:, heads[0]:heads[1]], p.io_dtype)
    for j, s in enumerate(seqs):
        Hn.check_state(out["cache"][p.slot_idx[s], heads[0]:heads[1]],
                       ref["final"][j, heads[0]:heads[1]], p.state_dtype)


def test_withheld_handover_times_out_and_the_context_stays_usable():
    p = _segmented(101)
    binding.set_test_hooks(wait_cycles=2_000_000, withhold_handover=0)     # ~1 ms per wait
    try:
        out = Hn.run_gpu(p, slots_disjoint=True)
    finally:
        binding.set_test_hooks()
    assert out["path"] == "chunked_tc" and out["launches"] == 2
    assert out["status"] & binding.SSD_DEV_TIMEOUT
    again = Hn.run_gpu(p, slots_disjoint=True)                           # same context
    assert again["status"] == 0
    _sampled_ok(p, again)


def test_forced_unsegmented_fallback_matches_the_oracle():
    p = _segmented(102)
    binding.set_test_hooks(force_unsegmented=True)
    try:
        out = Hn.run_gpu(p, slots_disjoint=True)
    finally:
        binding.set_test_hooks()
    assert out["status"] == 0
    _sampled_ok(p, out)

"""Host-side helpers the benchmark's CPU legs use to sample the workloads: the
compact slot selection, sequence prefixes and the bounded oracle sample (no
GPU; small problems)."""
import dataclasses

import numpy as np

import bench
import oracle
from state_space_model_varlen_gb300 import workloads as W


def _crossed_problem():
    p = W.make_problem([40, 0, 75, 33], nheads=4, headdim=8, dstate=16, ngroups=2,
                       io_dtype="bf16", state_dtype="f32", num_slots=9, slots=[7, 2, 5, 0],
                       has_init=True, seed=11)
    # sequence 0 writes the slot sequence 2 reads, sequence 3 writes one nobody reads
    return dataclasses.replace(p, final_slot_idx=np.array([5, 2, 8, 3], dtype=np.int32))


def test_compact_selection_keeps_results_and_slot_roles():
    p = _crossed_problem()
    for seqs in ([0, 2], [2, 0, 3], [1]):
        full = W.select_sequences(p, seqs)
        comp = W.select_sequences(p, seqs, compact=True)
        a, b = oracle.ssd_scan_reference(full), oracle.ssd_scan_reference(comp)
        np.testing.assert_array_equal(a["y"], b["y"])
        np.testing.assert_array_equal(a["final"], b["final"])
        # the compact cache holds exactly the named slots, in slot order
        named = np.unique(np.concatenate([p.slot_idx[seqs], p.final_slot_idx[seqs]]))
        assert comp.cache.shape[0] == len(named)
        np.testing.assert_array_equal(comp.cache, p.cache[named])
        np.testing.assert_array_equal(b["cache"], a["cache"][named])
        # crossed roles survive the renumbering
        for i, s in enumerate(seqs):
            assert named[comp.slot_idx[i]] == p.slot_idx[s]
            assert named[comp.final_slot_idx[i]] == p.final_slot_idx[s]


def test_sequence_prefix_gives_the_first_outputs():
    """A prefix of a sequence is a sequence: its outputs are the first rows of
    the whole sequence's (the recurrence is causal)."""
    p = _crossed_problem()
    whole = oracle.ssd_scan_reference(W.select_sequences(p, [2]))
    for n in (1, 17, 75, 200):
        q = W.sequence_prefix(p, 2, n)
        assert q.total_tokens == min(n, 75) and q.num_seqs == 1
        got = oracle.ssd_scan_reference(q)
        np.testing.assert_array_equal(got["y"], whole["y"][:q.total_tokens])


def test_oracle_sample_shrinks_to_the_budget():
    p = W.workload("tiny")
    rate = bench._oracle_calibrate(p)
    tok, el, threads, nseq, passes, heads = bench._oracle_sample(p, 1e-6, rate)
    assert nseq == 1 and passes == 1 and heads == p.nheads
    assert tok == 16                                     # the smallest prefix
    tok, el, *_ = bench._oracle_sample(p, 0.2, rate)
    assert tok >= p.total_tokens                         # whole workload, repeated

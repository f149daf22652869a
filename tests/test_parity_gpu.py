"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs.  Small cases are compared element by element in full;
the named full-size workloads run in the benchmark's launch configuration and
are compared on sampled sequences/heads the oracle computes one by one."""
import numpy as np
import pytest

import oracle
from state_space_model_varlen_gb300 import workloads as W
from tests import harness as Hn

pytestmark = pytest.mark.gpu


def _run_and_check(p, **kw):
    out = Hn.run_gpu(p, **kw)
    ref = oracle.ssd_scan_reference(p)
    assert out["status"] == 0
    Hn.check_all(p, out, ref)
    return out, ref


def _positive_dt(p):
    # without softplus and bias the raw dt is dt' itself: keep it a valid step size
    p.dt = (1e-3 + 0.05 * np.abs(p.dt)).astype(np.float32)
    return p


SMALL = {
    "tiny_fp32": lambda: W.workload("tiny"),
    "bf16_ragged": lambda: W.make_problem([1, 5, 127, 128, 129, 300, 0, 513], nheads=8, headdim=64,
                                          dstate=128, ngroups=2, num_slots=64, seed=31),
    "bf16_cache_continue": lambda: W.make_problem([32, 200, 1, 0], nheads=8, headdim=64, dstate=128,
                                                  ngroups=4, state_dtype="bf16", num_slots=16,
                                                  has_init=[1, 1, 0, 1], cache_std=0.1, seed=32),
    "fp16_cache_continue": lambda: W.make_problem([70, 3], nheads=4, headdim=64, dstate=128,
                                                  ngroups=1, state_dtype="f16", num_slots=5,
                                                  has_init=True, cache_std=0.1, seed=33),
    "mtp_small": lambda: W.make_problem([3] * 16, nheads=8, headdim=64, dstate=128, ngroups=2,
                                        num_slots=32, has_init=True, write_final=False,
                                        want_intermediate=True, cache_std=0.1, seed=34),
    "no_softplus_no_bias_no_D": lambda: _positive_dt(W.make_problem(
        [40, 257], nheads=4, headdim=64, dstate=128, ngroups=2, dt_softplus=False,
        with_dt_bias=False, with_D=False, num_slots=4, seed=35)),
    "odd_shape_fp32": lambda: W.make_problem([17, 1, 90], nheads=6, headdim=24, dstate=40,
                                             ngroups=3, io_dtype="f32", num_slots=3,
                                             has_init=[0, 1, 1], seed=36),
    "odd_shape_bf16_inter": lambda: W.make_problem([9, 4], nheads=2, headdim=72, dstate=200,
                                                   ngroups=1, state_dtype="bf16", num_slots=2,
                                                   want_intermediate=True, seed=37),
    "no_final_writeback": lambda: W.make_problem([64, 130], nheads=4, headdim=64, dstate=128,
                                                 ngroups=2, write_final=False, num_slots=2,
                                                 has_init=True, seed=38),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_parity_small(name):
    _run_and_check(SMALL[name]())


def _check_d_zero(p):
    out = Hn.run_gpu(p)
    ref = oracle.ssd_scan_reference(p)
    assert out["status"] == 0
    ry = Hn.check_y(out["y"], ref["y"], p.io_dtype)
    rs = max(Hn.check_state(out["cache"][int(p.slot_idx[s])], ref["final"][s], p.state_dtype)
             for s in range(p.num_seqs))
    print("D = 0 %s: max y error %.3f x tolerance, max state error %.3f x tolerance"
          % (p.name, ry, rs))
    return ry


@pytest.mark.parametrize("init,state_dtype", [(False, "f32"), (True, "bf16"), (True, "f32")])
def test_d_zero_checks_scan_part_tightly(init, state_dtype):
    """With D = 0, y is the scan part alone, so the 2e-2 rms bound applies to it.
    Initial states use the continued-prefill scale N(0, 0.1); from an fp32 cache
    they enter y through the hi + lo bf16 parts of the state."""
    p = W.make_problem([100, 250, 7], nheads=8, headdim=64, dstate=128, ngroups=2, with_D=False,
                       num_slots=8, has_init=[1, 0, 1] if init else False, cache_std=0.1,
                       state_dtype=state_dtype, seed=39, name="small_%s_init%d" % (state_dtype, init))
    _check_d_zero(p)


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_d_zero_continued_prefill_shapes(state_dtype):
    """The continued-prefill shapes (suffixes 32, 600 and 1600 tokens, 128 heads in 8
    groups) from initial states, D = 0: the state's contribution to y is checked at
    the y bound with nothing else to hide it."""
    p = W.make_problem([32, 600, 1600], nheads=128, headdim=64, dstate=128, ngroups=8,
                       with_D=False, state_dtype=state_dtype, num_slots=16, has_init=True,
                       cache_std=0.1, seed=58, name="continued_%s" % state_dtype)
    _check_d_zero(p)


def test_d_zero_varlen_batch_with_initial_states():
    """A packed varlen batch (1 to 1,500 tokens, unaligned boundaries) where every
    other sequence continues from an fp32 initial state, D = 0."""
    rng = np.random.default_rng(59)
    lens = rng.integers(1, 1500, size=12)
    p = W.make_problem(lens, nheads=16, headdim=64, dstate=128, ngroups=4, with_D=False,
                       num_slots=24, has_init=(np.arange(12) % 2).astype(np.uint8),
                       cache_std=0.3, seed=59, name="varlen_init")
    _check_d_zero(p)


def test_block_alignment_invariance():
    """The tensor-core kernel cuts every sequence into 128-token blocks counted
    from the sequence's own first token.  The same sequences packed after a
    filler of 0, 1, 64 or 127 tokens (so at every alignment mod 128) must give
    bit-identical y and final states."""
    base = W.make_problem([300, 129, 45], nheads=4, headdim=64, dstate=128, ngroups=1,
                          num_slots=8, has_init=[1, 0, 1], cache_std=0.1, seed=40)
    outs = []
    for off in (0, 1, 64, 127):
        filler = W.make_problem([off], nheads=4, headdim=64, dstate=128, ngroups=1,
                                num_slots=8, seed=140 + off)
        p = W.select_sequences(base, [0, 1, 2])
        # prepend the filler's tokens as a sequence of its own (slot 7, no initial state)
        cat = lambda a, b: np.concatenate([a, b])
        p.x, p.dt, p.B, p.C = cat(filler.x, p.x), cat(filler.dt, p.dt), cat(filler.B, p.B), cat(filler.C, p.C)
        p.cu_seqlens = np.concatenate([[0], off + base.cu_seqlens]).astype(np.int32)
        p.slot_idx = np.concatenate([[7], base.slot_idx]).astype(np.int32)
        p.has_init = np.concatenate([[0], base.has_init]).astype(np.uint8)
        out = Hn.run_gpu(p, slots_disjoint=True)
        assert out["status"] == 0 and out["path"] == "chunked_tc"
        outs.append((out["y"][off:], out["cache"][base.slot_idx]))
    for y, cache in outs[1:]:
        np.testing.assert_array_equal(y, outs[0][0])
        np.testing.assert_array_equal(cache, outs[0][1])
    Hn.check_y(outs[0][0], oracle.ssd_scan_reference(base)["y"], base.io_dtype)


def test_sequence_permutation_bit_identical():
    p = W.make_problem([50, 180, 7, 129], nheads=4, headdim=64, dstate=128, ngroups=2,
                       num_slots=8, has_init=[1, 0, 1, 0], seed=41)
    out = Hn.run_gpu(p)
    order = [2, 0, 3, 1]
    q = W.select_sequences(p, order)
    outq = Hn.run_gpu(q)
    cu, cq = p.cu_seqlens, q.cu_seqlens
    for j, s in enumerate(order):
        np.testing.assert_array_equal(outq["y"][cq[j]:cq[j + 1]], out["y"][cu[s]:cu[s + 1]])
        np.testing.assert_array_equal(outq["cache"][p.slot_idx[s]], out["cache"][p.slot_idx[s]])


@pytest.mark.parametrize("P,N,io,lens", [
    (64, 128, "bf16", [3, 3, 2, 40]),       # eight rows a warp, staged asynchronously, > 16 tokens
    (64, 128, "f32", [3, 1, 3]),            # the same with fp32 inputs
    (48, 96, "bf16", [3, 2, 3]),            # rows not a multiple of the CTA's: register-free plain loop
    (64, 100, "bf16", [2, 3]),              # N not 128: the plain loop
])
def test_token_path_variants_with_per_token_states(P, N, io, lens):
    """The token-by-token kernel's wide-state variants, with the state after
    every token written (the MTP shape) and initial states from the cache."""
    p = W.make_problem(lens, nheads=4, headdim=P, dstate=N, ngroups=2, io_dtype=io,
                       num_slots=len(lens) + 2, has_init=True, want_intermediate=True,
                       cache_std=0.1, seed=50 + P + N + len(lens))
    out = Hn.run_gpu(p, max_seqlen=3 if max(lens) <= 3 else 0)
    assert out["path"] == "recurrent"
    Hn.check_all(p, out, oracle.ssd_scan_reference(p))


def test_short_path_hint_agrees_with_general_path():
    p = W.make_problem([3, 2, 1, 3], nheads=8, headdim=64, dstate=128, ngroups=2, num_slots=8,
                       has_init=True, cache_std=0.1, seed=42)
    a = Hn.run_gpu(p, max_seqlen=3)
    b = Hn.run_gpu(p, max_seqlen=0)
    ref = oracle.ssd_scan_reference(p)
    Hn.check_all(p, a, ref)
    Hn.check_all(p, b, ref)


def test_bad_slot_sets_device_status_and_skips_only_that_sequence():
    p = W.make_problem([20, 30, 10], nheads=4, headdim=64, dstate=128, ngroups=2, num_slots=4,
                       slots=[1, 9, 2], seed=43)
    out = Hn.run_gpu(p)
    assert out["status"] & 1
    good = W.select_sequences(p, [0, 2])
    ref = oracle.ssd_scan_reference(good)
    cu = p.cu_seqlens
    rows = np.r_[cu[0]:cu[1], cu[2]:cu[3]]
    Hn.check_y(out["y"][rows], ref["y"], p.io_dtype)
    assert np.all(np.isnan(out["y"][cu[1]:cu[2]]))        # skipped: left unwritten
    for s, q in ((0, 0), (2, 1)):
        Hn.check_state(out["cache"][p.slot_idx[s]], ref["final"][q], p.state_dtype)
    np.testing.assert_array_equal(out["cache"][[0, 3]], p.cache[[0, 3]])


def test_bad_cu_seqlens_sets_device_status():
    p = W.make_problem([20, 30], nheads=4, headdim=64, dstate=128, ngroups=2, num_slots=2, seed=44)
    p.cu_seqlens = np.array([0, 60, 50], dtype=np.int32)    # decreasing, beyond T
    out = Hn.run_gpu(p, max_seqlen=64)
    assert out["status"] & 2


# ---------------------------------------------------------------------------
# named full-size workloads: full GPU run, sampled oracle comparison
# ---------------------------------------------------------------------------
def _sampled(p, seqs, heads):
    out = Hn.run_gpu(p)
    assert out["status"] == 0
    q = W.select_sequences(p, seqs)
    ref = oracle.ssd_scan_reference(q, heads=heads)
    rows = np.concatenate([np.arange(p.cu_seqlens[s], p.cu_seqlens[s + 1]) for s in seqs])
    h0, h1 = heads
    Hn.check_y(out["y"][rows][:, h0:h1], ref["y"][:, h0:h1], p.io_dtype)
    named = set(int(s) for s in p.slot_idx) if p.write_final else set()
    untouched = [i for i in range(p.num_slots) if i not in named]
    np.testing.assert_array_equal(out["cache"][untouched], p.cache[untouched])
    if p.write_final:
        for j, s in enumerate(seqs):
            Hn.check_state(out["cache"][p.slot_idx[s], h0:h1], ref["final"][j, h0:h1],
                           p.state_dtype)
    if p.want_intermediate:
        for j, t in enumerate(rows):
            Hn.check_state(out["inter"][t, h0:h1], ref["inter"][j, h0:h1], p.state_dtype)
    assert out["launches"] <= 2
    return out


def test_workload_dense_prefill_sampled():
    _sampled(W.workload("dense_prefill"), [0, 7], (0, 16))


def test_workload_varlen_prefill_sampled():
    p = W.workload("varlen_prefill")
    lens = p.seqlens
    order = np.argsort(lens)
    seqs = sorted(set([int(order[0]), int(order[1]), int(order[-1]), 3, 17]))
    _sampled(p, seqs, (16, 32))


def test_workload_continued_a():
    _sampled(W.workload("continued_a"), [0], (0, 128))


def test_workload_continued_b_sampled():
    _sampled(W.workload("continued_b"), [0, 1, 2], (0, 32))


def test_workload_mtp_sampled():
    _sampled(W.workload("mtp"), [0, 5, 127], (0, 128))


def test_tensor_core_path_is_taken_for_bf16_prefill():
    """bf16 I/O with headdim 64 / d_state 128 runs the tcgen05 path: one launch for a
    batch of at most 32 sequences (sorted inside the scan kernel), two beyond."""
    p = W.make_problem([200, 64], nheads=4, headdim=64, dstate=128, ngroups=2, num_slots=4,
                       seed=45)
    out, _ = _run_and_check(p)
    assert out["path"] == "chunked_tc"
    assert out["launches"] == 1
    r = W.make_problem(np.arange(33) * 3 + 1, nheads=4, headdim=64, dstate=128, ngroups=2,
                       num_slots=33, seed=56)
    outr, _ = _run_and_check(r)
    assert outr["path"] == "chunked_tc" and outr["launches"] == 2
    q = W.make_problem([3, 3], nheads=4, headdim=64, dstate=128, ngroups=2, num_slots=4,
                       has_init=True, seed=46)
    outq = Hn.run_gpu(q, max_seqlen=3, slots_disjoint=True)
    assert outq["path"] == "recurrent" and outq["launches"] == 1
    # without the caller's promise of disjoint slots the snapshot pass runs first
    assert Hn.run_gpu(q, max_seqlen=3)["launches"] == 2


def test_many_short_sequences_and_empty_ones():
    """Varlen batch with more work items than SMs, empty sequences and 1-token tails."""
    rng = np.random.default_rng(47)
    lens = rng.integers(0, 300, size=60)
    lens[::7] = 0
    lens[1::9] = 1
    p = W.make_problem(lens, nheads=8, headdim=64, dstate=128, ngroups=2, num_slots=80,
                       has_init=(rng.random(60) < 0.5).astype(np.uint8), cache_std=0.3, seed=47)
    _run_and_check(p)


@pytest.mark.parametrize("regime", ["steep", "flat"])
def test_decay_regimes(regime):
    """Steep decay (32-token blocks decaying by more than e^80: per-element exp path and a
    renormalised state every block) and near-zero decay (the running scale never renormalises)."""
    p = W.make_problem([700, 129, 40], nheads=4, headdim=64, dstate=128, ngroups=2, num_slots=4,
                       has_init=[1, 0, 1], cache_std=0.1, dt_softplus=False, with_dt_bias=False,
                       state_dtype="f32", seed=48)
    rng = np.random.default_rng(49)
    if regime == "steep":
        p.dt = rng.uniform(0.3, 0.6, size=p.dt.shape).astype(np.float32)
        p.A = np.array([-16.0, -12.0, -9.0, -3.0], dtype=np.float32)
    else:
        p.dt = rng.uniform(0.001, 0.1, size=p.dt.shape).astype(np.float32)
        p.A = np.array([-1e-3, -1e-4, -2e-3, 0.0], dtype=np.float32)
    _run_and_check(p)


def test_long_single_sequence_keeps_state_accuracy():
    """One 40,000-token sequence (313 blocks) from an initial state: the final
    state still meets the fp32-storage tolerance after every block's update, and
    y agrees at the start, the middle and the end of the sequence."""
    p = W.make_problem([40000], nheads=2, headdim=64, dstate=128, ngroups=1, num_slots=3,
                       has_init=[1], cache_std=0.3, seed=51)
    out = Hn.run_gpu(p)
    assert out["status"] == 0 and out["path"] == "chunked_tc"
    ref = oracle.ssd_scan_reference(p)
    Hn.check_state(out["cache"][p.slot_idx[0]], ref["final"][0], p.state_dtype)
    for a, b in ((0, 512), (19968, 20480), (39488, 40000)):
        Hn.check_y(out["y"][a:b], ref["y"][a:b], p.io_dtype)


def test_more_sequences_than_the_longest_first_sort_holds():
    """8,200 short sequences (4 to 9 tokens) on the tensor-core path: more than the
    prep kernel sorts, so the sequences are dealt in their given order."""
    rng = np.random.default_rng(52)
    lens = rng.integers(4, 10, size=8200)
    p = W.make_problem(lens, nheads=2, headdim=64, dstate=128, ngroups=1, num_slots=8200,
                       cache_std=0.1, seed=52)
    out, _ = _run_and_check(p)
    assert out["path"] == "chunked_tc"


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_segments_hand_over_the_state_between_ctas(state_dtype):
    """Eight 2,900-5,200-token sequences x 40 head pairs (more items than SMs): the
    prep kernel cuts each item into up to four 11-block segments run by different
    CTAs, the state passing through the workspace in fp32.  Initial states from the
    cache for half of the sequences, final states written back."""
    rng = np.random.default_rng(53)
    lens = rng.integers(2900, 5200, size=8)
    p = W.make_problem(lens, nheads=80, headdim=64, dstate=128, ngroups=1, num_slots=12,
                       has_init=[1, 0, 1, 0, 0, 1, 1, 0], cache_std=0.1, state_dtype=state_dtype,
                       seed=53)
    out = _sampled(p, [0, 2, 7], (24, 40))
    assert out["path"] == "chunked_tc"


def test_seven_segments_per_item():
    """Four ~8,100-token sequences x 40 head pairs: 10-block segments, seven per
    item (a chain of six hand-overs through the workspace), every sequence from
    an initial state."""
    rng = np.random.default_rng(54)
    lens = rng.integers(8100, 8193, size=4)
    p = W.make_problem(lens, nheads=80, headdim=64, dstate=128, ngroups=2, num_slots=6,
                       has_init=True, cache_std=0.3, seed=54)
    out = _sampled(p, [1, 3], (56, 72))
    assert out["path"] == "chunked_tc"


def test_longest_first_sort_of_thousands_of_sequences():
    """3,000 sequences of 1-300 tokens (many equal block counts): the prep kernel's
    bitonic sort over 4,096 keys (padded) orders them longest first; every output
    and final state is compared."""
    rng = np.random.default_rng(55)
    lens = rng.integers(1, 41, size=3000)
    lens[::97] = rng.integers(200, 301, size=lens[::97].shape[0])
    p = W.make_problem(lens, nheads=2, headdim=64, dstate=128, ngroups=1, num_slots=3000,
                       has_init=(rng.random(3000) < 0.3).astype(np.uint8), cache_std=0.1, seed=55)
    out, _ = _run_and_check(p)
    assert out["path"] == "chunked_tc"


def test_segments_with_an_empty_sequence_and_a_bad_slot():
    """A batch the prep kernel cuts into segments that also holds an empty
    sequence and one whose slot is out of range: the bad sequence is skipped in
    every segment (its y rows stay unwritten, the device status says so), the
    empty one gets its slot zeroed, and the others match the oracle."""
    rng = np.random.default_rng(57)
    lens = rng.integers(2900, 5200, size=9)
    lens[4] = 0
    slots = list(range(9))
    slots[6] = 40                                   # outside [0, num_slots)
    p = W.make_problem(lens, nheads=80, headdim=64, dstate=128, ngroups=1, num_slots=12,
                       slots=slots, has_init=[1, 0, 1, 0, 0, 1, 0, 0, 1], cache_std=0.1, seed=57)
    out = Hn.run_gpu(p)
    assert out["status"] & 1 and out["path"] == "chunked_tc"
    cu = p.cu_seqlens
    assert np.all(np.isnan(out["y"][cu[6]:cu[7]]))
    np.testing.assert_array_equal(out["cache"][4], np.zeros_like(out["cache"][4]))
    good = [0, 3, 8]
    q = W.select_sequences(p, good)
    ref = oracle.ssd_scan_reference(q, heads=(40, 56))
    rows = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in good])
    Hn.check_y(out["y"][rows][:, 40:56], ref["y"][:, 40:56], p.io_dtype)
    for j, s in enumerate(good):
        Hn.check_state(out["cache"][p.slot_idx[s], 40:56], ref["final"][j, 40:56], p.state_dtype)
    untouched = [i for i in range(p.num_slots) if i not in set(slots)]
    np.testing.assert_array_equal(out["cache"][untouched], p.cache[untouched])

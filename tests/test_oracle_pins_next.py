"""Pins of the oracle's optional parts (CPU only): per-chunk checkpoint states,
snapshot slot semantics with separate final slots, the Philox4x32-10
generator, stochastic rounding to fp16 and the ReplaySSM verification step.
Each is checked against something other than the oracle's own code path: the
NumPy dual form on prefixes, single-sequence runs on the untouched cache, the
generator's published known-answer vectors, a brute-force search over fp16
values, and the dual form over the replayed history."""
import numpy as np
import pytest

import oracle
from state_space_model_varlen_gb300 import workloads as W
from tests.dual_form import dual_form_head


# --------------------------------------------------------------------------
# per-chunk (checkpoint) states
# --------------------------------------------------------------------------
@pytest.mark.parametrize("L", [1, 4, 7, 16])
def test_chunk_states_are_prefix_states_of_the_dual_form(L):
    """Row cu_chunks[s] + c is the state after token min((c+1) L, len) - 1 of
    sequence s: the dual form run on that prefix gives it independently."""
    p = W.make_problem([13, 0, 16, 5], nheads=4, headdim=3, dstate=5, ngroups=2, io_dtype="f32",
                       num_slots=6, has_init=[1, 0, 0, 1], chunk_size=L, seed=61)
    p.want_chunk_states = 1
    r = oracle.ssd_scan_reference(p)
    cuc, cu = p.cu_chunks, p.cu_seqlens
    assert r["chunks"].shape[0] == cuc[-1]
    for s in range(p.num_seqs):
        a, b = int(cu[s]), int(cu[s + 1])
        for c in range(int(cuc[s + 1] - cuc[s])):
            end = min((c + 1) * L, b - a)
            for h in range(p.nheads):
                g = h // 2
                h0 = p.cache[p.slot_idx[s], h].astype(np.float64) if p.has_init[s] else None
                _, hh = dual_form_head(p.x[a:a + end, h], p.dt[a:a + end, h], float(p.A[h]),
                                       p.B[a:a + end, g].astype(np.float64),
                                       p.C[a:a + end, g].astype(np.float64),
                                       D=float(p.D[h]), h0=h0, dt_bias=float(p.dt_bias[h]))
                np.testing.assert_allclose(r["chunks"][cuc[s] + c, h], hh, rtol=1e-10, atol=1e-12)
        if b > a:
            np.testing.assert_array_equal(r["chunks"][cuc[s + 1] - 1], r["final"][s])


# --------------------------------------------------------------------------
# snapshot semantics: crossed and shared slots, separate final slots
# --------------------------------------------------------------------------
def test_crossed_and_shared_slots_read_the_cache_before_the_call():
    """Sequence 0 reads slot 1 and writes slot 2, sequence 1 reads slot 2 and
    writes slot 1 (crossed); sequences 2 and 3 both read slot 4 (shared) and
    write slots 0 and 5.  Each must see the cache as it was before the call:
    its result equals that sequence run alone on the untouched cache."""
    p = W.make_problem([9, 14, 6, 11], nheads=4, headdim=3, dstate=4, ngroups=2, io_dtype="f32",
                       num_slots=6, slots=[1, 2, 4, 4], has_init=True, seed=62)
    p.final_slot_idx = np.array([2, 1, 0, 5], dtype=np.int32)
    r = oracle.ssd_scan_reference(p)
    cu = p.cu_seqlens
    for s in range(p.num_seqs):
        q = W.select_sequences(p, [s])
        q.final_slot_idx = None
        alone = oracle.ssd_scan_reference(q)
        np.testing.assert_array_equal(r["y"][cu[s]:cu[s + 1]], alone["y"])
        np.testing.assert_array_equal(r["cache"][p.final_slot_idx[s]], alone["cache"][p.slot_idx[s]])
    np.testing.assert_array_equal(r["cache"][3], p.cache[3])         # neither read nor written
    np.testing.assert_array_equal(r["cache"][4], p.cache[4])         # read only


# --------------------------------------------------------------------------
# Philox4x32-10
# --------------------------------------------------------------------------
# Known-answer vectors published with the generator (Random123 distribution,
# kat_vectors, philox4x32 with 10 rounds): counter, key -> output.
PHILOX_KAT = [
    ((0x00000000, 0x00000000, 0x00000000, 0x00000000), (0x00000000, 0x00000000),
     (0x6627e8d5, 0xe169c58d, 0xbc57ac4c, 0x9b00dbd8)),
    ((0xffffffff, 0xffffffff, 0xffffffff, 0xffffffff), (0xffffffff, 0xffffffff),
     (0x408f276d, 0x41c83b0e, 0xa20bc7c6, 0x6d5451fd)),
    ((0x243f6a88, 0x85a308d3, 0x13198a2e, 0x03707344), (0xa4093822, 0x299f31d0),
     (0xd16cfe09, 0x94fdcceb, 0x5001e420, 0x24126ea1)),
]


@pytest.mark.parametrize("ctr,key,want", PHILOX_KAT)
def test_philox_known_answers(ctr, key, want):
    got = oracle.philox4x32_10([np.array([c], np.uint32) for c in ctr], key)
    assert tuple(int(g[0]) for g in got) == want


# --------------------------------------------------------------------------
# stochastic rounding to fp16
# --------------------------------------------------------------------------
def _f16_neighbours(v32):
    """Brute force: the fp16 values just below and above |v| (toward and away
    from zero) found with NumPy's own float16 conversion and nextafter."""
    a = np.abs(v32.astype(np.float64))
    near = a.astype(np.float16).astype(np.float64)
    lo = np.where(near > a, np.nextafter(near.astype(np.float16), np.float16(0)).astype(np.float64), near)
    hi = np.nextafter(lo.astype(np.float16), np.float16(np.inf)).astype(np.float64)
    return lo, hi


def test_sr_picks_a_neighbour_with_the_defined_probability():
    rng = np.random.default_rng(63)
    v = (rng.standard_normal(20000) * 10.0 ** rng.integers(-6, 4, 20000)).astype(np.float32)
    r = rng.integers(0, 2 ** 32, size=v.shape, dtype=np.uint64).astype(np.uint32)
    got = np.abs(oracle.sr_round_f16(v, r).astype(np.float64))
    lo, hi = _f16_neighbours(v)
    frac = (np.abs(v.astype(np.float64)) - lo) / (hi - lo)
    want = np.where(frac * 2.0 ** 32 > r.astype(np.float64), hi, lo)
    np.testing.assert_array_equal(got, want)
    assert np.all(np.signbit(oracle.sr_round_f16(v, r)) == np.signbit(v))


def test_sr_exact_values_and_extreme_words():
    ex = np.array([0.0, 1.0, -2.5, 65504.0, 2.0 ** -24, -(2.0 ** -14)], dtype=np.float32)
    for r in (0, 2 ** 31, 2 ** 32 - 1):
        np.testing.assert_array_equal(oracle.sr_round_f16(ex, np.full(ex.shape, r, np.uint32)),
                                      ex.astype(np.float16))
    v = np.array([1.0 + 2.0 ** -12, 1.0 + 2.0 ** -11 + 2.0 ** -13], dtype=np.float32)
    up = oracle.sr_round_f16(v, np.zeros(2, np.uint32)).astype(np.float64)       # r = 0: away from 0
    dn = oracle.sr_round_f16(v, np.full(2, 2 ** 32 - 1, np.uint32)).astype(np.float64)
    np.testing.assert_array_equal(up, [1.0 + 2.0 ** -10, 1.0 + 2.0 ** -10])
    np.testing.assert_array_equal(dn, [1.0, 1.0])                                 # fractions < 1
    assert np.isinf(oracle.sr_round_f16(np.array([70000.0], np.float32), np.zeros(1, np.uint32))[0])


def test_sr_is_unbiased():
    """The mean of many stochastic roundings of v is v (within 5 sigma)."""
    rng = np.random.default_rng(64)
    for v in (1.0 + 2.0 ** -13, 3.14159, -0.000123, 1000.3):
        n = 200000
        r = rng.integers(0, 2 ** 32, size=n, dtype=np.uint64).astype(np.uint32)
        out = oracle.sr_round_f16(np.full(n, v, np.float32), r).astype(np.float64)
        lo, hi = _f16_neighbours(np.array([v], np.float32))
        sd = (hi[0] - lo[0]) / 2 / np.sqrt(n)
        assert abs(out.mean() - np.float32(v)) < 5 * sd + 1e-12


def test_sr_words_follow_the_element_index():
    """Element e of the written rows takes word e mod 4 of the block e >> 2."""
    seed = 0x123456789
    w = oracle.sr_words(seed, 3, (1, 2), 4, 2, 8, stream=0)
    base = (3 * 4 + 1) * 2 * 8
    for k in (0, 1, 5, 15):
        e = base + k
        ref = oracle.philox4x32_10([np.array([e >> 2], np.uint32), np.array([0], np.uint32),
                                    np.array([0], np.uint32), np.array([0], np.uint32)],
                                   (seed & 0xFFFFFFFF, seed >> 32))
        assert int(w.reshape(-1)[k]) == int(ref[e & 3][0])


# --------------------------------------------------------------------------
# ReplaySSM verification step
# --------------------------------------------------------------------------
def _replay_problem(K, S, seed, R=8, window=5, counts=None, slots=None):
    p = W.make_problem([K] * S, nheads=4, headdim=3, dstate=4, ngroups=2, io_dtype="f32",
                       num_slots=S + 2, slots=slots, has_init=True, write_final=False,
                       cache_std=0.3, seed=seed)
    rng = np.random.default_rng(seed + 1000)
    H, P, N, G = p.nheads, p.headdim, p.dstate, p.ngroups
    ring = {"x": rng.standard_normal((p.num_slots, R, H, P)).astype(np.float32),
            "dt": np.clip(rng.standard_normal((p.num_slots, R, H)), -2.3, 2.3).astype(np.float32),
            "B": (rng.standard_normal((p.num_slots, R, G, N)) / 2).astype(np.float32),
            "start": rng.integers(0, R, size=S),
            "count": np.array(counts if counts is not None else rng.integers(0, window + 1, size=S)),
            "window": window}
    return p, ring


def test_replay_matches_the_dual_form_over_the_history():
    """y of the window equals the dual form run from the checkpoint over the
    pending ring inputs followed by the window; a folded checkpoint equals the
    dual-form state after the pending inputs; the window lands in the ring after
    the pending entries."""
    p, ring = _replay_problem(3, 5, seed=65, counts=[0, 1, 2, 4, 5])
    r = oracle.replay_reference(p, ring)
    R = ring["x"].shape[1]
    cu = p.cu_seqlens
    for s in range(p.num_seqs):
        q = int(p.slot_idx[s])
        cnt, st = int(ring["count"][s]), int(ring["start"][s])
        pos = [(st + j) % R for j in range(cnt)]
        a, b = int(cu[s]), int(cu[s + 1])
        for h in range(p.nheads):
            g = h // 2
            xs = np.concatenate([ring["x"][q, pos, h], p.x[a:b, h]]).astype(np.float64)
            dts = np.concatenate([ring["dt"][q, pos, h], p.dt[a:b, h]])
            Bs = np.concatenate([ring["B"][q, pos, g], p.B[a:b, g]]).astype(np.float64)
            Cs = np.concatenate([np.zeros((cnt, p.dstate)), p.C[a:b, g]])
            y, _ = dual_form_head(xs, dts, float(p.A[h]), Bs, Cs, D=float(p.D[h]),
                                  h0=p.cache[q, h].astype(np.float64), dt_bias=float(p.dt_bias[h]))
            np.testing.assert_allclose(r["y"][a:b, h], y[cnt:], rtol=1e-10, atol=1e-12)
            fold = cnt + (b - a) > ring["window"]
            if fold:
                _, hp = dual_form_head(xs[:cnt], dts[:cnt], float(p.A[h]), Bs[:cnt], Cs[:cnt],
                                       h0=p.cache[q, h].astype(np.float64), dt_bias=float(p.dt_bias[h]))
                np.testing.assert_allclose(r["cache"][q, h], hp.astype(np.float32), rtol=1e-6)
                assert (r["start"][s], r["count"][s]) == ((st + cnt) % R, 0)
            else:
                np.testing.assert_array_equal(r["cache"][q, h], p.cache[q, h])
                assert (r["start"][s], r["count"][s]) == (st, cnt)
        for i in range(b - a):
            w = (st + cnt + i) % R
            np.testing.assert_array_equal(r["ring_x"][q, w], p.x[a + i])
            np.testing.assert_array_equal(r["ring_B"][q, w], p.B[a + i])


def test_two_replay_steps_equal_one_scan_over_the_accepted_tokens():
    """Step 1 verifies a window of 3, the caller accepts 2; step 2 verifies the
    next window: its y equals a plain scan from the original checkpoint over
    (pending, accepted tokens of step 1, window of step 2)."""
    p1, ring = _replay_problem(3, 4, seed=66, counts=[0, 2, 3, 1])
    r1 = oracle.replay_reference(p1, ring)
    acc = 2
    ring2 = {"x": r1["ring_x"], "dt": r1["ring_dt"], "B": r1["ring_B"], "window": ring["window"],
             "start": r1["start"], "count": r1["count"] + acc}
    p2, _ = _replay_problem(3, 4, seed=67, slots=list(p1.slot_idx))
    p2.cache = r1["cache"]
    p2.A, p2.D, p2.dt_bias = p1.A, p1.D, p1.dt_bias          # the same layer
    r2 = oracle.replay_reference(p2, ring2)
    R = ring["x"].shape[1]
    folded = 0
    for s in range(p1.num_seqs):
        q1 = int(p1.slot_idx[s])
        folded += int(r1["count"][s] == 0 and ring["count"][s] > 0) + int(r2["count"][s] == 0)
        cnt, st = int(ring["count"][s]), int(ring["start"][s])
        pos = [(st + j) % R for j in range(cnt)]
        a1, b1 = int(p1.cu_seqlens[s]), int(p1.cu_seqlens[s]) + acc
        a2, b2 = int(p2.cu_seqlens[s]), int(p2.cu_seqlens[s + 1])
        for h in range(p1.nheads):
            g = h // 2
            xs = np.concatenate([ring["x"][q1, pos, h], p1.x[a1:b1, h], p2.x[a2:b2, h]]).astype(np.float64)
            dts = np.concatenate([ring["dt"][q1, pos, h], p1.dt[a1:b1, h], p2.dt[a2:b2, h]])
            Bs = np.concatenate([ring["B"][q1, pos, g], p1.B[a1:b1, g], p2.B[a2:b2, g]]).astype(np.float64)
            Cs = np.concatenate([np.zeros((cnt + acc, p1.dstate)), p2.C[a2:b2, g]])
            y, _ = dual_form_head(xs, dts, float(p2.A[h]), Bs, Cs, D=float(p2.D[h]),
                                  h0=p1.cache[q1, h].astype(np.float64),
                                  dt_bias=float(p2.dt_bias[h]))
            np.testing.assert_allclose(r2["y"][a2:b2, h], y[cnt + acc:], rtol=1e-5, atol=1e-6)
    assert folded > 0           # some request folded its ring into the checkpoint on the way

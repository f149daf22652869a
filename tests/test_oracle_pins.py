"""Pins of the fp64 oracle against things other than itself (CPU only).

Each test checks the oracle against a value fixed by the mathematics of the
recurrence, not by re-typing the oracle's loop: a hand-worked example, closed
forms (A = 0 prefix sums, constant-input geometric decay), the O(T^2) dual
form, split/resume invariance through the state cache, linearity, sequence
independence of a packed batch and the head-to-group mapping.  A plausible
slip in the oracle (dropped term, wrong sign or index, transposed p/n,
y taken before the update, wrong group) fails at least one of them; the
``test_planted_*`` cases show that for a few such slips, planted in a copy of
the oracle's arithmetic on the CPU.
"""
import os

import numpy as np
import pytest

import oracle
from state_space_model_varlen_gb300 import workloads as W
from tests.dual_form import dual_form_head

HERE = os.path.dirname(os.path.abspath(__file__))


def _golden(name):
    vals = {}
    with open(os.path.join(HERE, "golden", name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, *v = line.split()
                vals[k] = np.array([float(t) for t in v])
    return vals


def _rand(rng, *shape):
    return rng.standard_normal(shape)


# --------------------------------------------------------------------------
# hand-worked example
# --------------------------------------------------------------------------
def test_hand_worked_example():
    g = _golden("hand_worked_3tok.txt")
    x = g["x"].reshape(3, 1, 2)
    B = g["B"].reshape(3, 1, 2)
    C = g["C"].reshape(3, 1, 2)
    dt = g["dt"].reshape(3, 1)
    y, hf, hint = oracle.scan(x, dt, g["A"], B, C, [0, 3], dt_softplus=False, D=g["D"],
                              h_init=g["h_init"].reshape(1, 1, 2, 2), want_inter=True)
    np.testing.assert_allclose(y.reshape(-1), g["y"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(hf.reshape(-1), g["h_final"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(hint[0].reshape(-1), g["h_after_t0"], atol=1e-12)
    np.testing.assert_allclose(hint[1].reshape(-1), g["h_after_t1"], atol=1e-12)
    np.testing.assert_allclose(hint[2].reshape(-1), g["h_final"], atol=1e-12)


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------
def test_closed_form_A_zero_prefix_sums():
    """A = 0: no decay, the state is h0 + prefix sum of dt' x B^T."""
    rng = np.random.default_rng(11)
    L, H, P, N = 40, 3, 5, 7
    x, B, C = _rand(rng, L, H, P), _rand(rng, L, 1, N), _rand(rng, L, 1, N)
    dt = rng.uniform(0.01, 0.5, (L, H))
    D = _rand(rng, H)
    h0 = _rand(rng, 1, H, P, N)
    y, hf, hint = oracle.scan(x, dt, np.zeros(H), B, C, [0, L], dt_softplus=False, D=D,
                              h_init=h0, want_inter=True)
    terms = np.einsum("th,thp,tn->thpn", dt, x, B[:, 0])
    h_ref = h0[0][None] + np.cumsum(terms, axis=0)
    y_ref = np.einsum("tn,thpn->thp", C[:, 0], h_ref) + D[None, :, None] * x
    np.testing.assert_allclose(hint, h_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(hf[0], h_ref[-1], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(y, y_ref, rtol=1e-12, atol=1e-12)


def test_closed_form_constant_inputs_geometric():
    """Constant dt, A, x, B: h_t = a^(t+1) h0 + dt x B^T (1 - a^(t+1)) / (1 - a)."""
    rng = np.random.default_rng(12)
    L, P, N = 50, 4, 6
    d, Ah = 0.07, -3.0
    a = np.exp(d * Ah)
    xv, Bv, Cv = _rand(rng, P), _rand(rng, N), _rand(rng, N)
    h0 = _rand(rng, P, N)
    x = np.tile(xv, (L, 1, 1))
    B = np.tile(Bv, (L, 1, 1))
    C = np.tile(Cv, (L, 1, 1))
    y, hf, hint = oracle.scan(x, np.full((L, 1), d), [Ah], B, C, [0, L], dt_softplus=False,
                              h_init=h0[None, None], want_inter=True)
    k = np.arange(1, L + 1)[:, None, None]
    h_ref = a ** k * h0[None] + d * np.outer(xv, Bv)[None] * (1 - a ** k) / (1 - a)
    np.testing.assert_allclose(hint[:, 0], h_ref, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(y[:, 0], h_ref @ Cv, rtol=1e-11, atol=1e-13)


def test_single_token_written_out():
    """One token from a cached state: y = C (exp(dt' A) h0 + dt' x B^T) + D x."""
    rng = np.random.default_rng(13)
    H, P, N, G = 4, 3, 5, 2
    x, B, C = _rand(rng, 1, H, P), _rand(rng, 1, G, N), _rand(rng, 1, G, N)
    dt, bias = _rand(rng, 1, H), _rand(rng, H)
    A, D = -rng.uniform(1, 5, H), _rand(rng, H)
    h0 = _rand(rng, 1, H, P, N)
    y, hf, _ = oracle.scan(x, dt, A, B, C, [0, 1], dt_bias=bias, D=D, h_init=h0)
    for h in range(H):
        g = h // (H // G)
        d = np.log1p(np.exp(dt[0, h] + bias[h]))
        hh = np.exp(d * A[h]) * h0[0, h] + d * np.outer(x[0, h], B[0, g])
        np.testing.assert_allclose(hf[0, h], hh, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(y[0, h], hh @ C[0, g] + D[h] * x[0, h], rtol=1e-13, atol=1e-14)


# --------------------------------------------------------------------------
# brute force: dual form
# --------------------------------------------------------------------------
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_dual_form_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    lens = [int(v) for v in rng.integers(0, 40, size=4)] + [1]
    H, P, N, G = 4, 3, 5, 2
    p = W.make_problem(lens, nheads=H, headdim=P, dstate=N, ngroups=G, io_dtype="f32",
                       num_slots=8, has_init=[1, 0, 1, 1, 0], seed=seed)
    r = oracle.ssd_scan_reference(p)
    cu = p.cu_seqlens
    for s in range(p.num_seqs):
        a, b = cu[s], cu[s + 1]
        for h in range(H):
            g = h // (H // G)
            h0 = p.cache[p.slot_idx[s], h].astype(np.float64) if p.has_init[s] else None
            y, hh = dual_form_head(p.x[a:b, h], p.dt[a:b, h], float(p.A[h]),
                                   p.B[a:b, g].astype(np.float64), p.C[a:b, g].astype(np.float64),
                                   D=float(p.D[h]), h0=h0, dt_bias=float(p.dt_bias[h]))
            np.testing.assert_allclose(r["y"][a:b, h], y, rtol=1e-10, atol=1e-12)
            if b > a or h0 is not None:
                np.testing.assert_allclose(r["final"][s, h], hh if h0 is not None or b > a else 0,
                                           rtol=1e-10, atol=1e-12)


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------
def test_split_resume_invariance():
    """Prefix, then continuation from the carried state == the unsplit run."""
    rng = np.random.default_rng(21)
    L, H, P, N, G = 97, 4, 6, 8, 2
    x, B, C = _rand(rng, L, H, P), _rand(rng, L, G, N), _rand(rng, L, G, N)
    dt, A, D = _rand(rng, L, H) - 3, -rng.uniform(1, 8, H), _rand(rng, H)
    h0 = _rand(rng, 1, H, P, N)
    y, hf, _ = oracle.scan(x, dt, A, B, C, [0, L], D=D, h_init=h0)
    for k in (0, 1, 33, 96, 97):
        y1, h1, _ = oracle.scan(x[:k], dt[:k], A, B[:k], C[:k], [0, k], D=D, h_init=h0)
        y2, h2, _ = oracle.scan(x[k:], dt[k:], A, B[k:], C[k:], [0, L - k], D=D, h_init=h1)
        np.testing.assert_allclose(np.concatenate([y1, y2]), y, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(h2, hf, rtol=1e-12, atol=1e-12)


def test_packed_sequences_are_independent():
    """A packed batch equals each sequence run alone (state restarts at cu_seqlens)."""
    rng = np.random.default_rng(22)
    lens = [5, 0, 17, 1, 30]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, H, P, N = cu[-1], 2, 3, 4
    x, B, C = _rand(rng, T, H, P), _rand(rng, T, 1, N), _rand(rng, T, 1, N)
    dt, A = _rand(rng, T, H) - 3, -rng.uniform(1, 8, H)
    h0 = _rand(rng, len(lens), H, P, N)
    y, hf, _ = oracle.scan(x, dt, A, B, C, cu, h_init=h0)
    for s in range(len(lens)):
        a, b = cu[s], cu[s + 1]
        ys, hs, _ = oracle.scan(x[a:b], dt[a:b], A, B[a:b], C[a:b], [0, b - a], h_init=h0[s:s + 1])
        np.testing.assert_array_equal(y[a:b], ys)
        np.testing.assert_array_equal(hf[s], hs[0])
    np.testing.assert_array_equal(hf[1], h0[1])          # empty sequence keeps its state


def test_linearity_in_x_and_D_term():
    rng = np.random.default_rng(23)
    L, H, P, N = 31, 3, 4, 5
    x1, x2 = _rand(rng, L, H, P), _rand(rng, L, H, P)
    B, C = _rand(rng, L, 1, N), _rand(rng, L, 1, N)
    dt, A, D = _rand(rng, L, H) - 3, -rng.uniform(1, 8, H), _rand(rng, H)
    run = lambda xx, DD=None: oracle.scan(xx, dt, A, B, C, [0, L], D=DD)
    ya, ha, _ = run(x1)
    yb, hb, _ = run(x2)
    yc, hc, _ = run(2.0 * x1 - 3.0 * x2)
    np.testing.assert_allclose(yc, 2 * ya - 3 * yb, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(hc, 2 * ha - 3 * hb, rtol=1e-11, atol=1e-12)
    yd, _, _ = run(x1, D)
    np.testing.assert_allclose(yd - ya, D[None, :, None] * x1, rtol=1e-12, atol=1e-13)


def test_softplus_matches_library_routine():
    """dt_softplus=1 equals feeding NumPy's logaddexp(0, dt + bias) with softplus off."""
    rng = np.random.default_rng(24)
    L, H, P, N = 20, 3, 2, 3
    x, B, C = _rand(rng, L, H, P), _rand(rng, L, 1, N), _rand(rng, L, 1, N)
    dt, bias, A = 4 * _rand(rng, L, H), _rand(rng, H), -rng.uniform(1, 8, H)
    y1, h1, _ = oracle.scan(x, dt, A, B, C, [0, L], dt_bias=bias, dt_softplus=True)
    y2, h2, _ = oracle.scan(x, np.logaddexp(0.0, dt + bias), A, B, C, [0, L], dt_softplus=False)
    np.testing.assert_allclose(y1, y2, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(h1, h2, rtol=1e-13, atol=1e-14)


def test_group_mapping_contiguous_heads():
    """Head h reads group h // (H/G): compare with one-group runs per head."""
    rng = np.random.default_rng(25)
    L, H, P, N, G = 12, 6, 2, 3, 3
    x, B, C = _rand(rng, L, H, P), _rand(rng, L, G, N), _rand(rng, L, G, N)
    dt, A = _rand(rng, L, H) - 3, -rng.uniform(1, 8, H)
    y, hf, _ = oracle.scan(x, dt, A, B, C, [0, L])
    for h in range(H):
        g = h // 2
        yh, hh, _ = oracle.scan(x[:, h:h + 1], dt[:, h:h + 1], A[h:h + 1], B[:, g:g + 1],
                                C[:, g:g + 1], [0, L])
        np.testing.assert_array_equal(y[:, h], yh[:, 0])
        np.testing.assert_array_equal(hf[0, h], hh[0, 0])


# --------------------------------------------------------------------------
# slot handling and rounding of the writeback
# --------------------------------------------------------------------------
def _bf16_table():
    bits = np.arange(0, 1 << 15, dtype=np.uint32)          # sign bit clear
    vals = (bits << 16).view(np.float32)
    ok = np.isfinite(vals)
    with np.errstate(invalid="ignore"):
        vals = vals.astype(np.float64)
    order = np.argsort(vals[ok], kind="stable")
    return vals[ok][order], bits[ok][order].astype(np.uint16)


def test_round_to_bf16_is_nearest_even():
    vals, bits = _bf16_table()
    rng = np.random.default_rng(26)
    v = np.concatenate([np.abs(rng.standard_normal(4000)) * 10.0 ** rng.integers(-8, 8, 4000),
                        [1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, 1 + 2.0 ** -8 + 2.0 ** -40, 0.0]])
    got = oracle.round_to(v, "bf16")
    i = np.clip(np.searchsorted(vals, v), 1, len(vals) - 1)
    lo, hi = vals[i - 1], vals[i]
    pick_hi = (hi - v < v - lo) | ((hi - v == v - lo) & (bits[i] % 2 == 0))
    want = np.where(pick_hi, bits[i], bits[i - 1])
    np.testing.assert_array_equal(got, want)
    assert oracle.round_to(np.array([1 + 2.0 ** -8]), "bf16")[0] == 0x3F80     # tie -> even
    assert oracle.round_to(np.array([1 + 3 * 2.0 ** -8]), "bf16")[0] == 0x3F82


def test_reference_reads_and_writes_only_named_slots():
    p = W.make_problem([7, 0, 4], nheads=2, headdim=3, dstate=4, ngroups=1, io_dtype="bf16",
                       state_dtype="bf16", num_slots=6, slots=[4, 1, 2], has_init=[1, 1, 0],
                       seed=5)
    r = oracle.ssd_scan_reference(p)
    untouched = [0, 3, 5]
    np.testing.assert_array_equal(r["cache"][untouched], p.cache[untouched])
    # slot 1 holds an empty sequence with an initial state: written back unchanged
    np.testing.assert_array_equal(r["cache"][1], p.cache[1])
    # slot 2 had has_init = 0: its old contents must not leak into the result
    q = W.select_sequences(p, [2])
    q.cache[2] = 0
    r2 = oracle.ssd_scan_reference(q)
    np.testing.assert_array_equal(r2["cache"][2], r["cache"][2])


# --------------------------------------------------------------------------
# planted mistakes: each must be caught by one of the pins above
# --------------------------------------------------------------------------
def _python_recurrence(x, dt, A, B, C, D, h0, slip=None):
    """Tiny pure-Python copy of the recurrence with an optional planted slip."""
    L, P = x.shape
    N = B.shape[1]
    h = h0.copy()
    ys = []
    for t in range(L):
        a = np.exp((-dt[t] if slip == "sign" else dt[t]) * A)
        prev = h.copy()
        h = a * h + dt[t] * np.outer(x[t], B[t])
        use = prev if slip == "y_before_update" else h
        y = use @ C[t] + (0.0 if slip == "drop_D" else D) * x[t]
        ys.append(y)
    return np.array(ys), h


@pytest.mark.parametrize("slip", ["sign", "y_before_update", "drop_D"])
def test_planted_slip_is_caught_by_hand_example(slip):
    g = _golden("hand_worked_3tok.txt")
    args = (g["x"].reshape(3, 2), g["dt"], g["A"][0], g["B"].reshape(3, 2),
            g["C"].reshape(3, 2), g["D"][0], g["h_init"].reshape(2, 2))
    y_ok, _ = _python_recurrence(*args)
    np.testing.assert_allclose(y_ok.reshape(-1), g["y"], atol=1e-12)
    y_bad, _ = _python_recurrence(*args, slip=slip)
    assert np.max(np.abs(y_bad.reshape(-1) - g["y"])) > 1e-3


# --------------------------------------------------------------------------
# the head slice and the no-softplus-with-bias activation
# --------------------------------------------------------------------------
def test_head_slice_equals_those_heads_of_a_full_run():
    """``heads=(h0, h1)`` (used by every sampled full-size parity test) computes
    exactly those heads of the full run and leaves the other heads' outputs at
    zero; the full run itself is pinned by the dual form above."""
    p = W.make_problem([9, 0, 23, 5], nheads=8, headdim=3, dstate=5, ngroups=4, io_dtype="f32",
                       num_slots=6, has_init=[1, 0, 0, 1], seed=27)
    full = oracle.ssd_scan_reference(p)
    for h0, h1 in ((0, 8), (2, 5), (7, 8), (3, 3)):
        part = oracle.ssd_scan_reference(p, heads=(h0, h1))
        np.testing.assert_array_equal(part["y"][:, h0:h1], full["y"][:, h0:h1])
        np.testing.assert_array_equal(part["final"][:, h0:h1], full["final"][:, h0:h1])
        others = [h for h in range(8) if not h0 <= h < h1]
        assert not np.any(part["y"][:, others])
        for s in range(p.num_seqs):
            slot = int(p.slot_idx[s])
            np.testing.assert_array_equal(part["cache"][slot, h0:h1], full["cache"][slot, h0:h1])
            np.testing.assert_array_equal(part["cache"][slot, others], p.cache[slot, others])


def test_bias_without_softplus_matches_dual_form():
    """dt_softplus = 0 with a bias: dt' = dt + dt_bias, checked against the
    independent dual form with its softplus switched off."""
    rng = np.random.default_rng(28)
    L, H, P, N = 26, 3, 4, 5
    x, B, C = _rand(rng, L, H, P), _rand(rng, L, 1, N), _rand(rng, L, 1, N)
    dt = rng.uniform(0.01, 0.2, (L, H))
    bias = rng.uniform(0.0, 0.05, H)
    A, D = -rng.uniform(1, 8, H), _rand(rng, H)
    h0 = _rand(rng, 1, H, P, N)
    y, hf, _ = oracle.scan(x, dt, A, B, C, [0, L], dt_bias=bias, dt_softplus=False, D=D, h_init=h0)
    for h in range(H):
        yd, hd = dual_form_head(x[:, h], dt[:, h], A[h], B[:, 0], C[:, 0], D=D[h], h0=h0[0, h],
                                dt_bias=bias[h], softplus=False)
        np.testing.assert_allclose(y[:, h], yd, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(hf[0, h], hd, rtol=1e-11, atol=1e-12)

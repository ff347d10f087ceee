"""Pins of the CPU oracle against what the pages and mathematics fix, not against
itself: hand-derived worked examples, brute-force top-k, the exact
error-feedback identity, the lag, reduction to dense AdamS (float64) at
sparsity 0, the closed-form first step, off-mask invariance and the exact sum
of quantised gradients.  CPU only."""
import json
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")
HP = O.Hyper(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _f32(x):
    return np.asarray(x, np.float32)


# --------------------------------------------------------------------------- layout
@pytest.mark.parametrize("P,W,s", [(4096, 4, 0.9), (354871296, 8, 0.9), (569570560, 32, 0.99),
                                   (1364297728, 8, 0.99), (1 << 20, 32, 0.999), (10, 4, 0.5),
                                   (3, 8, 0.9), (1000, 7, 0.0)])
def test_layout_even_partition_and_k(P, W, s):
    start, k = O.layout(P, W, s)
    n = np.diff(start)
    assert start[0] == 0 and start[-1] == P
    assert (n >= 0).all() and n.max() - n.min() <= 1          # "evenly partitioned"
    keep = 1 - Fraction(str(s))
    for ns, ks in zip(n.tolist(), k.tolist()):
        exact = Fraction(ns) * keep
        assert ks == -((-exact.numerator) // exact.denominator)   # ceil, exact rational
        if ns:
            assert 1 <= ks <= ns


def test_layout_known_geometry():
    # shard sizes and k of the workloads, derived by hand from floor(sP/W) and ceil(n(1-s))
    start, k = O.layout(569570560, 32, 0.99)
    assert set(np.diff(start).tolist()) == {17799080}
    assert set(k.tolist()) == {177991} and k.sum() == 5695712
    start, k = O.layout(4096, 4, 0.9)
    assert k.tolist() == [103] * 4


# --------------------------------------------------------------------------- top-k
def _brute_topk(m, start, k):
    """Independent brute force: float magnitude (not bit patterns), Python sort."""
    P = len(m)
    sel = np.zeros(P, bool)
    for s in range(len(k)):
        lo, hi = int(start[s]), int(start[s + 1])
        order = sorted(range(lo, hi), key=lambda i: (-abs(float(m[i])), i))
        sel[order[:int(k[s])]] = True
    return sel


def _bits_to_bool(bits, P):
    return ((bits[np.arange(P) // 32] >> (np.arange(P) % 32).astype(np.uint32)) & 1).astype(bool)


def test_golden_partitioned_topk():
    g = _golden()["partitioned_topk"]
    start, k = O.layout(g["P"], g["W"], g["sparsity"])
    bits, idx = O.topk_mask(_f32(g["m"]), start, k)
    assert bits.tolist() == g["bits"]
    assert idx.tolist() == g["idx"]


def _cases(rng):
    yield rng.standard_normal(257).astype(np.float32)                       # ragged
    yield np.full(100, 0.5, np.float32)                                     # all ties
    yield (rng.integers(-128, 128, 1000) * 2.0 ** -15).astype(np.float32)   # 256 levels
    yield np.array([0.0, -0.0] * 50, np.float32)                            # signed zeros
    yield (rng.standard_normal(300) * 1e-42).astype(np.float32)             # denormals
    yield rng.standard_normal(64).astype(np.float32) * np.float32(1e30)


@pytest.mark.parametrize("W,s", [(1, 0.9), (3, 0.5), (4, 0.9), (7, 0.99), (8, 0.0)])
def test_topk_matches_brute_force(W, s):
    rng = np.random.default_rng(1)
    for m in _cases(rng):
        start, k = O.layout(m.size, W, s)
        bits, idx = O.topk_mask(m, start, k)
        want = _brute_topk(m, start, k)
        assert (_bits_to_bool(bits, m.size) == want).all()
        assert idx.tolist() == np.flatnonzero(want).tolist()
        # padding bits of the last word stay clear
        assert int(bits.view(np.uint32).sum()) >= 0
        if m.size % 32:
            assert bits[-1] >> np.uint32(m.size % 32) == 0
        for sh in range(W):
            lo, hi = start[sh], start[sh + 1]
            assert want[lo:hi].sum() == k[sh]


# --------------------------------------------------------------------------- step
def _bf16_bits(x):
    """Round-to-nearest-even float32 -> bfloat16 bit patterns (test-side helper)."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def _widen(g):
    if g.dtype == np.uint16:
        return (g.astype(np.uint32) << 16).view(np.float32)
    return g


def _grads(rng, P, W, steps, bf16=False, quant=False):
    out = []
    shared = rng.standard_normal(P)
    for _ in range(steps):
        shared = 0.9 * shared + np.sqrt(1 - 0.81) * rng.standard_normal(P)
        gs = []
        for _ in range(W):
            x = 1e-3 * (shared + rng.standard_normal(P))
            if quant:
                x = np.clip(np.round(x / 2.0 ** -15), -128, 127) * 2.0 ** -15
            x = x.astype(np.float32)
            gs.append(_bf16_bits(x) if bf16 else x)
        out.append(gs)
    return out


def test_golden_first_step_closed_form():
    g = _golden()["first_step_closed_form"]
    st = O.new_state(_f32(g["w0"]), g["W"], 0.0, HP)
    O.advance(st, [_f32(x) for x in g["grads"]])
    np.testing.assert_allclose(st.m, g["m1"], rtol=g["rtol"])
    np.testing.assert_allclose(st.w, g["w1"], rtol=g["rtol"])
    for e in st.e:
        assert (e == 0).all()


def test_golden_lagged_mask():
    g = _golden()["lagged_mask"]
    st = O.new_state(_f32(g["w0"]), g["W"], g["sparsity"], HP)
    O.advance(st, [_f32(g["grads"][0])])
    rec = O.advance(st, [_f32(g["grads"][1])])
    assert rec["pack"][0].tolist() == g["pack_step2"]
    np.testing.assert_array_equal(st.e[0], _f32(g["e_after_step2"]))
    np.testing.assert_allclose(st.m, g["m_after_step2"], rtol=g["rtol"])
    assert rec["idx"].tolist() == g["idx_after_step2"]


def test_closed_form_first_step_random():
    rng = np.random.default_rng(2)
    P, W = 777, 5
    w0 = (rng.standard_normal(P) * 0.02).astype(np.float32)
    grads = _grads(rng, P, W, 1)[0]
    st = O.new_state(w0, W, 0.9, HP)
    O.advance(st, grads)
    gbar = np.mean([g.astype(np.float64) for g in grads], axis=0)
    w1 = w0 - HP.lr * (gbar / (np.abs(gbar) + HP.eps) + HP.weight_decay * w0.astype(np.float64))
    np.testing.assert_allclose(st.m, (1 - HP.beta1) * gbar, rtol=1e-5, atol=1e-12)
    np.testing.assert_allclose(st.w, w1, rtol=1e-6, atol=1e-9)


def _dense_adams_f64(w0, grad_steps, hp):
    """Dense AdamS on the mean gradient, float64, straight from Eq. 2 of the
    SCAPE paper (Sec. II-C) with its bias corrections."""
    w = w0.astype(np.float64)
    m = np.zeros_like(w)
    b1, b2 = np.float64(np.float32(hp.beta1)), np.float64(np.float32(hp.beta2))
    lr, eps, wd = (np.float64(np.float32(x)) for x in (hp.lr, hp.eps, hp.weight_decay))
    for t, gs in enumerate(grad_steps, start=1):
        g = np.mean([_widen(x).astype(np.float64) for x in gs], axis=0)
        v = b2 * m * m + (1 - b2) * g * g
        m = b1 * m + (1 - b1) * g
        mh, vh = m / (1 - b1 ** t), v / (1 - b2 ** t)
        w = w - lr * (mh / (np.sqrt(vh) + eps) + wd * w)
    return w, m


@pytest.mark.parametrize("W,bf16", [(1, False), (4, False), (8, True), (3, True)])
def test_sparsity_zero_is_dense_adams(W, bf16):
    rng = np.random.default_rng(3)
    P, T = 1000, 10
    w0 = (rng.standard_normal(P) * 0.02).astype(np.float32)
    steps = _grads(rng, P, W, T, bf16=bf16)
    st = O.new_state(w0, W, 0.0, HP)
    for gs in steps:
        rec = O.advance(st, gs)
        assert rec["used_idx"].size == P
        for e in st.e:
            assert (e == 0).all()
    w_ref, m_ref = _dense_adams_f64(w0, steps, HP)
    np.testing.assert_allclose(st.m, m_ref, rtol=1e-5, atol=1e-10)
    np.testing.assert_allclose(st.w, w_ref, rtol=1e-5, atol=1e-7)


@pytest.mark.parametrize("W,s,bf16", [(1, 0.9, False), (4, 0.9, False), (8, 0.99, True)])
def test_error_feedback_conservation_compaction_lag_offmask(W, s, bf16):
    rng = np.random.default_rng(4)
    P, T = 3000, 6
    w0 = (rng.standard_normal(P) * 0.02).astype(np.float32)
    st = O.new_state(w0, W, s, HP)
    prev_bits = None
    for gs in _grads(rng, P, W, T, bf16=bf16):
        e_before = [x.copy() for x in st.e]
        w_before, m_before = st.w.copy(), st.m.copy()
        m_prev_mask = None if prev_bits is None else O.topk_mask(m_before, st.shard_start, st.shard_k)
        rec = O.advance(st, gs)
        used = _bits_to_bool(rec["used_bits"], P)
        # lag: the mask used now is the one built from m after the previous step
        if prev_bits is not None:
            assert (rec["used_bits"] == prev_bits).all()
            assert (rec["used_bits"] == m_prev_mask[0]).all()
        idx = rec["used_idx"]
        assert idx.tolist() == np.flatnonzero(used).tolist()
        for w in range(W):
            a = (_widen(gs[w]) + e_before[w]).astype(np.float32)          # fl(g + e)
            # compaction: the packed buffer is a at the set positions, ascending
            assert (rec["pack"][w].view(np.uint32) == a[idx].view(np.uint32)).all()
            # conservation: sent + residual == g + e, bit for bit
            sent = np.zeros(P, np.float32)
            sent[idx] = rec["pack"][w]
            assert ((sent + st.e[w]).view(np.uint32) == (a + np.float32(0)).view(np.uint32)).all()
            assert (st.e[w][used] == 0).all()
        # off-mask coordinates keep w and m bit for bit
        assert (st.w[~used].view(np.uint32) == w_before[~used].view(np.uint32)).all()
        assert (st.m[~used].view(np.uint32) == m_before[~used].view(np.uint32)).all()
        prev_bits = rec["bits"]


@pytest.mark.parametrize("W", [1, 2, 8, 32])
def test_sum_exact_on_quantised_gradients(W):
    rng = np.random.default_rng(5)
    P, T = 512, 4
    st = O.new_state(np.zeros(P, np.float32), W, 0.9, HP)
    for gs in _grads(rng, P, W, T, quant=True):
        rec = O.advance(st, gs)
        for j in range(rec["gbar"].size):
            exact = sum(Fraction(float(rec["pack"][w][j])) for w in range(W)) / W
            assert Fraction(float(rec["gbar"][j])) == exact


def test_always_and_never_selected_coordinates():
    """A coordinate whose gradient dominates its shard is always selected and so
    follows dense AdamS on its own mean gradient; a coordinate with zero first
    moment that is never selected keeps w and m and accumulates its gradient sum
    in the residual exactly (quantised gradients)."""
    rng = np.random.default_rng(6)
    P, W, T = 256, 2, 8
    steps = _grads(rng, P, W, T, quant=True)
    big = 5
    for gs in steps:
        for w in range(W):
            gs[w][big] = np.float32(0.5 + 0.01 * w)
    w0 = (rng.standard_normal(P) * 0.02).astype(np.float32)
    st = O.new_state(w0, W, 0.99, HP)
    for gs in steps:
        O.advance(st, gs)
    w_ref, m_ref = _dense_adams_f64(w0[big:big + 1], [[g[big:big + 1] for g in gs] for gs in steps], HP)
    np.testing.assert_allclose(st.w[big], w_ref[0], rtol=1e-6)
    np.testing.assert_allclose(st.m[big], m_ref[0], rtol=1e-5)
    # coordinates never selected after step 1 carry the exact sum of their gradients
    sel_any = np.zeros(P, bool)
    st2 = O.new_state(w0, W, 0.99, HP)
    recs = [O.advance(st2, gs) for gs in steps]
    for r in recs[1:]:
        sel_any |= _bits_to_bool(r["used_bits"], P)
    never = np.flatnonzero(~sel_any)
    assert never.size > 0
    for w in range(W):
        exact = [sum(Fraction(float(gs[w][i])) for gs in steps[1:]) for i in never[:20]]
        assert [Fraction(float(x)) for x in st2.e[w][never[:20]]] == exact


def test_bf16_widening_is_exact():
    x = np.array([1.0, -2.5, 3.0e-3, 65504.0], np.float32)
    b = _bf16_bits(x)
    assert (_widen(b) == np.array([struct.unpack("<f", struct.pack("<I", int(v) << 16))[0]
                                   for v in b], np.float32)).all()

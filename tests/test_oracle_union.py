"""Pins of the oracle's union-mask gradient top-k baseline (CPU only):
brute-force per-worker top-k and their union, exact error-feedback
conservation over the union, no fill-in when every worker sees the same
gradient, and reduction to dense AdamS (float64) at sparsity 0."""
import numpy as np
import pytest

from oracle import oracle as O
from tests.test_oracle_pins import HP, _bits_to_bool, _dense_adams_f64, _grads, _widen


def _brute_union(a_list, k):
    sel = np.zeros(a_list[0].size, bool)
    for a in a_list:
        order = sorted(range(a.size), key=lambda i: (-abs(float(a[i])), i))
        sel[order[:k]] = True
    return sel


@pytest.mark.parametrize("W,s,quant", [(1, 0.9, False), (4, 0.9, False), (3, 0.99, True),
                                       (8, 0.5, True)])
def test_union_mask_and_conservation(W, s, quant):
    rng = np.random.default_rng(11)
    P, T = 900, 3
    w = (rng.standard_normal(P) * 0.02).astype(np.float32)
    m = np.zeros(P, np.float32)
    e = [np.zeros(P, np.float32) for _ in range(W)]
    kw = O.union_k_worker(P, s)
    for t, gs in enumerate(_grads(rng, P, W, T, quant=quant), start=1):
        a = [(_widen(g) + x).astype(np.float32) for g, x in zip(gs, e)]
        bits, idx, pack, gbar = O.union_topk_step(t, gs, e, w, m, kw, HP)
        want = _brute_union(a, kw)
        assert (_bits_to_bool(bits, P) == want).all()
        assert idx.tolist() == np.flatnonzero(want).tolist()
        for wk in range(W):
            assert (pack[wk].view(np.uint32) == a[wk][idx].view(np.uint32)).all()
            sent = np.zeros(P, np.float32)
            sent[idx] = pack[wk]
            assert ((sent + e[wk]).view(np.uint32) == a[wk].view(np.uint32)).all()
        assert kw <= idx.size <= min(P, W * kw)


def test_identical_gradients_give_no_fill_in():
    rng = np.random.default_rng(12)
    P, W = 1000, 6
    g = (rng.standard_normal(P) * 1e-3).astype(np.float32)
    e = [np.zeros(P, np.float32) for _ in range(W)]
    w, m = np.zeros(P, np.float32), np.zeros(P, np.float32)
    kw = O.union_k_worker(P, 0.95)
    _, idx, _, _ = O.union_topk_step(1, [g.copy() for _ in range(W)], e, w, m, kw, HP)
    assert idx.size == kw


def test_sparsity_zero_is_dense_adams():
    rng = np.random.default_rng(13)
    P, W, T = 500, 4, 6
    w0 = (rng.standard_normal(P) * 0.02).astype(np.float32)
    steps = _grads(rng, P, W, T)
    w, m = w0.copy(), np.zeros(P, np.float32)
    e = [np.zeros(P, np.float32) for _ in range(W)]
    for t, gs in enumerate(steps, start=1):
        O.union_topk_step(t, gs, e, w, m, P, HP)
        assert all((x == 0).all() for x in e)
    w_ref, m_ref = _dense_adams_f64(w0, steps, HP)
    np.testing.assert_allclose(m, m_ref, rtol=1e-5, atol=1e-10)
    np.testing.assert_allclose(w, w_ref, rtol=1e-5, atol=1e-7)

"""Randomised properties of the oracle's layout and per-shard top-k (CPU
only), checked against an independent brute force and against what the
sharding and the keep-fraction require -- not against the oracle's own
formulas.  Skipped where hypothesis is not installed."""
from fractions import Fraction

import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

from oracle import oracle as O  # noqa: E402
from tests.test_oracle_pins import _bits_to_bool, _brute_topk  # noqa: E402

_values = st.sampled_from([0.0, -0.0, 0.25, -0.25, 1e-40, -1e-40, 3.0, -3.0, 1e30,
                           float("inf"), -float("inf"), 0.5, -0.5])


@st.composite
def _problem(draw):
    P = draw(st.integers(1, 400))
    W = draw(st.integers(1, 12))
    s = draw(st.sampled_from([0.0, 0.5, 0.9, 0.99, 0.999, 0.123456, 0.7]))
    mode = draw(st.sampled_from(["gauss", "levels", "mixed"]))
    seed = draw(st.integers(0, 2**31 - 1))
    rng = np.random.default_rng(seed)
    if mode == "gauss":
        m = rng.standard_normal(P).astype(np.float32)
    elif mode == "levels":
        m = (rng.integers(-4, 5, P) * 0.125).astype(np.float32)
    else:
        m = np.array(draw(st.lists(_values, min_size=P, max_size=P)), np.float32)
    return m, W, s


@settings(max_examples=150, deadline=None)
@given(_problem())
def test_layout_partitions_and_keeps_the_fraction(prob):
    m, W, s = prob
    P = m.size
    start, k = O.layout(P, W, s)
    assert start[0] == 0 and start[-1] == P
    sizes = np.diff(start)
    assert (sizes >= 0).all() and sizes.max() - sizes.min() <= 1     # even split
    # the keep fraction 1 - s, with s taken to parts per million
    keep = Fraction(1_000_000 - round(s * 1_000_000), 1_000_000)
    for n, kk in zip(sizes.tolist(), k.tolist()):
        if n == 0:
            assert kk == 0
            continue
        # the smallest count that keeps at least that fraction of the shard
        assert kk >= n * keep
        assert kk - 1 < n * keep
        assert 1 <= kk <= n


@settings(max_examples=150, deadline=None)
@given(_problem())
def test_topk_matches_brute_force_on_random_shapes(prob):
    m, W, s = prob
    start, k = O.layout(m.size, W, s)
    bits, idx = O.topk_mask(m, start, k)
    want = _brute_topk(m, start, k)
    assert (_bits_to_bool(bits, m.size) == want).all()
    assert idx.tolist() == np.flatnonzero(want).tolist()
    if m.size % 32:
        assert bits[-1] >> np.uint32(m.size % 32) == 0


@st.composite
def _trajectory(draw):
    P = draw(st.integers(1, 300))
    W = draw(st.integers(1, 6))
    s = draw(st.sampled_from([0.0, 0.5, 0.9, 0.99]))
    bf16 = draw(st.booleans())
    quant = draw(st.booleans())
    seed = draw(st.integers(0, 2**31 - 1))
    return P, W, s, bf16, quant, seed


@settings(max_examples=60, deadline=None)
@given(_trajectory())
def test_step_invariants_on_random_trajectories(case):
    """Error-feedback conservation bit for bit, compaction order, the one-step
    lag and off-mask invariance, on random shapes and data."""
    from tests.test_oracle_pins import HP, _grads, _widen
    P, W, s, bf16, quant, seed = case
    rng = np.random.default_rng(seed)
    w0 = (rng.standard_normal(P) * 0.02).astype(np.float32)
    st_ = O.new_state(w0, W, s, HP)
    prev_bits = None
    for gs in _grads(rng, P, W, 4, bf16=bf16, quant=quant):
        e_before = [x.copy() for x in st_.e]
        w_before, m_before = st_.w.copy(), st_.m.copy()
        rec = O.advance(st_, gs)
        used = _bits_to_bool(rec["used_bits"], P)
        if prev_bits is not None:
            assert (rec["used_bits"] == prev_bits).all()
        idx = rec["used_idx"]
        assert idx.tolist() == np.flatnonzero(used).tolist()
        for w in range(W):
            a = (_widen(gs[w]) + e_before[w]).astype(np.float32)
            assert (rec["pack"][w].view(np.uint32) == a[idx].view(np.uint32)).all()
            sent = np.zeros(P, np.float32)
            sent[idx] = rec["pack"][w]
            assert ((sent + st_.e[w]).view(np.uint32) == (a + np.float32(0)).view(np.uint32)).all()
        assert (st_.w[~used].view(np.uint32) == w_before[~used].view(np.uint32)).all()
        assert (st_.m[~used].view(np.uint32) == m_before[~used].view(np.uint32)).all()
        prev_bits = rec["bits"]

"""Pins of the oracle's variant readings and dense baselines (CPU only).

* DENSE_OFFMASK (unselected coordinates also take AdamS with a zero
  gradient): at sparsity 0 it is dense AdamS (float64, Eq. 2 of the SCAPE
  paper); a coordinate never selected after step 1 follows the float64 AdamS
  recursion with g = 0.
* MOMENT_SYNC (the synchronised buffer holds first moments): at sparsity 0 it
  is dense AdamS; with one worker the synchronised buffer is exactly that
  worker's first moment and the recovered gradient its error-fed gradient.
* Dense AdamS baseline: float64 dense AdamS on the plain mean gradient.
* AdamW baseline: torch.optim.AdamW in float64 (a library routine).
"""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from tests.test_oracle_pins import HP, _bits_to_bool, _dense_adams_f64, _grads, _widen


def _run(variant, P, W, s, T, seed, bf16=False):
    rng = np.random.default_rng(seed)
    w0 = (rng.standard_normal(P) * 0.02).astype(np.float32)
    steps = _grads(rng, P, W, T, bf16=bf16)
    st = O.new_state(w0, W, s, HP)
    recs = [O.advance(st, gs, variant=variant) for gs in steps]
    return w0, steps, st, recs


def test_variant_zero_is_the_paper_reading():
    a = _run(0, 1500, 3, 0.9, 5, seed=1)[2]
    rng = np.random.default_rng(1)
    w0 = (rng.standard_normal(1500) * 0.02).astype(np.float32)
    steps = _grads(rng, 1500, 3, 5)
    st = O.new_state(w0, 3, 0.9, HP)
    for gs in steps:
        pack, gbar = O.step_variant(st.t + 1, gs, st.e, st.w, st.m,
                                    *(O.dense_mask(1500) if st.bits is None else (st.bits, st.idx)),
                                    HP, 0)
        st.t += 1
        st.bits, st.idx = O.topk_mask(st.m, st.shard_start, st.shard_k)
    assert np.array_equal(a.w.view(np.uint32), st.w.view(np.uint32))


@pytest.mark.parametrize("variant", [O.DENSE_OFFMASK, O.MOMENT_SYNC, O.DENSE_OFFMASK | O.MOMENT_SYNC])
def test_variants_at_sparsity_zero_are_dense_adams(variant):
    w0, steps, st, _ = _run(variant, 800, 4, 0.0, 8, seed=2)
    w_ref, m_ref = _dense_adams_f64(w0, steps, HP)
    np.testing.assert_allclose(st.m, m_ref, rtol=1e-5, atol=1e-10)
    np.testing.assert_allclose(st.w, w_ref, rtol=1e-5, atol=1e-7)


def test_dense_offmask_unselected_follow_zero_gradient_adams():
    P, W, T = 2000, 2, 6
    w0, steps, st, recs = _run(O.DENSE_OFFMASK, P, W, 0.99, T, seed=3)
    never = np.ones(P, bool)
    for r in recs[1:]:
        never &= ~_bits_to_bool(r["used_bits"], P)
    cand = np.flatnonzero(never)[:50]
    assert cand.size > 0
    for i in cand:
        # step 1 on the mean gradient, then steps 2..T with g = 0
        g_steps = [[x[i:i + 1] for x in steps[0]]] + \
                  [[np.zeros(1, np.float32)] * W for _ in range(T - 1)]
        w_ref, m_ref = _dense_adams_f64(w0[i:i + 1], g_steps, HP)
        np.testing.assert_allclose(st.w[i], w_ref[0], rtol=1e-6, atol=1e-9)
        np.testing.assert_allclose(st.m[i], m_ref[0], rtol=1e-5, atol=1e-12)


def test_dense_offmask_leaves_the_paper_reading_on_selected_coordinates():
    P, W, T = 3000, 4, 4
    _, _, a, ra = _run(O.DENSE_OFFMASK, P, W, 0.9, T, seed=4)
    _, _, b, rb = _run(0, P, W, 0.9, T, seed=4)
    # the masks differ once m differs off the mask, but step 2 shares step 1's mask
    assert np.array_equal(ra[1]["used_bits"], rb[1]["used_bits"])
    assert np.array_equal(ra[1]["pack"].view(np.uint32), rb[1]["pack"].view(np.uint32))


def test_moment_sync_single_worker_buffer_is_its_first_moment():
    P, T = 1000, 4
    w0, steps, st, recs = _run(O.MOMENT_SYNC, P, 1, 0.9, T, seed=5)
    # replay: with W = 1 the synchronised buffer of step t at the selected
    # coordinates equals b1 * m_{t-1} + (1 - b1) * (g + e) in float64
    rng = np.random.default_rng(5)
    st2 = O.new_state(w0, 1, 0.9, HP)
    for t, gs in enumerate(steps, start=1):
        e_prev = st2.e[0].astype(np.float64).copy()
        m_prev = st2.m.astype(np.float64).copy()
        rec = O.advance(st2, gs, variant=O.MOMENT_SYNC)
        idx = rec["used_idx"].astype(np.int64)
        a = _widen(gs[0]).astype(np.float64)[idx] + e_prev[idx]
        b1 = np.float64(np.float32(HP.beta1))
        want = b1 * m_prev[idx] + (1 - b1) * a
        np.testing.assert_allclose(rec["gbar"], want, rtol=1e-6, atol=1e-12)
        np.testing.assert_allclose(st2.m[idx], want, rtol=1e-6, atol=1e-12)


@pytest.mark.parametrize("W,bf16", [(1, False), (4, True)])
def test_dense_adams_baseline(W, bf16):
    rng = np.random.default_rng(6)
    P, T = 700, 7
    w0 = (rng.standard_normal(P) * 0.02).astype(np.float32)
    steps = _grads(rng, P, W, T, bf16=bf16)
    w, m = w0.copy(), np.zeros(P, np.float32)
    for t, gs in enumerate(steps, start=1):
        O.dense_adams_step(t, gs, w, m, HP)
    w_ref, m_ref = _dense_adams_f64(w0, steps, HP)
    np.testing.assert_allclose(m, m_ref, rtol=1e-5, atol=1e-10)
    np.testing.assert_allclose(w, w_ref, rtol=1e-5, atol=1e-7)


@pytest.mark.parametrize("W,bf16", [(1, False), (3, True)])
def test_adamw_baseline_matches_torch_adamw(W, bf16):
    rng = np.random.default_rng(7)
    P, T = 600, 9
    w0 = (rng.standard_normal(P) * 0.02).astype(np.float32)
    steps = _grads(rng, P, W, T, bf16=bf16)
    w, m, v = w0.copy(), np.zeros(P, np.float32), np.zeros(P, np.float32)
    for t, gs in enumerate(steps, start=1):
        O.adamw_step(t, gs, w, m, v, HP)
    f = lambda x: float(np.float32(x))
    p = torch.nn.Parameter(torch.from_numpy(w0.astype(np.float64)))
    opt = torch.optim.AdamW([p], lr=f(HP.lr), betas=(f(HP.beta1), f(HP.beta2)), eps=f(HP.eps),
                            weight_decay=f(HP.weight_decay))
    for gs in steps:
        p.grad = torch.from_numpy(np.mean([_widen(x).astype(np.float64) for x in gs], axis=0))
        opt.step()
    np.testing.assert_allclose(w, p.detach().numpy(), rtol=1e-5, atol=1e-7)
    np.testing.assert_allclose(m, opt.state[p]["exp_avg"].numpy(), rtol=1e-5, atol=1e-10)
    np.testing.assert_allclose(v, opt.state[p]["exp_avg_sq"].numpy(), rtol=1e-5, atol=1e-14)

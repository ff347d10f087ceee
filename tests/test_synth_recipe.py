"""The synthetic inputs follow the stated recipe (CPU only): parameter counts of
the three model shapes, the gradient model's variances, AR(1) step-to-step
correlation, heavy tails of the Student-t noise, per-layer log-uniform scales,
256-level quantisation, and determinism per seed."""
import math

import numpy as np
import torch

from sparse_communication_sharded_gb300 import synth


def test_parameter_counts_of_the_model_shapes():
    # per-layer arithmetic of the three architectures, counted by hand
    h, f, v = 1024, 4096, 50304
    gpt_layer = (2 * h) + (3 * h * h + 3 * h) + (h * h + h) + (2 * h) + (h * f + f) + (f * h + h)
    assert synth.WORKLOADS["gpt345m"].P == v * h + 1024 * h + 24 * gpt_layer + 2 * h == 354871296
    for name, (h, f, P) in {"llama500m": (1280, 3584, 569570560),
                            "llama1p8b": (2048, 5632, 1364297728)}.items():
        layer = 4 * h * h + 3 * h * f + 2 * h
        assert synth.WORKLOADS[name].P == 2 * 32000 * h + 24 * layer + h == P


def _stream(noise="gauss", rho=0.9, P=200_000, W=4, layer_scale=None, quantum=None, seed=3):
    wl = synth.Workload("t", (("a", P // 2), ("b", P - P // 2)), W=W, sparsity=0.9, steps=4,
                        grad_dtype="f32", rho=rho, noise=noise, layer_scale=layer_scale,
                        quantum=quantum)
    return wl, synth.GradientStream(wl, seed=seed, device="cpu")


def test_gaussian_model_variances_and_ar1_correlation():
    wl, gen = _stream()
    g1 = torch.stack(gen.next()).double()
    g2 = torch.stack(gen.next()).double()
    c = wl.sigma
    # g = c (s + n): unit-variance shared signal and noise
    assert abs(g1.std().item() / (c * math.sqrt(2)) - 1) < 0.01
    # two workers share only the signal: covariance c^2
    cov = ((g1[0] * g1[1]).mean() - g1[0].mean() * g1[1].mean()).item()
    assert abs(cov / c ** 2 - 1) < 0.03
    # step to step, the same worker: covariance rho c^2 through the signal
    cov_t = ((g1[0] * g2[0]).mean()).item()
    assert abs(cov_t / (wl.rho * c ** 2) - 1) < 0.05


def test_student_t_noise_has_heavy_tails():
    _, gen = _stream(noise="student_t3", rho=0.95)
    g = torch.stack(gen.next()).double()
    n = (g[0] - g[1]).flatten()          # the shared signal cancels
    kurt = ((n - n.mean()) ** 4).mean() / n.var() ** 2
    assert kurt > 6.0                    # Gaussian differences would give 3


def test_per_layer_log_uniform_scale():
    wl, gen = _stream(layer_scale=(1e-4, 1e-2))
    sc = gen.scale
    P = wl.P
    a = sc[:P // 2]
    b = sc[P // 2:]
    assert bool((a == a[0]).all()) and bool((b == b[0]).all())   # one scale per layer
    for x in (a[0].item(), b[0].item()):
        assert 1e-4 <= x <= 1e-2


def test_quantised_gradients_have_256_levels():
    _, gen = _stream(quantum=2.0 ** -15)
    g = torch.stack(gen.next())
    q = g / 2.0 ** -15
    assert bool((q == q.round()).all())
    assert q.min().item() >= -128 and q.max().item() <= 127
    assert len(torch.unique(g)) <= 256


def test_same_seed_same_bytes():
    _, a = _stream(seed=11)
    _, b = _stream(seed=11)
    _, c = _stream(seed=12)
    ga, gb, gc = a.next(), b.next(), c.next()
    assert all(torch.equal(x, y) for x, y in zip(ga, gb))
    assert not torch.equal(ga[0], gc[0])
    assert torch.equal(synth.init_params(1000, seed=5), synth.init_params(1000, seed=5))
    w = synth.init_params(400_000, seed=5).double()
    assert abs(w.std().item() / 0.02 - 1) < 0.01

"""GPU parity of the variant readings and the dense baselines against the CPU
oracle (same seeded inputs, element by element).  Masks, packed buffers and
the synchronised buffer must match exactly; float states within 1e-5 relative
/ 1e-7 absolute, and in practice bit-identical (asserted too)."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from sparse_communication_sharded_gb300 import _scape as C
from sparse_communication_sharded_gb300 import synth
from tests._harness import HP, assert_close_f32, make_opt, run_full_trajectory, u32

pytestmark = pytest.mark.gpu

VARIANTS = [C.SCAPE_VARIANT_DENSE_OFFMASK, C.SCAPE_VARIANT_MOMENT_SYNC,
            C.SCAPE_VARIANT_DENSE_OFFMASK | C.SCAPE_VARIANT_MOMENT_SYNC]


def _wl(P, W, s, dtype):
    return synth.Workload(f"p{P}", (("flat", P),), W=W, sparsity=s, steps=8, grad_dtype=dtype)


def test_variant_flags_match_the_oracle():
    assert (C.SCAPE_VARIANT_DENSE_OFFMASK, C.SCAPE_VARIANT_MOMENT_SYNC) == \
           (O.DENSE_OFFMASK, O.MOMENT_SYNC)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("P,W,s,dtype", [(4096, 4, 0.9, "f32"), (70001, 8, 0.99, "bf16"),
                                         (20000, 3, 0.0, "f32")])
def test_variant_trajectory_matches_oracle(cuda_device, variant, P, W, s, dtype):
    rep = run_full_trajectory(_wl(P, W, s, dtype), cuda_device, steps=8, variant=variant)
    assert rep.exact


@pytest.mark.parametrize("fusion", [0, 1])
@pytest.mark.parametrize("variant", VARIANTS)
def test_variant_trajectory_other_fusion_levels(cuda_device, variant, fusion):
    rep = run_full_trajectory(_wl(70001, 8, 0.99, "bf16"), cuda_device, steps=6, variant=variant,
                              fusion=fusion)
    assert rep.exact


def test_unknown_variant_flag_is_rejected(cuda_device):
    opt = make_opt(torch.zeros(64, device=cuda_device), 2, 0.5, torch.float32)
    with pytest.raises(C.ScapeError):
        opt.set_variant(4)
    opt.close()


@pytest.mark.parametrize("adamw", [False, True])
@pytest.mark.parametrize("P,W,dtype", [(50003, 4, "bf16"), (4096, 1, "f32"), (2048 * 5, 8, "f32")])
def test_dense_baselines_match_oracle(cuda_device, adamw, P, W, dtype):
    gdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    gen = synth.GradientStream(_wl(P, W, 0.9, dtype), seed=4, device="cpu")
    w0 = synth.init_params(P, seed=4)
    params = w0.to(cuda_device)
    opt = make_opt(params, W, 0.9, gdt)
    v = torch.zeros(P, device=cuda_device)
    w, m, vh = w0.numpy().copy(), np.zeros(P, np.float32), np.zeros(P, np.float32)
    for t in range(1, 7):
        grads = gen.next()
        dg = [g.to(cuda_device) for g in grads]
        hg = [synth.to_numpy_grad(g) for g in grads]
        if adamw:
            opt.adamw_step(dg, v)
            O.adamw_step(t, hg, w, m, vh, HP)
        else:
            opt.dense_adams_step(dg)
            O.dense_adams_step(t, hg, w, m, HP)
    torch.cuda.synchronize()
    assert_close_f32(params.cpu().numpy(), w, "w")
    assert_close_f32(opt.m.cpu().numpy(), m, "m")
    assert np.array_equal(u32(params), w.view(np.uint32))
    assert np.array_equal(u32(opt.m), m.view(np.uint32))
    if adamw:
        assert np.array_equal(u32(v), vh.view(np.uint32))
    for e in opt.e:                                  # residuals untouched
        assert not e.any()
    opt.close()


# ------------------------------------------------------------ union-mask baseline
@pytest.mark.parametrize("P,W,s,dtype,quant", [(4096, 4, 0.9, "f32", False),
                                               (70001, 8, 0.99, "bf16", False),
                                               (30000, 3, 0.9, "f32", True),
                                               (5000, 2, 0.0, "f32", False)])
def test_union_baseline_matches_oracle(cuda_device, P, W, s, dtype, quant):
    gdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    wl = synth.Workload(f"p{P}", (("flat", P),), W=W, sparsity=s, steps=5, grad_dtype=dtype,
                        quantum=2.0 ** -15 if quant else None)
    gen = synth.GradientStream(wl, seed=6, device="cpu")
    w0 = synth.init_params(P, seed=6)
    params = w0.to(cuda_device)
    opt = make_opt(params, W, s, gdt)
    w, m = w0.numpy().copy(), np.zeros(P, np.float32)
    e = [np.zeros(P, np.float32) for _ in range(W)]
    kw = O.union_k_worker(P, s)
    for t in range(1, 6):
        grads = gen.next()
        ku = opt.union_step([g.to(cuda_device) for g in grads])
        bits, idx, pack, gbar = O.union_topk_step(t, [synth.to_numpy_grad(g) for g in grads],
                                                  e, w, m, kw, HP)
        assert ku == idx.size
    torch.cuda.synchronize()
    assert_close_f32(params.cpu().numpy(), w, "w")
    assert np.array_equal(u32(params), w.view(np.uint32))
    assert np.array_equal(u32(opt.m), m.view(np.uint32))
    for wk in range(W):
        assert np.array_equal(u32(opt.e[wk]), e[wk].view(np.uint32))
    opt.close()


def test_union_capacity_overflow_is_reported(cuda_device):
    P, W = 8192, 8
    opt = make_opt(torch.zeros(P, device=cuda_device), W, 0.9, torch.float32)
    g = [torch.randn(P, device=cuda_device) for _ in range(W)]
    with pytest.raises(C.ScapeError):
        opt.union_step(g, capacity=O.union_k_worker(P, 0.9))   # independent noise fills in
    opt.close()

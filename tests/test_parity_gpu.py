"""GPU parity: the CUDA path through the C ABI against the CPU oracle, element by
element, on identical seeded inputs.

Bars: masks, packed indices and packed values bit-exact given identical
inputs; float states within 1e-5 relative / 1e-7 absolute after the
trajectory, with at most 1e-4 of the mask bits flipped at the threshold.  (The
kernels follow the oracle's operation order, so in practice every value is
bit-identical; `rep.exact` records that and is asserted too.)
"""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from sparse_communication_sharded_gb300 import Scape, ScapeError, synth
from sparse_communication_sharded_gb300 import _scape as C
from tests._harness import HP, bits_to_bool, make_opt, run_full_trajectory, run_sampled_shards, u32

pytestmark = pytest.mark.gpu


def _wl(P, W, s, dtype, steps=10, quant=False, noise="gauss"):
    return synth.Workload(f"p{P}", (("flat", P),), W=W, sparsity=s, steps=steps,
                          grad_dtype=dtype, noise=noise,
                          quantum=2.0 ** -15 if quant else None)


# ------------------------------------------------------------ whole-problem trajectories
TRAJ = [
    # (P, W, sparsity, grad dtype, quantised)
    (4096, 4, 0.90, "f32", False),      # the tiny workload
    (5003, 3, 0.90, "f32", False),      # ragged tail, non-power-of-two W
    (100003, 8, 0.99, "bf16", False),   # several tiles, ragged, bf16
    (65536, 1, 0.90, "bf16", False),    # single worker
    (20000, 8, 0.0, "f32", False),      # sparsity 0: dense AdamS every step
    (50000, 32, 0.999, "f32", True),    # 256-level gradients: massive ties
    (33333, 7, 0.99, "f32", True),      # ties + shard boundaries mid-word
    (5, 8, 0.5, "f32", False),          # P < W: empty shards
    (2048 * 3, 2, 0.75, "bf16", False),  # exact multiple of the tile
    (1 << 16, 256, 0.99, "bf16", False),  # the largest W the ABI accepts
    (3000, 256, 0.9, "f32", False),       # W = 256 with shards of 11-12 parameters
]


@pytest.mark.parametrize("P,W,s,dtype,quant", TRAJ)
def test_trajectory_matches_oracle(cuda_device, P, W, s, dtype, quant):
    rep = run_full_trajectory(_wl(P, W, s, dtype, quant=quant), cuda_device, steps=10)
    assert rep.exact, "trajectory not bit-identical to the oracle"


@pytest.mark.parametrize("fusion", [C.FUSE_NONE, C.FUSE_SUM, C.FUSE_UPDATE])
@pytest.mark.parametrize("P,W,s,dtype,quant", [TRAJ[1], TRAJ[2], TRAJ[4], TRAJ[5], TRAJ[6],
                                                TRAJ[7], TRAJ[9], TRAJ[10],
                                                (11, 8, 0.5, "f32", False),
                                                (300001, 3, 0.9, "bf16", False)])
def test_trajectory_every_fusion_level(cuda_device, fusion, P, W, s, dtype, quant):
    """Separate launches (ordered sum, then unpack + AdamS), the sum inside the
    compaction, and sum + update inside it all give the oracle's bits.
    (11, 8, 0.5) mixes shards that keep every coordinate with searched ones."""
    rep = run_full_trajectory(_wl(P, W, s, dtype, quant=quant), cuda_device, steps=6,
                              fusion=fusion)
    assert rep.exact


@pytest.mark.parametrize("P,W,s,dtype,quant", [TRAJ[2], TRAJ[5], TRAJ[6], TRAJ[9]])
def test_trajectory_refresh_graph_off(cuda_device, P, W, s, dtype, quant):
    """Every refresh enqueued launch by launch (the steady warm refresh is
    otherwise replayed from a captured graph): the same oracle bits."""
    rep = run_full_trajectory(_wl(P, W, s, dtype, quant=quant), cuda_device, steps=10,
                              graphs=False)
    assert rep.exact


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_unaligned_gradients_scalar_path(cuda_device, dtype):
    rep = run_full_trajectory(_wl(30001, 4, 0.9, dtype), cuda_device, steps=5, grad_offset_elems=1)
    assert rep.exact


def test_flat_sweep_small_points(cuda_device):
    """The flat sweep's 2^20 point at every W and sparsity (256-level gradients)."""
    for W in (1, 8, 32):
        for s in (0.0, 0.9, 0.99, 0.999):
            rep = run_full_trajectory(synth.flat_workload(1 << 20, W, s), cuda_device, steps=5)
            assert rep.exact, (W, s)


# ------------------------------------------------------------ mask refresh on identical m
def _refresh_on(cuda_device, m_host: np.ndarray, W: int, s: float):
    P = m_host.size
    params = torch.zeros(P, device=cuda_device)
    opt = make_opt(params, W, s, torch.float32)
    grads = [torch.zeros(P, device=cuda_device) for _ in range(W)]
    opt.step(grads)                       # t = 1 so a refresh is legal
    opt.m.copy_(torch.from_numpy(m_host))
    opt.refresh_mask()
    torch.cuda.synchronize()
    start, ks = O.layout(P, W, s)
    bits, idx = O.topk_mask(m_host, start, ks)
    got_bits, got_idx = u32(opt.bits()), u32(opt.idx())
    opt.close()
    return got_bits, got_idx, bits, idx


M_CASES = {
    "gauss": lambda r, n: (r.standard_normal(n) * 1e-3).astype(np.float32),
    "all_equal": lambda r, n: np.full(n, 0.25, np.float32),
    "levels": lambda r, n: (r.integers(-128, 128, n) * 2.0 ** -15).astype(np.float32),
    "signed_zero": lambda r, n: np.where(r.random(n) < 0.5, -0.0, 0.0).astype(np.float32),
    "denormal": lambda r, n: (r.standard_normal(n) * 1e-41).astype(np.float32),
    "huge": lambda r, n: (r.standard_normal(n) * 1e37).astype(np.float32),
    "few_levels": lambda r, n: r.choice(np.array([1.0, -1.0, 0.5, 0.0], np.float32), n),
}


@pytest.mark.parametrize("case", sorted(M_CASES))
@pytest.mark.parametrize("P,W,s", [(70001, 5, 0.9), (4096, 4, 0.99), (300000, 32, 0.999),
                                   (1000, 1, 0.5)])
def test_refresh_bit_exact_on_same_m(cuda_device, case, P, W, s):
    m = M_CASES[case](np.random.default_rng(P + W), P)
    got_bits, got_idx, bits, idx = _refresh_on(cuda_device, m, W, s)
    assert np.array_equal(got_bits, bits)
    assert np.array_equal(got_idx, idx.view(np.uint32))


# ------------------------------------------------------------ warm refresh (speculative bitmap)
def _drift(m, r, rel):
    return (m * (1.0 + rel * r.standard_normal(m.size))).astype(np.float32)


def _mixed(m, r, W):
    # every other shard's magnitudes jump by 8x (its threshold leaves the
    # bucket window); the rest drift slightly
    out = _drift(m, r, 0.01)
    start, _ = O.layout(m.size, W, 0.5)
    for s in range(0, W, 2):
        out[start[s]:start[s + 1]] *= 8.0
    return out


WARM_CASES = {
    "same": lambda m, r, W: m.copy(),
    "drift": lambda m, r, W: _drift(m, r, 0.02),
    "drift_large": lambda m, r, W: _drift(m, r, 0.3),
    "scaled_up": lambda m, r, W: (m * 4.0).astype(np.float32),
    "scaled_down": lambda m, r, W: (m * 0.25).astype(np.float32),
    "permuted": lambda m, r, W: r.permutation(m),
    "mixed": _mixed,
    "levels": lambda m, r, W: (r.integers(-128, 128, m.size) * 2.0 ** -15).astype(np.float32),
    "zeros": lambda m, r, W: np.zeros_like(m),
}


@pytest.mark.parametrize("case", sorted(WARM_CASES))
@pytest.mark.parametrize("P,W,s", [(70001, 5, 0.9), (300000, 32, 0.99), (1 << 16, 4, 0.999),
                                   (1500, 3, 0.5), (20000, 256, 0.9), (4096, 2, 0.0)])
def test_warm_refresh_bit_exact(cuda_device, case, P, W, s):
    """Refreshes after the first correct the previous refresh's bitmap; three in
    a row (m1 cold, then m2 and m3 warm) must each equal the oracle's mask."""
    r = np.random.default_rng(P + 7 * W)
    m1 = (r.standard_normal(P) * 1e-3).astype(np.float32)
    m2 = WARM_CASES[case](m1, r, W)
    m3 = _drift(m2, r, 0.05)
    params = torch.zeros(P, device=cuda_device)
    opt = make_opt(params, W, s, torch.float32)
    opt.step([torch.zeros(P, device=cuda_device) for _ in range(W)])
    start, ks = O.layout(P, W, s)
    for mh in (m1, m2, m3):
        opt.m.copy_(torch.from_numpy(mh))
        opt.refresh_mask()
        torch.cuda.synchronize()
        bits, idx = O.topk_mask(mh, start, ks)
        assert np.array_equal(u32(opt.bits()), bits)
        assert np.array_equal(u32(opt.idx()), idx.view(np.uint32))
    opt.close()


@pytest.mark.parametrize("rate", [1.12, 1.3, 0.85, 1.02])
@pytest.mark.parametrize("P,W,s", [(70001, 5, 0.9), (300000, 32, 0.99)])
def test_warm_refresh_trending_threshold(cuda_device, rate, P, W, s):
    """First moments growing (or shrinking) by a steady factor per refresh,
    as early in training: the staged window follows the thresholds' trend;
    every refresh must still equal the oracle's mask."""
    r = np.random.default_rng(P + W)
    base = (r.standard_normal(P) * 1e-3).astype(np.float32)
    params = torch.zeros(P, device=cuda_device)
    opt = make_opt(params, W, s, torch.float32)
    opt.step([torch.zeros(P, device=cuda_device) for _ in range(W)])
    start, ks = O.layout(P, W, s)
    for t in range(7):
        mh = _drift((base * rate ** t).astype(np.float32), r, 0.01)
        opt.m.copy_(torch.from_numpy(mh))
        opt.refresh_mask()
        torch.cuda.synchronize()
        bits, idx = O.topk_mask(mh, start, ks)
        assert np.array_equal(u32(opt.bits()), bits), t
        assert np.array_equal(u32(opt.idx()), idx.view(np.uint32)), t
    opt.close()


# ------------------------------------------------------------ lag, checkpoint, host path
def test_lag_step_uses_previous_refresh(cuda_device):
    P, W, s = 40000, 4, 0.9
    wl = _wl(P, W, s, "f32")
    gen = synth.GradientStream(wl, seed=3, device=cuda_device)
    params = synth.init_params(P, seed=3, device=cuda_device)
    opt = make_opt(params, W, s, torch.float32)
    bufs = gen.alloc()
    gen.next_into(bufs)
    opt.step(bufs)
    opt.refresh_mask()
    for _ in range(3):
        idx_built = opt.idx().clone()
        e_before = [x.clone() for x in opt.e]
        gen.next_into(bufs)
        opt.step(bufs)
        torch.cuda.synchronize()
        used = idx_built.long().cpu().numpy()
        for w in range(W):
            a = bufs[w].cpu().numpy() + e_before[w].cpu().numpy()      # fl(g + e)
            assert np.array_equal(u32(opt.pack()[w]), a[used].view(np.uint32))
        opt.refresh_mask()
    opt.close()


def test_checkpoint_resume_bit_identical(cuda_device):
    P, W, s = 60000, 4, 0.99
    wl = _wl(P, W, s, "bf16")

    def run(split):
        gen = synth.GradientStream(wl, seed=5, device=cuda_device)
        params = synth.init_params(P, seed=5, device=cuda_device)
        opt = make_opt(params, W, s, torch.bfloat16)
        bufs = gen.alloc()
        for t in range(10):
            if t == split:
                saved = (params.clone(), opt.m.clone(), [x.clone() for x in opt.e],
                         opt.bits().clone(), opt.t)
                opt.close()
                params = saved[0]
                opt = make_opt(params, W, s, torch.bfloat16)
                opt.m.copy_(saved[1])
                for dst, src in zip(opt.e, saved[2]):
                    dst.copy_(src)
                opt.set_state(saved[4], saved[3])
            gen.next_into(bufs)
            opt.step(bufs)
            opt.refresh_mask()
        torch.cuda.synchronize()
        out = (u32(params), u32(opt.m), [u32(x) for x in opt.e], u32(opt.bits()))
        opt.close()
        return out

    a, b = run(None), run(5)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert all(np.array_equal(x, y) for x, y in zip(a[2], b[2]))
    assert np.array_equal(a[3], b[3])


def test_state_dict_round_trip(cuda_device):
    """Scape.state_dict / load_state_dict (t, mask, m, residuals, lr) into a
    new instance continues the trajectory bit for bit, with an lr change on
    the way; host-resident residuals included."""
    P, W, s = 70001, 4, 0.95
    wl = _wl(P, W, s, "bf16")

    def run(split, residuals):
        gen = synth.GradientStream(wl, seed=9, device=cuda_device)
        params = synth.init_params(P, seed=9, device=cuda_device)
        opt = make_opt(params, W, s, torch.bfloat16, residuals=residuals)
        bufs = gen.alloc()
        for t in range(8):
            if t == 3:
                opt.set_lr(5e-4)
            if t == split:
                sd, w_ck = opt.state_dict(), params.clone()
                opt.close()
                params = w_ck
                opt = make_opt(params, W, s, torch.bfloat16, residuals=residuals)
                opt.load_state_dict(sd)
            gen.next_into(bufs)
            opt.step(bufs)
            opt.refresh_mask()
        torch.cuda.synchronize()
        out = (u32(params), u32(opt.m), [u32(x) for x in opt.e], u32(opt.bits()))
        opt.close()
        return out

    for residuals in ("device", "host"):
        a, b = run(None, residuals), run(5, residuals)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]), residuals
        assert all(np.array_equal(x, y) for x, y in zip(a[2], b[2])), residuals
        assert np.array_equal(a[3], b[3]), residuals


def test_resume_into_a_live_handle(cuda_device):
    """set_state on a handle that already ran another trajectory: its next
    refresh starts from thresholds of unrelated data and must still give the
    same result as a fresh handle resumed from the same checkpoint."""
    P, W, s = 70001, 5, 0.99
    wl = _wl(P, W, s, "bf16")

    def trajectory(seed, steps):
        gen = synth.GradientStream(wl, seed=seed, device=cuda_device)
        params = synth.init_params(P, seed=seed, device=cuda_device)
        opt = make_opt(params, W, s, torch.bfloat16)
        bufs = gen.alloc()
        for _ in range(steps):
            gen.next_into(bufs)
            opt.step(bufs)
            opt.refresh_mask()
        return opt, params, gen, bufs

    # the checkpoint: 4 steps of seed 21
    src, sp, _, _ = trajectory(21, 4)
    ckpt = (sp.clone(), src.m.clone(), [x.clone() for x in src.e], src.bits().clone(), src.t)
    src.close()
    outs = []
    for live in (False, True):
        if live:
            opt, params, _, _ = trajectory(22, 6)  # a different run on the same handle
            params.copy_(ckpt[0])
        else:
            params = ckpt[0].clone()
            opt = make_opt(params, W, s, torch.bfloat16)
        opt.m.copy_(ckpt[1])
        for dst, x in zip(opt.e, ckpt[2]):
            dst.copy_(x)
        opt.set_state(ckpt[4], ckpt[3])
        gen = synth.GradientStream(wl, seed=23, device=cuda_device)
        bufs = gen.alloc()
        for _ in range(4):
            gen.next_into(bufs)
            opt.step(bufs)
            opt.refresh_mask()
        torch.cuda.synchronize()
        outs.append((u32(params), u32(opt.m), u32(opt.bits()), u32(opt.idx())))
        opt.close()
    for a, b in zip(*outs):
        assert np.array_equal(a, b)


def test_set_state_rejects_wrong_counts(cuda_device):
    P, W, s = 10000, 4, 0.9
    params = torch.zeros(P, device=cuda_device)
    opt = make_opt(params, W, s, torch.float32)
    bad = torch.zeros((P + 31) // 32, dtype=torch.int32, device=cuda_device)
    with pytest.raises(ScapeError):
        opt.set_state(1, bad)
    opt.close()


@pytest.mark.parametrize("P,W,variant,fusion", [(50000, 4, 0, None), (30011, 32, 0, C.FUSE_UPDATE),
                                                (30011, 32, 0, C.FUSE_SUM),
                                                (30011, 32, 0, C.FUSE_NONE),
                                                (20000, 3, 1, None)])
def test_host_buffer_path_matches_device_path(cuda_device, P, W, variant, fusion):
    """scape_step_host (uploads in worker groups, the parameter download before
    the update plus a patch of the changed coordinates, or after it under the
    dense off-mask reading) leaves the same parameters on the host after every
    step as the device path; the host output is poisoned before each step."""
    s = 0.9
    wl = _wl(P, W, s, "bf16")
    per_step = []
    for host in (False, True):
        gen = synth.GradientStream(wl, seed=9, device="cpu")
        params = synth.init_params(P, seed=9).to(cuda_device)
        opt = make_opt(params, W, s, torch.bfloat16)
        if variant:
            opt.set_variant(variant)
        if fusion is not None:
            opt.set_fusion(fusion)
        dev = [torch.empty(P, dtype=torch.bfloat16, device=cuda_device) for _ in range(W)]
        pin = [torch.empty(P, dtype=torch.bfloat16).pin_memory() for _ in range(W)]
        out = torch.empty(P, dtype=torch.float32).pin_memory()
        got = []
        for _ in range(5):
            grads = gen.next()
            out.fill_(float("nan"))
            if host:
                for p_, g in zip(pin, grads):
                    p_.copy_(g)
                opt.step_host(pin, dev, out)
            else:
                for d, g in zip(dev, grads):
                    d.copy_(g)
                opt.step(dev)
                opt.refresh_mask()
                out.copy_(params)
            torch.cuda.synchronize()
            got.append(out.numpy().copy())
        per_step.append(got)
        opt.close()
    for a, b in zip(*per_step):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("fusion", [C.FUSE_NONE, C.FUSE_SUM, C.FUSE_UPDATE])
def test_step_without_refresh_reuses_the_older_mask(cuda_device, fusion):
    """Skipping a refresh reuses the older mask.  Pattern: step 1,
    refresh, steps 2 and 3 on that mask, refresh, step 4, refresh -- against
    the oracle's steps taken in the same order."""
    P, W, s = 70001, 4, 0.99
    wl = _wl(P, W, s, "bf16")
    gen = synth.GradientStream(wl, seed=31, device="cpu")
    w0 = synth.init_params(P, seed=31)
    params = w0.to(cuda_device)
    opt = make_opt(params, W, s, torch.bfloat16)
    opt.set_fusion(fusion)
    st = O.new_state(w0.numpy(), W, s, HP)
    bits, idx = O.dense_mask(P)
    for t, refresh in ((1, True), (2, False), (3, True), (4, True)):
        grads = gen.next()
        opt.step([g.to(cuda_device) for g in grads])
        O.step(t, [synth.to_numpy_grad(g) for g in grads], st.e, st.w, st.m, bits, idx, HP)
        if refresh:
            opt.refresh_mask()
            bits, idx = O.topk_mask(st.m, st.shard_start, st.shard_k)
    torch.cuda.synchronize()
    assert np.array_equal(u32(opt.bits()), bits)
    assert np.array_equal(u32(params), st.w.view(np.uint32))
    assert np.array_equal(u32(opt.m), st.m.view(np.uint32))
    for w in range(W):
        assert np.array_equal(u32(opt.e[w]), st.e[w].view(np.uint32))
    opt.close()


def test_random_access_probe_changes_nothing(cuda_device):
    """The timing probe reads and writes back w and m at the mask's
    coordinates: both stay bit for bit what they were."""
    P, W, s = 100003, 4, 0.99
    wl = _wl(P, W, s, "bf16")
    gen = synth.GradientStream(wl, seed=2, device=cuda_device)
    params = synth.init_params(P, seed=2, device=cuda_device)
    opt = make_opt(params, W, s, torch.bfloat16)
    bufs = gen.alloc()
    with pytest.raises(ScapeError):
        opt.probe_random_access()          # no mask yet
    for _ in range(3):
        gen.next_into(bufs)
        opt.step(bufs)
        opt.refresh_mask()
    w0, m0 = params.clone(), opt.m.clone()
    opt.probe_random_access()
    torch.cuda.synchronize()
    assert torch.equal(params.view(torch.int32), w0.view(torch.int32))
    assert torch.equal(opt.m.view(torch.int32), m0.view(torch.int32))
    opt.close()


def test_state_errors(cuda_device):
    P, W = 1000, 2
    params = torch.zeros(P, device=cuda_device)
    opt = make_opt(params, W, 0.9, torch.float32)
    with pytest.raises(ScapeError):
        opt.refresh_mask()                         # nothing to build a mask from
    g = [torch.zeros(P, device=cuda_device) for _ in range(W)]
    opt.step(g)
    with pytest.raises(ScapeError):
        opt.step(g)                                # no mask built after step 1
    opt.close()


def test_profiling_counts_launches(cuda_device):
    P, W = 100000, 4
    params = torch.zeros(P, device=cuda_device)
    opt = make_opt(params, W, 0.9, torch.float32)
    g = [torch.randn(P, device=cuda_device) * 1e-3 for _ in range(W)]
    opt.profile(True)
    n0 = opt.launch_count()
    for _ in range(3):
        opt.step(g)
        opt.refresh_mask()
    torch.cuda.synchronize()
    opt.profile_collect()
    prof = opt.profile_read()
    assert prof["ef_compact"][1] == 2 and prof["dense_step"][1] == 1
    assert prof["ef_compact"][0] > 0
    assert opt.launch_count() - n0 == sum(n for _, n in prof.values())
    # launches of one sparse step at each fusion level
    for level, n_red, n_upd in ((C.FUSE_NONE, 1, 1), (C.FUSE_SUM, 0, 1), (C.FUSE_UPDATE, 0, 0)):
        opt.set_fusion(level)
        opt.profile_reset()
        opt.step(g)
        torch.cuda.synchronize()
        opt.profile_collect()
        prof = opt.profile_read()
        assert prof["ef_compact"][1] == 1
        assert (prof["reduce"][1], prof["adams_sparse"][1]) == (n_red, n_upd), level
    with pytest.raises(ScapeError):
        opt.set_fusion(3)
    # profiling restricted to one kernel brackets only its launches
    opt.profile_select(["ef_compact"])
    opt.profile_reset()
    opt.step(g)
    opt.refresh_mask()
    torch.cuda.synchronize()
    opt.profile_collect()
    prof = opt.profile_read()
    assert {k for k, (_, n) in prof.items() if n} == {"ef_compact"}
    opt.close()


# ------------------------------------------------------------ full-size workloads, sampled shards
@pytest.mark.parametrize("name,steps,shards", [
    # ten steps at full size: nine lagged sparse steps and ten refreshes (eight
    # of them warm), each mask used by the next step; first, a middle and the
    # last shard, the oracle running them in parallel processes
    ("gpt345m", 10, (0, 3, 7)),
    ("llama500m", 10, (0, 17, 31)),
    ("llama1p8b", 10, (0, 3, 7)),
])
def test_full_size_sampled_shards(cuda_device, name, steps, shards):
    wl = synth.WORKLOADS[name]
    torch.cuda.empty_cache()
    rep = run_sampled_shards(wl, cuda_device, steps, shards)
    assert rep.exact, f"not bit-identical ({rep.flips} mask flips of {rep.mask_bits})"
    torch.cuda.empty_cache()


def test_flat_sweep_largest_point_sampled(cuda_device):
    wl = synth.flat_workload(1 << 30, 8, 0.99)
    rep = run_sampled_shards(wl, cuda_device, 3, (0, 7))
    assert rep.exact
    torch.cuda.empty_cache()


# ------------------------------------------------------------ residuals in host memory
@pytest.mark.parametrize("P,W,s,dtype", [(70001, 4, 0.99, "bf16"), (4096, 2, 0.9, "f32"),
                                         (50003, 13, 0.99, "bf16")])
@pytest.mark.parametrize("staging", [0, 3, 4, 7, 64])
def test_host_resident_residuals_match_oracle(cuda_device, P, W, s, dtype, staging):
    """Error-feedback buffers in pinned host memory, read and written in place
    by the kernels (staging 0), or moved through a device staging buffer of
    that many rows in worker groups: same trajectory as the oracle, bit for
    bit."""
    gdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    wl = _wl(P, W, s, dtype)
    gen = synth.GradientStream(wl, seed=8, device="cpu")
    w0 = synth.init_params(P, seed=8)
    params = w0.to(cuda_device)
    opt = Scape(params, W, s, lr=HP.lr, beta1=HP.beta1, beta2=HP.beta2, eps=HP.eps,
                weight_decay=HP.weight_decay, grad_dtype=gdt, residuals="host",
                staging_rows=staging)
    assert (opt.staging is None) == (staging == 0)
    assert not opt.e[0].is_cuda
    st = O.new_state(w0.numpy(), W, s, HP)
    for _ in range(6):
        grads = gen.next()
        opt.step([g.to(cuda_device) for g in grads])
        opt.refresh_mask()
        O.advance(st, [synth.to_numpy_grad(g) for g in grads])
    torch.cuda.synchronize()
    assert np.array_equal(u32(params), st.w.view(np.uint32))
    assert np.array_equal(u32(opt.m), st.m.view(np.uint32))
    for w in range(W):
        assert np.array_equal(opt.e[w].numpy().view(np.uint32), st.e[w].view(np.uint32))
    assert np.array_equal(u32(opt.bits()), st.bits)
    opt.close()


# ------------------------------------------------------------ writes stay inside their buffers
_PAD_WORDS = 1024
_CANARY = 0x7FBADBAD


def _canaried(n, dtype, device):
    """n elements of `dtype` followed by _PAD_WORDS canary words; returns the
    element view and the 32-bit words behind it."""
    esz = torch.empty(0, dtype=dtype).element_size()
    words = (n * esz + 3) // 4
    full = torch.full((words + _PAD_WORDS,), _CANARY, dtype=torch.int32, device=device)
    view = full[:words].view(dtype)[:n]
    return view, full, words


@pytest.mark.parametrize("P,W,s,dtype", [(70001, 5, 0.9, "bf16"), (5003, 3, 0.99, "f32"),
                                         (1 << 16, 4, 0.999, "bf16"), (3000, 256, 0.9, "f32")])
def test_no_write_past_any_buffer(cuda_device, P, W, s, dtype):
    """Every buffer the library writes (w, m, residuals, workspace, union
    workspace) is followed by canary words; after dense, sparse and union
    steps and cold and warm refreshes they must be intact."""
    gdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    wl = _wl(P, W, s, dtype)
    gen = synth.GradientStream(wl, seed=4, device="cpu")
    checks = []
    params, fp, wp = _canaried(P, torch.float32, cuda_device)
    params.copy_(synth.init_params(P, seed=4))
    m, fm, wm = _canaried(P, torch.float32, cuda_device)
    m.zero_()
    checks += [(fp, wp), (fm, wm)]
    es = []
    for _ in range(W):
        e, fe, we = _canaried(P, torch.float32, cuda_device)
        e.zero_()
        es.append(e)
        checks.append((fe, we))
    gs = []
    for _ in range(W):
        g, fg, wg = _canaried(P, gdt, cuda_device)
        gs.append(g)
        checks.append((fg, wg))
    h = C.scape_create([P], W, s, HP.beta1, HP.beta2, HP.lr, HP.eps, HP.weight_decay,
                       C.SCAPE_BF16 if dtype == "bf16" else C.SCAPE_F32)
    nws = C.scape_workspace_bytes(h)
    ws, fws, wws = _canaried(nws, torch.uint8, cuda_device)
    checks.append((fws, wws))
    C.scape_bind(h, params.data_ptr(), m.data_ptr(), [e.data_ptr() for e in es], ws.data_ptr(),
                 nws)
    st = torch.cuda.current_stream().cuda_stream
    for t in range(5):
        for g, x in zip(gs, gen.next()):
            g.copy_(x.to(cuda_device))
        C.scape_step(h, [g.data_ptr() for g in gs], st)
        C.scape_refresh_mask(h, st)
    nu = C.scape_union_workspace_bytes(h, P)
    uws, fu, wu = _canaried(nu, torch.uint8, cuda_device)
    checks.append((fu, wu))
    for g, x in zip(gs, gen.next()):
        g.copy_(x.to(cuda_device))
    C.scape_union_step(h, [g.data_ptr() for g in gs], uws.data_ptr(), nu, P, st)
    torch.cuda.synchronize()
    C.scape_destroy(h)
    for full, words in checks:
        assert bool((full[words:] == _CANARY).all())

"""GPU parity of the exchange-based multi-rank step (scape_xc_*, exchange.py)
against the CPU oracle's single-process trajectory.

Rank r of G owns the workers and optimizer shards rank_shards(W, G, r); it has
the full gradients and residuals of its own workers only, so the step needs
the three collectives of "SCAPE" Sec. I (sparse reduce-scatter of the packed
values, done as an all-to-all with the owner summing in worker order; sparse
parameter all-gather) and the mask all-gather of "Sintesi Tecnica: SCAPE"
Sec. 2.  Whatever G, the result must be the oracle's bit for bit: the global
mask after every step, every rank's parameter replica, the owners' first
moments and every worker's residual.

G = 1 runs in this process (the collectives reduce to copies); G = 2 and 3 run
as gloo ranks in child processes that all use cuda:0 (their kernels never
wait on each other; only the host-side collectives synchronise them)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import oracle as O
from sparse_communication_sharded_gb300 import synth

pytestmark = pytest.mark.gpu

HPV = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
CASES = {
    "bf16": dict(layers=(("a", 120000), ("b", 30011)), W=8, s=0.99, dtype="bf16", steps=7),
    "f32_ties": dict(layers=(("a", 50003),), W=6, s=0.9, dtype="f32", steps=6, quant=True),
}


def _wl(c):
    return synth.Workload("xc", c["layers"], W=c["W"], sparsity=c["s"], steps=c["steps"],
                          grad_dtype=c["dtype"], quantum=2.0 ** -15 if c.get("quant") else None)


def _run(c, rank, world, out_path):
    import sparse_communication_sharded_gb300 as pkg  # noqa: F401  (loads the library)
    from sparse_communication_sharded_gb300 import multirank
    from sparse_communication_sharded_gb300.exchange import ScapeDP

    dev = torch.device("cuda:0")
    wl = _wl(c)
    P, W = wl.P, wl.W
    mine = multirank.rank_shards(W, world, rank)
    gdt = torch.bfloat16 if c["dtype"] == "bf16" else torch.float32
    params = synth.init_params(P, seed=23).to(dev)
    # with several ranks, every step first checks on the host that all of them
    # reached it (check_peers over a file store)
    live = (dist.FileStore(os.path.join(os.path.dirname(out_path), "live"), world)
            if world > 1 else None)
    opt = ScapeDP(params, W, c["s"], layer_numel=[n for _, n in wl.layers], grad_dtype=gdt,
                  liveness=live, **HPV)
    assert opt.Wl == len(mine)
    gen = synth.GradientStream(wl, seed=23, device="cpu")
    bits = []
    for _ in range(c["steps"]):
        grads = gen.next()
        opt.step([grads[w].to(dev) for w in mine])
        torch.cuda.synchronize()
        bits.append(opt.global_bits().cpu().numpy().view(np.uint32).copy())
    assert opt.steps == c["steps"]
    res = {"w": params.cpu().numpy(), "m": opt.m.cpu().numpy(), "own": np.array(opt.own),
           "bits": np.stack(bits), "launches": opt.launch_count()}
    for j, w in enumerate(mine):
        res[f"e{w}"] = opt.e[j].cpu().numpy()
    opt.close()
    np.savez(out_path.format(rank=rank), **res)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, name, out_path):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        _run(CASES[name], rank, world, out_path)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _oracle(c):
    wl = _wl(c)
    gen = synth.GradientStream(wl, seed=23, device="cpu")
    st = O.new_state(synth.init_params(wl.P, seed=23).numpy(), wl.W, c["s"], O.Hyper(**HPV))
    bits = []
    for _ in range(c["steps"]):
        O.advance(st, [synth.to_numpy_grad(g) for g in gen.next()], keep=())
        bits.append(st.bits.copy())
    return st, np.stack(bits)


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("world", [1, 2, 3])
def test_exchange_step_matches_single_process_oracle(cuda_device, tmp_path, name, world):
    c = CASES[name]
    out = str(tmp_path / "rank{rank}.npz")
    if world == 1:
        _run(c, 0, 1, out)
    else:
        mp.spawn(_rank, args=(world, _free_port(), name, out), nprocs=world, join=True)
    st, bits = _oracle(c)
    for r in range(world):
        res = np.load(out.format(rank=r))
        assert np.array_equal(res["bits"], bits), f"rank {r}: mask differs"
        assert np.array_equal(res["w"].view(np.uint32), st.w.view(np.uint32)), f"rank {r}: w"
        lo, hi = res["own"]
        assert np.array_equal(res["m"].view(np.uint32), st.m[lo:hi].view(np.uint32))
        for key in res.files:
            if key.startswith("e"):
                w = int(key[1:])
                assert np.array_equal(res[key].view(np.uint32), st.e[w].view(np.uint32)), key


def _resume_rank(rank, world, port, name, out_path, split):
    """`split` steps, a checkpoint (w, the owned m, the local residuals, t and
    the global mask), a fresh handle resumed from it, then the remaining
    steps."""
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import sparse_communication_sharded_gb300 as pkg  # noqa: F401
        from sparse_communication_sharded_gb300 import multirank
        from sparse_communication_sharded_gb300.exchange import ScapeDP

        c = CASES[name]
        dev = torch.device("cuda:0")
        wl = _wl(c)
        mine = multirank.rank_shards(wl.W, world, rank)
        gdt = torch.bfloat16 if c["dtype"] == "bf16" else torch.float32
        kw = dict(layer_numel=[n for _, n in wl.layers], grad_dtype=gdt, **HPV)
        gen = synth.GradientStream(wl, seed=23, device="cpu")
        params = synth.init_params(wl.P, seed=23).to(dev)
        opt = ScapeDP(params, wl.W, c["s"], **kw)
        for _ in range(split):
            grads = gen.next()
            opt.step([grads[w].to(dev) for w in mine])
        t, bits = opt.get_state()
        ck = {"w": params.clone(), "m": opt.m.clone(), "e": [x.clone() for x in opt.e]}
        opt.close()
        # a new handle and new buffers, restored from the checkpoint
        params2 = ck["w"].clone()
        opt2 = ScapeDP(params2, wl.W, c["s"], **kw)
        opt2.m.copy_(ck["m"])
        for x, y in zip(opt2.e, ck["e"]):
            x.copy_(y)
        opt2.set_state(t, bits)
        assert opt2.t == t == split
        for _ in range(c["steps"] - split):
            grads = gen.next()
            opt2.step([grads[w].to(dev) for w in mine])
        torch.cuda.synchronize()
        res = {"w": params2.cpu().numpy(), "m": opt2.m.cpu().numpy(), "own": np.array(opt2.own),
               "bits": opt2.global_bits().cpu().numpy().view(np.uint32).copy()}
        for j, w in enumerate(mine):
            res[f"e{w}"] = opt2.e[j].cpu().numpy()
        opt2.close()
        np.savez(out_path.format(rank=rank), **res)
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("name", sorted(CASES))
def test_exchange_resume_matches_uninterrupted_oracle(cuda_device, tmp_path, name):
    """Checkpoint/resume of the multi-rank step (scape_xc_set_state): two ranks
    stop after 3 steps, new handles resume from the checkpoint, and the end
    state equals the oracle's uninterrupted trajectory bit for bit."""
    c = CASES[name]
    world = 2
    out = str(tmp_path / "rank{rank}.npz")
    mp.spawn(_resume_rank, args=(world, _free_port(), name, out, 3), nprocs=world, join=True)
    st, bits = _oracle(c)
    for r in range(world):
        res = np.load(out.format(rank=r))
        assert np.array_equal(res["bits"], bits[-1]), f"rank {r}: mask differs"
        assert np.array_equal(res["w"].view(np.uint32), st.w.view(np.uint32)), f"rank {r}: w"
        lo, hi = res["own"]
        assert np.array_equal(res["m"].view(np.uint32), st.m[lo:hi].view(np.uint32))
        for key in res.files:
            if key.startswith("e"):
                w = int(key[1:])
                assert np.array_equal(res[key].view(np.uint32), st.e[w].view(np.uint32)), key

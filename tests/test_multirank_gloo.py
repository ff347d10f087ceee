"""World-size-2 gloo test of the multi-rank path on CPU: ranks split the
optimizer shards, each runs its shards as independent problems (the CPU oracle
stands in for the GPU kernels here), and the gathered result equals the
single-process run bit for bit; the timing reduction takes the max over ranks."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import oracle as O
from sparse_communication_sharded_gb300 import multirank, synth

P, W, S, STEPS = 6000, 4, 0.9, 4


def _inputs():
    wl = synth.Workload("t", (("flat", P),), W=W, sparsity=S, steps=STEPS, grad_dtype="f32")
    gen = synth.GradientStream(wl, seed=11, device="cpu")
    grads = [[synth.to_numpy_grad(g) for g in gen.next()] for _ in range(STEPS)]
    w0 = synth.init_params(P, seed=11).numpy()
    return w0, grads


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_path):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w0, grads = _inputs()
    start, ks = O.layout(P, W, S)
    mine = multirank.rank_shards(W, world, rank)
    w_out = np.zeros(P, np.float32)
    m_out = np.zeros(P, np.float32)
    for sh in mine:
        lo, hi = int(start[sh]), int(start[sh + 1])
        st = O.new_state(w0[lo:hi], W, S, O.Hyper(), shard_start=np.array([0, hi - lo]),
                         shard_k=np.array([ks[sh]]))
        for g in grads:
            O.advance(st, [x[lo:hi].copy() for x in g], keep=())
        w_out[lo:hi] = st.w
        m_out[lo:hi] = st.m
    # gather the disjoint pieces (result collection only; nothing on the data path)
    wt, mt = torch.from_numpy(w_out), torch.from_numpy(m_out)
    dist.all_reduce(wt)
    dist.all_reduce(mt)
    t_max = multirank.max_over_ranks(1.0 + rank)
    if rank == 0:
        np.savez(out_path, w=wt.numpy(), m=mt.numpy(), t_max=t_max)
    dist.barrier()
    dist.destroy_process_group()


def test_rank_shards_partition():
    for n in (1, 4, 7, 32):
        for world in (1, 2, 3, 8):
            got = [s for r in range(world) for s in multirank.rank_shards(n, world, r)]
            assert got == list(range(n))
    with pytest.raises(ValueError):
        multirank.rank_shards(4, 2, 2)


def test_two_gloo_ranks_match_single_process(tmp_path):
    out = str(tmp_path / "res.npz")
    mp.spawn(_worker, args=(2, _free_port(), out), nprocs=2, join=True)
    res = np.load(out)
    w0, grads = _inputs()
    st = O.new_state(w0, W, S, O.Hyper())
    for g in grads:
        O.advance(st, g, keep=())
    assert np.array_equal(res["w"].view(np.uint32), st.w.view(np.uint32))
    assert np.array_equal(res["m"].view(np.uint32), st.m.view(np.uint32))
    assert float(res["t_max"]) == 2.0
    assert multirank.weak_scaling_value(100, 2, 0.5) == 400.0

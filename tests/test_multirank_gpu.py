"""The multi-rank split through the CUDA library: two processes, both on
cuda:0, each a rank of a gloo group.  Rank r owns the block of optimizer
shards rank_shards(W, 2, r) ("SCAPE" Sec. II-A: the distributed optimizer
partitions states and parameters evenly; "Sintesi Tecnica: SCAPE" Sec. 2:
each worker builds the mask of its own partition), holds a range handle over
its parameter slice and steps the slices of all W workers' gradients through
libscape.so.  Nothing is exchanged on the data path; at the end the ranks
gather their w, m and mask slices, which must equal the single-process CPU
oracle's whole-problem results bit for bit.

The two processes' kernels never wait on each other (only the host-side
gloo calls synchronise them), so sharing one GPU is safe."""
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

P, W, S, STEPS = 200003, 8, 0.99, 7
HPV = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)


def _wl():
    return synth.Workload("split", (("a", 150000), ("b", 50003)), W=W, sparsity=S, steps=STEPS,
                          grad_dtype="bf16")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out_path):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import sparse_communication_sharded_gb300 as pkg
    from sparse_communication_sharded_gb300 import multirank

    dev = torch.device("cuda:0")
    wl = _wl()
    shards = multirank.rank_shards(W, world, rank)
    lo, hi = multirank.shard_slice(P, W, shards)
    w0 = synth.init_params(P, seed=17)
    params = w0[lo:hi].clone().to(dev)
    opt = pkg.Scape(params, W, S, layer_numel=[n for _, n in wl.layers],
                    shard_range=(shards.start, shards.stop), grad_dtype=torch.bfloat16, **HPV)
    # every rank draws the same whole-problem gradients and keeps its slices
    gen = synth.GradientStream(wl, seed=17, device="cpu")
    for _ in range(STEPS):
        grads = gen.next()
        opt.step([g[lo:hi].to(dev) for g in grads])
        opt.refresh_mask()
    torch.cuda.synchronize()
    bits = opt.bits().cpu().numpy().view(np.uint32)
    mask = torch.from_numpy(np.unpackbits(bits.view(np.uint8), bitorder="little")[:hi - lo]
                            .astype(np.int32))
    w_all = multirank.gather_slices(params.cpu(), lo, P)
    m_all = multirank.gather_slices(opt.m.cpu(), lo, P)
    mask_all = multirank.gather_slices(mask, lo, P)
    opt.close()
    if rank == 0:
        np.savez(out_path, w=w_all.numpy(), m=m_all.numpy(), mask=mask_all.numpy())
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_on_one_gpu_match_single_process_oracle(cuda_device, tmp_path):
    out = str(tmp_path / "res.npz")
    mp.spawn(_rank, args=(2, _free_port(), out), nprocs=2, join=True)
    res = np.load(out)
    wl = _wl()
    gen = synth.GradientStream(wl, seed=17, device="cpu")
    st = O.new_state(synth.init_params(P, seed=17).numpy(), W, S, O.Hyper(**HPV))
    for _ in range(STEPS):
        O.advance(st, [synth.to_numpy_grad(g) for g in gen.next()], keep=())
    want_mask = np.unpackbits(st.bits.view(np.uint8), bitorder="little")[:P]
    assert np.array_equal(res["mask"].astype(np.uint8), want_mask)
    assert np.array_equal(res["w"].view(np.uint32), st.w.view(np.uint32))
    assert np.array_equal(res["m"].view(np.uint32), st.m.view(np.uint32))

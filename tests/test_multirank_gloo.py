"""World-size-2 (and 3) gloo tests of the multi-rank split on the CPU.

Each rank builds the library handle of its own block of optimizer shards
(scape_create_range: host-only, no GPU work) and the ranks gather what their
handles report.  Together the handles must tile the whole problem exactly as
the oracle lays it out ("SCAPE" Sec. II-A, even partition; "Sintesi Tecnica:
SCAPE" Sec. 2, per-partition masks): the parameter slices partition [0, P), the
local shard boundaries shifted by each slice's offset are the global ones, the
per-shard k_s are the global k_s and the k sum to the global k.  The same
gather helper the multi-GPU tests use reassembles a vector from the ranks'
slices, and the timing reductions take the max and the sum over ranks.  (The
GPU run of the split, each rank stepping its shards through the CUDA library,
is tests/test_multirank_gpu.py.)"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import oracle as O
from sparse_communication_sharded_gb300 import _scape as C
from sparse_communication_sharded_gb300 import build as B
from sparse_communication_sharded_gb300 import multirank

LAYERS = [1000, 70001, 33, 12345]   # P = 83379
W, S = 8, 0.99


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
    mine = multirank.rank_shards(W, world, rank)
    h = C.scape_create_range(LAYERS, W, mine.start, mine.stop, S, 0.9, 0.95, 1e-3, 1e-8, 0.1,
                             C.SCAPE_BF16)
    geo = C.scape_get_geometry(h)
    rng = C.scape_get_range(h)
    C.scape_destroy(h)
    P = sum(LAYERS)
    lo, hi = multirank.shard_slice(P, W, mine)
    assert (rng["offset"], rng["offset"] + geo["P"]) == (lo, hi)
    # per-shard global start and k, reassembled from every rank's handle
    starts = torch.tensor([rng["offset"] + x for x in geo["shard_start"][:-1]], dtype=torch.int64)
    ks = torch.tensor(geo["shard_k"], dtype=torch.int64)
    all_starts = multirank.gather_slices(starts, mine.start, W)
    all_k = multirank.gather_slices(ks, mine.start, W)
    # a parameter vector reassembled from the ranks' slices
    vec = multirank.gather_slices(torch.arange(lo, hi, dtype=torch.float64), lo, P)
    k_sum = multirank.sum_over_ranks(geo["k"])
    t_max = multirank.max_over_ranks(1.0 + rank)
    if rank == 0:
        np.savez(out_path, starts=all_starts.numpy(), k=all_k.numpy(), vec=vec.numpy(),
                 k_sum=k_sum, t_max=t_max, P_global=rng["P_global"])
    dist.barrier()
    dist.destroy_process_group()


def test_rank_shards_partition():
    for n in (1, 4, 7, 32):
        for world in (1, 2, 3, 8):
            got = [s for r in range(world) for s in multirank.rank_shards(n, world, r)]
            assert got == list(range(n))
    with pytest.raises(ValueError):
        multirank.rank_shards(4, 2, 2)


@pytest.mark.parametrize("world", [2, 3])
def test_rank_handles_tile_the_global_layout(tmp_path, world):
    B.build()
    out = str(tmp_path / "res.npz")
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    res = np.load(out)
    P = sum(LAYERS)
    start, ks = O.layout(P, W, S)
    assert int(res["P_global"]) == P
    assert np.array_equal(res["starts"], start[:-1])
    assert np.array_equal(res["k"], ks)
    assert int(res["k_sum"]) == int(ks.sum())
    assert np.array_equal(res["vec"], np.arange(P, dtype=np.float64))
    assert float(res["t_max"]) == float(world)
    assert multirank.weak_scaling_value(100, 2, 0.5) == 400.0
    assert multirank.strong_scaling_value(100, 0.5) == 200.0


def test_range_handle_argument_errors():
    B.build()
    for a, b in ((-1, 2), (3, 3), (5, 4), (0, W + 1)):
        with pytest.raises(C.ScapeError):
            C.scape_create_range(LAYERS, W, a, b, S, 0.9, 0.95, 1e-3, 1e-8, 0.1, C.SCAPE_F32)
    # P < W: a range of empty shards holds no parameter
    with pytest.raises(C.ScapeError):
        C.scape_create_range([5], 8, 0, 1, 0.5, 0.9, 0.95, 1e-3, 1e-8, 0.1, C.SCAPE_F32)
    h = C.scape_create_range([5], 8, 0, 2, 0.5, 0.9, 0.95, 1e-3, 1e-8, 0.1, C.SCAPE_F32)
    geo = C.scape_get_geometry(h)
    C.scape_destroy(h)
    assert geo["P"] == 1 and geo["shard_start"] == [0, 0, 1] and geo["shard_k"] == [0, 1]

"""The exchange's collectives and buffer layout, on CPU gloo ranks.

Each rank creates its exchange handle (scape_xc_create: host only) and reads
the per-rank element counts of the step's three collectives
(scape_xc_counts).  It fills a send buffer in the documented layout -- one
block per destination rank q, rows = its local workers in order, columns =
q's coordinates padded to a multiple of 4 -- with values that name (worker,
destination, column), and runs exchange.all_to_all and all_gather_rows as the
GPU step does.  Every owner must then hold the W workers' rows of its own
columns in global worker order (what the owner's ordered sum needs: "SCAPE"
Sec. I sparse reduce-scatter, Sec. II-A one optimizer shard per worker), and
every rank every owner's parameter values and mask words at that owner's
row.  The GPU trajectory through these buffers is tests/test_exchange_gpu.py."""
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
from sparse_communication_sharded_gb300.exchange import all_gather_rows, all_to_all

LAYERS, W, S = [5000, 3003], 6, 0.9


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _tag(w, q, j):
    return float(w * 1_000_000 + q * 100_000 + j)


def _worker(rank, world, port, out_path):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    h = C.scape_xc_create(LAYERS, W, world, rank, S, 0.9, 0.95, 1e-3, 1e-8, 0.1, C.SCAPE_F32)
    lay = C.scape_xc_layout(h)
    cnt = C.scape_xc_counts(h, world)
    C.scape_xc_destroy(h)
    mine = multirank.rank_shards(W, world, rank)
    P = sum(LAYERS)
    start, _ = O.layout(P, W, S)
    assert (lay["own_begin"], lay["own_end"]) == (start[mine.start], start[mine.stop])
    assert lay["local_workers"] == len(mine)
    # step 1 (dense): rank q's columns are its whole parameter range
    cols = [int(start[multirank.rank_shards(W, world, q).stop] -
                start[multirank.rank_shards(W, world, q).start]) for q in range(world)]
    pad = [(c + 3) // 4 * 4 for c in cols]
    assert cnt["send"] == [len(mine) * p for p in pad]
    assert cnt["params"] == cols
    send = []
    for q in range(world):
        blk = np.full((len(mine), pad[q]), np.nan, np.float32)
        for r, w in enumerate(mine):
            blk[r, :cols[q]] = [_tag(w, q, j) for j in range(cols[q])]
        send.append(blk.ravel())
    send = torch.from_numpy(np.concatenate(send))
    recv = torch.empty(sum(cnt["recv"]), dtype=torch.float32)
    all_to_all(recv, send, cnt["recv"], cnt["send"], via_host=True)
    got = recv.numpy().reshape(W, pad[rank])[:, :cols[rank]]
    want = np.array([[_tag(w, rank, j) for j in range(cols[rank])] for w in range(W)],
                    np.float32)
    ok_a2a = bool(np.array_equal(got, want))
    ps, ms = cnt["param_stride"], cnt["mask_stride"]
    prow = torch.full((ps,), -1.0)
    prow[:cols[rank]] = torch.arange(cols[rank], dtype=torch.float32) + 10_000 * rank
    pout = torch.empty(world * ps)
    all_gather_rows(pout, prow, world, via_host=True)
    mrow = torch.full((ms,), rank + 1, dtype=torch.int32)
    mout = torch.empty(world * ms, dtype=torch.int32)
    all_gather_rows(mout, mrow, world, via_host=True)
    ok_p = all(np.array_equal(pout.numpy()[q * ps:q * ps + cols[q]],
                              np.arange(cols[q], dtype=np.float32) + 10_000 * q)
               for q in range(world))
    ok_m = all((mout.numpy()[q * ms:(q + 1) * ms] == q + 1).all() for q in range(world))
    words = cnt["mask_words"]
    ok_w = all(words[q] == (int(start[multirank.rank_shards(W, world, q).stop]) + 31) // 32
               - int(start[multirank.rank_shards(W, world, q).start]) // 32
               for q in range(world))
    flags = torch.tensor([ok_a2a, ok_p, ok_m, ok_w], dtype=torch.int32)
    dist.all_reduce(flags, op=dist.ReduceOp.MIN)
    if rank == 0:
        np.save(out_path, flags.numpy())
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_exchange_layout_and_collectives(tmp_path, world):
    B.build()
    out = str(tmp_path / "flags.npy")
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert np.load(out).tolist() == [1, 1, 1, 1]


def test_exchange_handle_argument_errors():
    B.build()
    for G, rank in ((0, 0), (W + 1, 0), (2, 2), (2, -1)):
        with pytest.raises(C.ScapeError):
            C.scape_xc_create(LAYERS, W, G, rank, S, 0.9, 0.95, 1e-3, 1e-8, 0.1, C.SCAPE_F32)

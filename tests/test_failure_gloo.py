"""Failure detection of the multi-rank step on CPU ranks (gloo), with no GPU
work: a rank that leaves between steps is noticed by the others on the host,
before they launch the next step's kernels or collectives (check_peers over a
store), or, without that check, as an error of the next collective once the
process group's timeout expires."""
import json
import os
import socket
import time
from datetime import timedelta

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from sparse_communication_sharded_gb300 import exchange


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _liveness_worker(rank, world, store_path, out_dir, leaver, leave_at):
    store = dist.FileStore(store_path, world)
    log = []
    for step in range(3):
        if rank == leaver and step == leave_at:
            log.append({"step": step, "left": True})
            break
        t0 = time.monotonic()
        try:
            exchange.check_peers(store, rank, world, step, timeout=timedelta(seconds=2))
            log.append({"step": step, "ok": True})
        except exchange.PeerLost as e:
            log.append({"step": step, "missing": e.missing, "secs": time.monotonic() - t0})
            break
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(log, f)


def test_check_peers_names_the_rank_that_left(tmp_path):
    world, leaver, leave_at = 3, 2, 1
    mp.spawn(_liveness_worker, args=(world, str(tmp_path / "store"), str(tmp_path), leaver,
                                     leave_at), nprocs=world, join=True)
    logs = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    assert logs[leaver] == [{"step": 0, "ok": True}, {"step": 1, "left": True}]
    for r in range(world):
        if r == leaver:
            continue
        assert logs[r][0] == {"step": 0, "ok": True}
        last = logs[r][1]
        assert last["step"] == 1 and last["missing"] == [leaver]
        assert last["secs"] < 15


def test_check_peers_passes_when_all_arrive(tmp_path):
    world = 2
    mp.spawn(_liveness_worker, args=(world, str(tmp_path / "store"), str(tmp_path), -1, -1),
             nprocs=world, join=True)
    for r in range(world):
        log = json.load(open(tmp_path / f"rank{r}.json"))
        assert log == [{"step": s, "ok": True} for s in range(3)]


def _collective_worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=timedelta(seconds=3))
    row = torch.full((4,), float(rank))
    out = torch.empty(4 * world)
    exchange.all_gather_rows(out, row, world, via_host=True)   # step 0: everyone
    result = {"first": out.tolist()}
    if rank == 1:
        result["left"] = True          # leaves between steps, nothing in flight
    else:
        t0 = time.monotonic()
        try:
            exchange.all_gather_rows(out, row, world, via_host=True)
            result["second"] = "completed"
        except Exception as e:  # gloo reports the lost peer or the timeout
            result["second"] = type(e).__name__
            result["secs"] = time.monotonic() - t0
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(result, f)
    os._exit(0)  # no teardown collective with a peer that has left


def test_collective_errors_after_a_rank_left(tmp_path):
    world = 2
    mp.spawn(_collective_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
             join=True)
    r0 = json.load(open(tmp_path / "rank0.json"))
    r1 = json.load(open(tmp_path / "rank1.json"))
    assert r0["first"] == r1["first"] == [0.0] * 4 + [1.0] * 4
    assert r1["left"]
    assert r0["second"] != "completed"
    assert r0["secs"] < 60

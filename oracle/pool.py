"""Shard-parallel runner of the CPU oracle: one worker process per optimizer
shard, inputs and outputs in shared memory.

TEST INFRASTRUCTURE ONLY.  The tests and the CPU-baseline / reference leg of
the benchmark use it; the product path never does.

Optimizer shards are independent sub-problems ("SCAPE" arXiv 2607.01678,
Sec. II-A: the distributed optimizer partitions states and parameters evenly;
"Sintesi Tecnica: SCAPE" Sec. 2: each worker selects its mask only inside its
own partition): a shard's mask, packed values, synchronised buffer and update
depend only on that shard's slices of the W workers' gradients and on the
global step count.  So the oracle of a large problem can run shard by shard,
each shard in its own process, unchanged: every worker calls
``oracle.advance`` on its shard as an independent problem with one shard.

The caller fills each shard's gradient buffer (``grads(j)``, a [W, n] array
in shared memory, page-locked when a GPU is present so that device copies go
straight into it), then calls ``step()``; the workers advance in parallel and
leave the mask built after the step, its index list, the packed buffers and
the synchronised buffer in shared memory (``out(j)``).  ``dump()`` exposes
the final w, m and the chosen residual rows.

Processes are started with the ``spawn`` method, so the pool may be created
after the parent has used the GPU.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import time
from multiprocessing import shared_memory

import numpy as np

from . import oracle as O


def _nbytes(shape, dtype):
    return int(np.prod(shape, dtype=np.int64)) * np.dtype(dtype).itemsize


class _Block:
    """Named shared-memory arrays of one shard (created by the parent)."""

    def __init__(self, specs, create=True, names=None):
        self.specs = specs                      # {name: (shape, dtype)}
        self.shm = {}
        self.arr = {}
        for key, (shape, dtype) in specs.items():
            size = max(_nbytes(shape, dtype), 1)
            if create:
                sm = shared_memory.SharedMemory(create=True, size=size)
            else:
                sm = shared_memory.SharedMemory(name=names[key])
            self.shm[key] = sm
            self.arr[key] = np.ndarray(shape, dtype=dtype, buffer=sm.buf)

    def names(self):
        return {k: v.name for k, v in self.shm.items()}

    def close(self, unlink=False):
        self.arr.clear()
        for sm in self.shm.values():
            try:
                sm.close()
            except BufferError:
                pass
            if unlink:
                try:
                    sm.unlink()
                except FileNotFoundError:
                    pass
        self.shm.clear()


def _worker(conn, specs, names, W, k_s, hp, dump_rows):
    """Child process: one shard as an independent one-shard oracle problem."""
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    blk = _Block(specs, create=False, names=names)
    a = blk.arr
    n = a["w0"].shape[0]
    st = O.new_state(a["w0"], W, 0.0, hp, shard_start=np.array([0, n], np.int64),
                     shard_k=np.array([k_s], np.int64))
    try:
        while True:
            msg = conn.recv()
            if msg == "step":
                grads = [a["grads"][w] for w in range(W)]
                t0 = time.perf_counter()
                rec = O.advance(st, grads, keep=("bits", "idx", "pack", "gbar"))
                dt = time.perf_counter() - t0
                a["bits"][:] = rec["bits"]
                a["idx"][:] = rec["idx"]
                if rec["t"] >= 2:
                    a["pack"][:] = rec["pack"]
                    a["gbar"][:] = rec["gbar"]
                conn.send(dt)
            elif msg == "dump":
                a["w"][:] = st.w
                a["m"][:] = st.m
                for r, w in enumerate(dump_rows):
                    a["e"][r] = st.e[w]
                conn.send(0.0)
            else:
                break
    finally:
        blk.close()
        conn.close()


class ShardOracles:
    """Oracle workers for a list of shards of one problem.

    shards     list of (lo, hi, k_s): the shard's parameter range in the flat
               vector and its number of selected coordinates
    W          workers (gradient slices per shard)
    grad_dtype "bf16" (uint16 bit patterns) or "f32"
    w0         callable lo, hi -> float32 numpy array of the initial params
    dump_rows  which workers' residual rows dump() exposes
    pin        page-lock the gradient buffers for direct device copies
    """

    def __init__(self, shards, W, grad_dtype, hp, w0, dump_rows=(), pin=None):
        self.shards = [(int(lo), int(hi), int(k)) for lo, hi, k in shards]
        self.W = int(W)
        self.gdtype = np.uint16 if grad_dtype == "bf16" else np.float32
        self.dump_rows = tuple(int(w) for w in dump_rows)
        self.blocks, self.procs, self.conns = [], [], []
        self.pinned = []
        self.t = 0
        ctx = mp.get_context("spawn")
        try:
            for lo, hi, k in self.shards:
                n = hi - lo
                specs = {
                    "w0": ((n,), np.float32),
                    "grads": ((self.W, n), self.gdtype),
                    "bits": (((n + 31) // 32,), np.uint32),
                    "idx": ((k,), np.uint32),
                    "pack": ((self.W, k), np.float32),
                    "gbar": ((k,), np.float32),
                    "w": ((n,), np.float32),
                    "m": ((n,), np.float32),
                    "e": ((len(self.dump_rows), n), np.float32),
                }
                blk = _Block(specs)
                blk.arr["w0"][:] = w0(lo, hi)
                self.blocks.append(blk)
                parent, child = ctx.Pipe()
                p = ctx.Process(target=_worker,
                                args=(child, specs, blk.names(), self.W, k, hp, self.dump_rows),
                                daemon=True)
                p.start()
                child.close()
                self.procs.append(p)
                self.conns.append(parent)
            if pin is None:
                pin = _cuda_available()
            if pin:
                for blk in self.blocks:
                    self._pin(blk.arr["grads"])
        except BaseException:
            self.close()
            raise

    # ------------------------------------------------------------ inputs / outputs
    def grads(self, j):
        """[W, n] gradient buffer of shard j for the next step."""
        return self.blocks[j].arr["grads"]

    def out(self, j):
        """Results of shard j's last step: the mask built after it (bits of
        the shard in local coordinates, idx local), and for steps >= 2 the
        packed buffers [W, k_s] and the synchronised buffer [k_s]."""
        a = self.blocks[j].arr
        return {"bits": a["bits"], "idx": a["idx"], "pack": a["pack"], "gbar": a["gbar"]}

    def step(self):
        """Advance every shard one step in parallel; returns each worker's
        oracle time in seconds."""
        for c in self.conns:
            c.send("step")
        times = [c.recv() for c in self.conns]
        self.t += 1
        return times

    def dump(self):
        """Final w, m and the residual rows dump_rows of every shard."""
        for c in self.conns:
            c.send("dump")
        for c in self.conns:
            c.recv()
        return [{"w": b.arr["w"], "m": b.arr["m"], "e": b.arr["e"]} for b in self.blocks]

    # ------------------------------------------------------------ teardown
    def _pin(self, arr):
        import torch

        rt = torch.cuda.cudart()
        ptr = arr.ctypes.data
        if arr.nbytes and int(rt.cudaHostRegister(ptr, arr.nbytes, 0)) == 0:
            self.pinned.append(ptr)

    def close(self):
        for c in self.conns:
            try:
                c.send("stop")
            except (BrokenPipeError, OSError):
                pass
        for p in self.procs:
            p.join(timeout=30)
            if p.is_alive():
                p.kill()
        if self.pinned:
            import torch

            rt = torch.cuda.cudart()
            for ptr in self.pinned:
                rt.cudaHostUnregister(ptr)
            self.pinned = []
        for blk in self.blocks:
            blk.close(unlink=True)
        self.blocks, self.procs, self.conns = [], [], []

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


def _cuda_available():
    try:
        import torch

        return torch.cuda.is_available()
    except ImportError:
        return False

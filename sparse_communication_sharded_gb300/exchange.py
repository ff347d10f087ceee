"""SCAPE on several data-parallel ranks with a real exchange.

Each rank owns the workers and optimizer shards ``rank_shards(W, G, rank)``
("SCAPE" Sec. II-A: sharded data parallelism with a distributed optimizer): it
holds a full replica of the parameters, the first moment of its own parameter
range, and the full-length gradient and residual of each of its workers.  A
step is the library's four phases (scape_xc_pack / update / refresh / finish,
all kernels of libscape.so) around three torch.distributed collectives this
module issues on buffers inside the library's workspace:

* an all-to-all of the packed values (each owner receives every worker's
  selected values of its shards: the sparse reduce-scatter of "SCAPE"
  Sec. I, summed by the owner in worker order);
* an all-gather of the owners' updated parameters (the sparse parameter
  all-gather, "SCAPE" Sec. I);
* an all-gather of the owners' mask words ("Sintesi Tecnica: SCAPE" Sec. 2,
  partitioned mask), which may overlap the parameter all-gather: the mask is
  only used by the next step (the one-step lag).

With NCCL the collectives run on device memory, asynchronously, ordered with
the library's work on the current stream; with gloo (CPU) the buffers are
staged through host memory.  Only argument marshalling and the collectives
live here; every computation is a library kernel.
"""
from __future__ import annotations

from datetime import timedelta

import torch
import torch.distributed as dist

from . import _scape as C


class PeerLost(RuntimeError):
    """A rank of the group did not reach a step; the others stop before it,
    with none of the step's kernels or collectives launched."""

    def __init__(self, missing, step):
        self.missing = sorted(missing)
        self.step = step
        super().__init__(f"ranks {self.missing} did not reach step {step}")


def check_peers(store, rank, world, step, timeout=timedelta(seconds=30)):
    """Host-side liveness check before a step's first launch.  Every rank
    announces `step` in the store (any torch.distributed Store, e.g. the
    process group's) and waits at most `timeout` for the announcements of the
    others; a rank that has left (raised, exited, never joined) is named in
    the PeerLost raised on the others, before they launch anything."""
    key = "scape/alive/{}/{}".format
    store.set(key(step, rank), "1")
    others = [q for q in range(world) if q != rank]
    try:
        store.wait([key(step, q) for q in others], timeout)
    except RuntimeError as e:  # the store's timeout (DistStoreError is one)
        missing = [q for q in others if not store.check([key(step, q)])]
        if not missing:  # the wait failed for another reason
            raise
        raise PeerLost(missing, step) from e


def _ws_view(workspace, ptr, n, dtype):
    off = ptr - workspace.data_ptr()
    esz = torch.empty(0, dtype=dtype).element_size()
    return workspace[off:off + n * esz].view(dtype)


class ExchangeBuffers:
    """torch views of the exchange buffers of one handle (device memory)."""

    def __init__(self, h, workspace, G):
        self.h, self.workspace, self.G = h, workspace, G
        self.ptr = C.scape_xc_buffers(h)

    def counts(self):
        return C.scape_xc_counts(self.h, self.G)

    def view(self, name, n, dtype=torch.float32):
        return _ws_view(self.workspace, self.ptr[name], n, dtype)


def all_to_all(recv, send, recv_counts, send_counts, group=None, via_host=False):
    """Variable-size all-to-all of flat buffers (rank q's block of `send` goes
    to rank q; rank q's block arrives in `recv` at position q)."""
    if not dist.is_initialized():
        recv.copy_(send[:recv.numel()])  # one rank: its own block
        return None
    if via_host:
        r = torch.empty(recv.numel(), dtype=recv.dtype)
        dist.all_to_all_single(r, send.cpu(), recv_counts, send_counts, group=group)
        recv.copy_(r)
        return None
    return dist.all_to_all_single(recv, send, recv_counts, send_counts, group=group,
                                  async_op=True)


def all_gather_rows(out, row, G, group=None, via_host=False):
    """out (G rows of len(row)) receives every rank's `row`, rank q at row q."""
    n = row.numel()
    if not dist.is_initialized():
        out[:n].copy_(row)
        return None
    if via_host:
        parts = [torch.empty(n, dtype=row.dtype) for _ in range(G)]
        dist.all_gather(parts, row.cpu(), group=group)
        out.copy_(torch.cat(parts))
        return None
    return dist.all_gather([out[q * n:(q + 1) * n] for q in range(G)], row, group=group,
                           async_op=True)


class ScapeDP:
    """One rank of the exchange-based SCAPE step.

    params       float32 CUDA tensor of all P parameters (this rank's replica)
    W            workers = optimizer shards of the whole job
    layer_numel  the layer sizes (sum P); default one layer
    group        torch.distributed process group (default: the world)
    liveness     optional torch.distributed Store: before each step the ranks
                 check that all of them reached it (check_peers) and raise
                 PeerLost on the others if one has left; without it a rank
                 that has left shows as an error of the next collective once
                 the process group's timeout expires
    """

    def __init__(self, params: torch.Tensor, W: int, sparsity: float, *, layer_numel=None,
                 lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1,
                 grad_dtype=torch.bfloat16, group=None, liveness=None,
                 liveness_timeout=timedelta(seconds=30)):
        if not params.is_cuda or params.dtype != torch.float32 or not params.is_contiguous():
            raise ValueError("params must be a contiguous float32 CUDA tensor")
        self.group = group
        self.G = dist.get_world_size(group) if dist.is_initialized() else 1
        self.rank = dist.get_rank(group) if dist.is_initialized() else 0
        self.via_host = dist.is_initialized() and dist.get_backend(group) == "gloo"
        P = params.numel()
        layer_numel = [P] if layer_numel is None else list(layer_numel)
        dt = C.SCAPE_BF16 if grad_dtype == torch.bfloat16 else C.SCAPE_F32
        self.grad_dtype = grad_dtype
        self.h = C.scape_xc_create(layer_numel, W, self.G, self.rank, sparsity, beta1, beta2, lr,
                                   eps, weight_decay, dt)
        lay = C.scape_xc_layout(self.h)
        if lay["P"] != P:
            raise ValueError("layer sizes must sum to params.numel()")
        self.P, self.W, self.k = P, W, lay["k"]
        self.Wl = lay["local_workers"]
        self.own = (lay["own_begin"], lay["own_end"])
        dev = params.device
        self.params = params
        self.m = torch.zeros(self.own[1] - self.own[0], dtype=torch.float32, device=dev)
        stride = (P + 63) // 64 * 64
        self._e_storage = torch.zeros(max(self.Wl, 1) * stride, dtype=torch.float32, device=dev)
        self.e = [self._e_storage[w * stride:w * stride + P] for w in range(self.Wl)]
        self.workspace = torch.empty(lay["ws_bytes"], dtype=torch.uint8, device=dev)
        C.scape_xc_bind(self.h, params.data_ptr(), self.m.data_ptr(),
                        [x.data_ptr() for x in self.e], self.workspace.data_ptr(),
                        lay["ws_bytes"])
        self.buf = ExchangeBuffers(self.h, self.workspace, self.G)
        self.bytes_sent = 0
        # optional store for check_peers before every step
        self.liveness, self.liveness_timeout = liveness, liveness_timeout
        self.steps = 0

    @staticmethod
    def _stream():
        return torch.cuda.current_stream().cuda_stream

    def step(self, grads):
        """One step from the local workers' full-length gradients (b - a
        tensors of P elements); afterwards every rank's params hold the same
        updated parameters, and the mask of the next step is in place."""
        if len(grads) != self.Wl:
            raise ValueError(f"expected {self.Wl} local gradients")
        for g in grads:
            if g.dtype != self.grad_dtype or g.numel() != self.P or not g.is_cuda:
                raise ValueError("gradient dtype/size/device mismatch")
        if self.liveness is not None:
            check_peers(self.liveness, self.rank, self.G, self.steps, self.liveness_timeout)
        st = self._stream()
        cnt = self.buf.counts()
        G, b = self.G, self.buf
        C.scape_xc_pack(self.h, [g.data_ptr() for g in grads], st)
        send = b.view("send", sum(cnt["send"]))
        recv = b.view("recv", sum(cnt["recv"]))
        work = all_to_all(recv, send, cnt["recv"], cnt["send"], self.group, self.via_host)
        if work is not None:
            work.wait()
        C.scape_xc_update(self.h, st)
        ps, ms = cnt["param_stride"], cnt["mask_stride"]
        pwork = all_gather_rows(b.view("param_recv", G * ps), b.view("param_send", ps), G,
                                self.group, self.via_host)
        C.scape_xc_refresh(self.h, st)
        mwork = all_gather_rows(b.view("mask_recv", G * ms, torch.int32),
                                b.view("mask_send", ms, torch.int32), G, self.group,
                                self.via_host)
        for wk in (pwork, mwork):
            if wk is not None:
                wk.wait()
        C.scape_xc_finish(self.h, st)
        self.bytes_sent += 4 * (sum(cnt["send"]) + ps + ms)
        self.steps += 1

    # ----------------------------------------------------------- state views
    @property
    def t(self):
        return C.scape_xc_get_state(self.h)[0]

    def global_bits(self):
        """The global mask the next step uses (int32 view, ceil(P/32) words)."""
        return _ws_view(self.workspace, self.buf.ptr["global_bits"], (self.P + 31) // 32,
                        torch.int32)

    def get_state(self):
        """(t, a copy of the global mask the next step uses): with w, m and the
        residuals, what a checkpoint needs to resume."""
        return self.t, self.global_bits().clone()

    def set_state(self, t, global_bits):
        """Resume after t completed steps from a checkpoint's global mask (an
        int32 CUDA tensor of ceil(P/32) words, the same on every rank); w, m
        and the residuals are restored by the caller.  The next refresh of the
        owned shards is a cold one."""
        if not global_bits.is_cuda or global_bits.numel() != (self.P + 31) // 32:
            raise ValueError("global_bits must be a CUDA tensor of ceil(P/32) words")
        bits = global_bits.contiguous()
        C.scape_xc_set_state(self.h, t, bits.data_ptr(), self._stream())
        self.steps = int(t)

    def launch_count(self):
        return C.scape_xc_launch_count(self.h)

    def close(self):
        if getattr(self, "h", None) is not None:
            C.scape_xc_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

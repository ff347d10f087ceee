"""SCAPE optimizer over torch-allocated device memory.

PyTorch provides the device buffers (parameters, first moment, per-worker
residuals, workspace) and the stream; every computation is a kernel of
libscape.so reached through the C ABI.  W data-parallel workers are held as W
gradient tensors on one GPU.
"""
from __future__ import annotations

import torch

from . import _scape as C


class Scape:
    """One SCAPE instance bound to `params` (float32, CUDA, flat)."""

    def __init__(self, params: torch.Tensor, W: int, sparsity: float, *, layer_numel=None,
                 lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1,
                 grad_dtype=torch.bfloat16, residuals: str = "device", staging_rows=None,
                 shard_range=None):
        """residuals: "device" (HBM) or "host": the W error-feedback buffers
        live in pinned host memory (keeps W*P*4 bytes out of HBM).  With host
        residuals, staging_rows (default min(W, 12); 0 for none) residual rows
        of device memory stage them: sparse steps copy them in and out in
        worker groups, overlapped with the compaction; without staging the
        kernels read and write them in place over the host link.

        shard_range=(a, b): this instance covers only the optimizer shards
        [a, b) of the problem that layer_numel (the global layer sizes, then
        required) and W define; `params` is the slice [offset, offset + P)
        of the global parameters that those shards hold (see
        scape_create_range), and every gradient passed to step() is the same
        slice of that worker's gradient."""
        if not params.is_cuda or params.dtype != torch.float32 or not params.is_contiguous():
            raise ValueError("params must be a contiguous float32 CUDA tensor")
        P = params.numel()
        self.grad_dtype = grad_dtype
        dt = C.SCAPE_BF16 if grad_dtype == torch.bfloat16 else C.SCAPE_F32
        if grad_dtype not in (torch.bfloat16, torch.float32):
            raise ValueError("grad_dtype must be torch.bfloat16 or torch.float32")
        if shard_range is None:
            layer_numel = [P] if layer_numel is None else list(layer_numel)
            if sum(layer_numel) != P:
                raise ValueError("layer sizes must sum to params.numel()")
            self.h = C.scape_create(layer_numel, W, sparsity, beta1, beta2, lr, eps,
                                    weight_decay, dt)
        else:
            if layer_numel is None:
                raise ValueError("a shard range needs the global layer sizes")
            a, b = shard_range
            self.h = C.scape_create_range(list(layer_numel), W, a, b, sparsity, beta1, beta2, lr,
                                          eps, weight_decay, dt)
        rng = C.scape_get_range(self.h)
        self.P_global, self.offset = rng["P_global"], rng["offset"]
        self.shard_range = (rng["shard_begin"], rng["shard_end"])
        geo = C.scape_get_geometry(self.h)
        if geo["P"] != P:
            C.scape_destroy(self.h)
            self.h = None
            raise ValueError(f"params holds {P} elements; the shard range covers {geo['P']}")
        self.P, self.W, self.k = geo["P"], geo["W"], geo["k"]
        self.shard_start, self.shard_k = geo["shard_start"], geo["shard_k"]
        dev = params.device
        self.params = params
        self.m = torch.zeros(P, dtype=torch.float32, device=dev)
        if residuals == "device":
            # one allocation for all W residuals, rows 256-byte aligned: measured
            # faster for the compaction than W separate allocations (26.5 vs
            # 27.3 ms on the Llama-500M shape)
            stride = (P + 63) // 64 * 64
            self._e_storage = torch.zeros(W * stride, dtype=torch.float32, device=dev)
            self.e = [self._e_storage[w * stride:w * stride + P] for w in range(W)]
        elif residuals == "host":
            self.e = [torch.zeros(P, dtype=torch.float32).pin_memory() for _ in range(W)]
        else:
            raise ValueError('residuals must be "device" or "host"')
        self._lr = float(lr)
        self.ws_bytes = C.scape_workspace_bytes(self.h)
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        C.scape_bind(self.h, params.data_ptr(), self.m.data_ptr(), [x.data_ptr() for x in self.e],
                     self.workspace.data_ptr(), self.ws_bytes)
        self.staging = None
        if residuals == "host":
            rows = min(W, 12) if staging_rows is None else int(staging_rows)
            if rows:
                rows = max(rows, 3)
                nbytes = C.scape_residual_staging_bytes(self.h, rows)
                self.staging = torch.empty(nbytes, dtype=torch.uint8, device=dev)
                C.scape_set_residual_staging(self.h, self.staging.data_ptr(), nbytes)

    # ----------------------------------------------------------- hot path
    @staticmethod
    def _stream():
        return torch.cuda.current_stream().cuda_stream

    def step(self, grads):
        if len(grads) != self.W:
            raise ValueError(f"expected {self.W} gradients")
        for g in grads:
            if g.dtype != self.grad_dtype or g.numel() != self.P or not g.is_cuda:
                raise ValueError("gradient dtype/size/device mismatch")
        C.scape_step(self.h, [g.data_ptr() for g in grads], self._stream())

    def refresh_mask(self):
        C.scape_refresh_mask(self.h, self._stream())

    def step_host(self, host_grads, dev_grads, host_params_out):
        C.scape_step_host(self.h, [g.data_ptr() for g in host_grads],
                          [g.data_ptr() for g in dev_grads], host_params_out.data_ptr(),
                          self._stream())

    def set_variant(self, flags):
        C.scape_set_variant(self.h, flags)

    def set_fusion(self, level):
        """How much of the step the compaction pass does: C.FUSE_NONE (separate
        reduce and adams_sparse launches), C.FUSE_SUM (it writes g_bar) or
        C.FUSE_UPDATE (it also applies AdamS); results are bit-identical.  The
        default depends on the density (C.FUSE_UPDATE from 5% selected)."""
        C.scape_set_fusion(self.h, level)

    def fusion(self):
        """The current fusion level."""
        return C.scape_get_fusion(self.h)

    def dense_adams_step(self, grads):
        """Dense AdamS baseline on the mean gradient (no error feedback, no mask)."""
        C.scape_dense_adams_step(self.h, [g.data_ptr() for g in grads], self._stream())

    def adamw_step(self, grads, v: torch.Tensor):
        """Dense AdamW baseline; v is the caller's float32 second moment."""
        if v.dtype != torch.float32 or v.numel() != self.P or not v.is_cuda:
            raise ValueError("v must be a float32 CUDA tensor of P elements")
        C.scape_adamw_step(self.h, [g.data_ptr() for g in grads], v.data_ptr(), self._stream())

    def union_step(self, grads, capacity=None):
        """Union-mask gradient top-k baseline step; returns the union size.
        The workspace (packed buffers for `capacity` union positions, default
        P) is allocated on first use and kept."""
        cap = self.P if capacity is None else int(capacity)
        if getattr(self, "_union_cap", None) != cap:
            nbytes = C.scape_union_workspace_bytes(self.h, cap)
            self._union_ws = torch.empty(nbytes, dtype=torch.uint8, device=self.params.device)
            self._union_cap = cap
        return C.scape_union_step(self.h, [g.data_ptr() for g in grads],
                                  self._union_ws.data_ptr(), self._union_ws.numel(), cap,
                                  self._stream())

    def set_lr(self, lr):
        C.scape_set_lr(self.h, lr)
        self._lr = float(lr)

    def set_graphs(self, on):
        """Replay the steady warm mask refresh as a CUDA graph (default on)."""
        C.scape_set_graphs(self.h, on)

    # ----------------------------------------------------------- state views
    def _view(self, ptr, n, dtype):
        off = ptr - self.workspace.data_ptr()
        esz = torch.empty(0, dtype=dtype).element_size()
        return self.workspace[off:off + n * esz].view(dtype)

    @property
    def t(self):
        return C.scape_get_state(self.h)[0]

    def bits(self):
        _, _, bits, _ = C.scape_get_state(self.h)
        return self._view(bits, (self.P + 31) // 32, torch.int32)

    def idx(self):
        _, k, _, idx = C.scape_get_state(self.h)
        return self._view(idx, k, torch.int32)

    def pack(self):
        ptr, stride, _ = C.scape_get_buffers(self.h)
        full = self._view(ptr, stride * self.W, torch.float32).view(self.W, stride)
        return full[:, :self.k]

    def gbar(self):
        _, _, ptr = C.scape_get_buffers(self.h)
        return self._view(ptr, self.k, torch.float32)

    def set_state(self, t, bits: torch.Tensor):
        C.scape_set_state(self.h, t, bits.data_ptr(), self._stream())

    def state_dict(self):
        """What a resume needs besides the parameters, as copies: the steps
        taken, the mask the next step uses (take it after refresh_mask), the
        first moment, the W residuals and the learning rate."""
        t = self.t
        return {"t": t, "bits": self.bits().clone() if t >= 1 else None, "m": self.m.clone(),
                "e": [x.clone() for x in self.e], "lr": self._lr}

    def load_state_dict(self, sd):
        """Restore a state_dict() into this instance (same layout; the
        parameters are the caller's).  The next mask refresh is a cold one."""
        if len(sd["e"]) != self.W or sd["m"].numel() != self.P:
            raise ValueError("state_dict of another layout")
        self.m.copy_(sd["m"])
        for x, y in zip(self.e, sd["e"]):
            x.copy_(y)
        self.set_lr(sd["lr"])
        if sd["t"] >= 1:
            self.set_state(sd["t"], sd["bits"])

    # ----------------------------------------------------------- profiling
    def profile(self, on=True):
        C.scape_profile_enable(self.h, on)

    def profile_select(self, names_or_mask):
        """Bracket only these kernels (names or a bit mask) while profiling."""
        C.scape_profile_select(self.h, names_or_mask)

    def profile_collect(self):
        C.scape_profile_collect(self.h)

    def profile_read(self):
        return C.scape_profile_read(self.h)

    def profile_reset(self):
        C.scape_profile_reset(self.h)

    def launch_count(self):
        return C.scape_launch_count(self.h)

    def probe_random_access(self):
        """Timing probe: the sparse update's memory accesses without its
        arithmetic (w and m are left unchanged)."""
        C.scape_probe_random_access(self.h, self._stream())

    def close(self):
        if getattr(self, "h", None) is not None:
            C.scape_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

"""Seeded synthetic inputs for the SCAPE optimizer step: parameter-set shapes,
initial parameters and per-worker gradient streams.

This module holds no part of the optimizer's arithmetic.  It only draws random
numbers with the shapes, scales and structure of the workloads the SCAPE pages
train on (GPT-345M on OpenWebText, Llama-500M on SlimPajama-6B, Llama-1.8B:
"SCAPE" arXiv 2607.01678, abstract and Sec. I), which stand in for those
datasets: only the parameter shapes matter to the optimizer step.

Gradient model, per worker w and step t (one value per parameter):
    s_1 ~ N(0, 1),  s_t = rho * s_{t-1} + sqrt(1 - rho^2) * z_t       (shared, unit variance)
    g^w_t = c * (s_t + n^w_t)
with n^w_t ~ N(0, 1) (or Student-t with 3 degrees of freedom) and c the
per-element scale: 1e-3, or a per-layer log-uniform scale.  The flat sweep
quantises g to 256 levels of 2^-15 to force ties in |m|.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    layers: tuple                 # ((layer name, numel), ...) in flat-vector order
    W: int                        # simulated data-parallel workers (= optimizer shards)
    sparsity: float
    steps: int
    grad_dtype: str               # "bf16" or "f32"
    rho: float = 0.9
    sigma: float = 1e-3           # stationary std of the shared signal and of the noise
    noise: str = "gauss"          # "gauss" or "student_t3"
    layer_scale: tuple | None = None   # (lo, hi) log-uniform per-layer scale replacing sigma
    quantum: float | None = None       # quantisation step (256 levels) or None

    @property
    def P(self) -> int:
        return sum(n for _, n in self.layers)


def _gpt_layers(n_layer=24, h=1024, ffn=4096, vocab=50304, n_pos=1024):
    """GPT-2-style block: LN, fused QKV (+bias), proj (+bias), LN, fc1 (+bias),
    fc2 (+bias); tied embedding, learned positions, final LN."""
    out = [("wte", vocab * h), ("wpe", n_pos * h)]
    for i in range(n_layer):
        out.append((f"h{i}", 2 * h + 3 * h * h + 3 * h + h * h + h + 2 * h
                    + h * ffn + ffn + ffn * h + h))
    out.append(("ln_f", 2 * h))
    return tuple(out)


def _llama_layers(n_layer, h, ffn, vocab):
    """Llama block without biases: RMSNorm, q/k/v/o, RMSNorm, SwiGLU gate/up/down;
    untied input embedding and LM head, final RMSNorm."""
    out = [("embed", vocab * h)]
    for i in range(n_layer):
        out.append((f"layer{i}", 4 * h * h + 3 * h * ffn + 2 * h))
    out.append(("norm", h))
    out.append(("lm_head", vocab * h))
    return tuple(out)


WORKLOADS = {
    "tiny": Workload("tiny", (("flat", 4096),), W=4, sparsity=0.90, steps=10,
                     grad_dtype="f32"),
    "gpt345m": Workload("gpt345m", _gpt_layers(), W=8, sparsity=0.90, steps=20,
                        grad_dtype="bf16", layer_scale=(1e-4, 1e-2)),
    "llama500m": Workload("llama500m", _llama_layers(24, 1280, 3584, 32000), W=32,
                          sparsity=0.99, steps=20, grad_dtype="bf16"),
    "llama1p8b": Workload("llama1p8b", _llama_layers(24, 2048, 5632, 32000), W=8,
                          sparsity=0.99, steps=20, grad_dtype="bf16", rho=0.95,
                          noise="student_t3"),
}


def flat_workload(P: int, W: int, sparsity: float, steps: int = 5) -> Workload:
    """A point of the flat sweep: fp32 gradients quantised to 256 levels."""
    return Workload(f"flat_p{P}_w{W}_s{sparsity}", (("flat", P),), W=W,
                    sparsity=sparsity, steps=steps, grad_dtype="f32",
                    quantum=2.0 ** -15)


def init_params(P: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """Initial parameters ~ N(0, 0.02^2), float32."""
    g = torch.Generator(device=device).manual_seed(seed)
    return torch.randn(P, generator=g, device=device, dtype=torch.float32) * 0.02


class GradientStream:
    """Per-step, per-worker gradients of one workload, drawn on `device`.

    `next_into(bufs)` fills W caller-owned tensors (bf16 or f32, each P long)
    with the gradients of the next step.  Work is chunked so that temporary
    memory stays at a few chunk-sized float32 tensors."""

    CHUNK = 1 << 26

    def __init__(self, wl: Workload, seed: int = 0, device="cpu", P: int | None = None,
                 offset: int = 0):
        self.wl = wl
        self.device = torch.device(device)
        self.P = wl.P if P is None else P
        self.offset = offset
        self.gen = torch.Generator(device=self.device).manual_seed(seed + 1)
        self.t = 0
        self.s = None
        self.scale = self._scale(seed)

    @property
    def dtype(self):
        return torch.bfloat16 if self.wl.grad_dtype == "bf16" else torch.float32

    def _scale(self, seed):
        wl = self.wl
        if wl.layer_scale is None:
            return wl.sigma
        lo, hi = wl.layer_scale
        g = torch.Generator().manual_seed(seed + 7)
        u = torch.rand(len(wl.layers), generator=g, dtype=torch.float64)
        c = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))).to(torch.float32)
        sizes = torch.tensor([n for _, n in wl.layers])
        full = torch.repeat_interleave(c, sizes)
        return full[self.offset:self.offset + self.P].to(self.device)

    def _noise(self, n):
        z = torch.randn(n, generator=self.gen, device=self.device)
        if self.wl.noise == "student_t3":
            chi = torch.randn(3, n, generator=self.gen, device=self.device).square_().sum(0)
            z = z / torch.sqrt(chi / 3.0)
        return z

    def alloc(self):
        return [torch.empty(self.P, dtype=self.dtype, device=self.device)
                for _ in range(self.wl.W)]

    def next_into(self, bufs):
        wl = self.wl
        self.t += 1
        if self.s is None:
            self.s = torch.randn(self.P, generator=self.gen, device=self.device)
        else:
            a = math.sqrt(1.0 - wl.rho * wl.rho)
            for c0 in range(0, self.P, self.CHUNK):
                n = min(self.CHUNK, self.P - c0)
                z = torch.randn(n, generator=self.gen, device=self.device)
                self.s[c0:c0 + n].mul_(wl.rho).add_(z, alpha=a)
        for w in range(wl.W):
            for c0 in range(0, self.P, self.CHUNK):
                n = min(self.CHUNK, self.P - c0)
                x = self._noise(n).add_(self.s[c0:c0 + n])
                sc = self.scale if isinstance(self.scale, float) else self.scale[c0:c0 + n]
                x.mul_(sc)
                if wl.quantum is not None:
                    x.div_(wl.quantum).round_().clamp_(-128, 127).mul_(wl.quantum)
                bufs[w][c0:c0 + n].copy_(x)
        return bufs

    def next(self):
        return self.next_into(self.alloc())


def to_numpy_grad(t: torch.Tensor):
    """CPU numpy view of one gradient: float32, or uint16 bit patterns for bf16."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16").copy()
    return t.numpy().copy()

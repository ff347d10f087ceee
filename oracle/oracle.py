"""Python face of the plain CPU oracle of the SCAPE sharded optimizer step.

TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the CPU-baseline leg
of the benchmark may import this module; the product path (the CUDA library and
its binding) never does, and shares no code with it.

The arithmetic lives in ``scape_oracle.c`` (plain C, binary32 one operation at a
time, built with ``-O2 -ffp-contract=off``).  This module only marshals numpy
arrays and encodes the step order the pages give:

* the mask is refreshed from the first moment after step t and used at step
  t + 1 ("SCAPE" arXiv 2607.01678, Sec. I; "Sintesi Tecnica: SCAPE", Sec. 2,
  lagged mask use);
* step 1 runs with the mask of all ones (the pages say nothing about the first
  mask; with m_0 = 0 any top-k would be an arbitrary index-ordered prefix);
* the error-feedback residual, the packed buffers, their average and the
  AdamS update follow Sec. II-B and Sec. II-C (Eq. 2) of the SCAPE paper.

Gradients are numpy ``float32`` arrays, or ``uint16`` arrays holding bfloat16
bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "scape_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libscape_oracle.so")

F32 = 0
BF16 = 1

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C99, no contraction, no fast math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math",
                        "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        f32 = ctypes.c_float
        lib.oracle_layout.argtypes = [i64, i32, i64, vp, vp]
        lib.oracle_topk_mask.argtypes = [vp, i64, i32, vp, vp, vp, vp, vp]
        lib.oracle_step.argtypes = [i64, i64, i32, i32, vp, vp, vp, vp, vp, vp, i64,
                                    f32, f32, f32, f32, f32, vp, vp]
        lib.oracle_step_variant.argtypes = [i64, i64, i32, i32, vp, vp, vp, vp, vp, vp, i64,
                                            f32, f32, f32, f32, f32, i32, vp, vp]
        lib.oracle_dense_adams_step.argtypes = [i64, i64, i32, i32, vp, vp, vp,
                                                f32, f32, f32, f32, f32]
        lib.oracle_adamw_step.argtypes = [i64, i64, i32, i32, vp, vp, vp, vp,
                                          f32, f32, f32, f32, f32]
        lib.oracle_union_topk_step.argtypes = [i64, i64, i32, i32, vp, vp, vp, vp, i64,
                                               f32, f32, f32, f32, f32, vp, vp, vp, vp, vp]
        for fn in (lib.oracle_layout, lib.oracle_topk_mask, lib.oracle_step,
                   lib.oracle_step_variant, lib.oracle_dense_adams_step, lib.oracle_adamw_step,
                   lib.oracle_union_topk_step):
            fn.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def sparsity_ppm(sparsity: float) -> int:
    """Sparsity as an integer number of parts per million."""
    return int(round(float(sparsity) * 1e6))


def layout(P: int, W: int, sparsity: float):
    """Shard boundaries (W + 1 entries) and per-shard k (W entries)."""
    start = np.zeros(W + 1, np.int64)
    kk = np.zeros(W, np.int64)
    rc = _load().oracle_layout(P, W, sparsity_ppm(sparsity), _ptr(start), _ptr(kk))
    if rc != 0:
        raise ValueError(f"oracle_layout rejected P={P} W={W} sparsity={sparsity}")
    return start, kk


def topk_mask(m: np.ndarray, shard_start: np.ndarray, shard_k: np.ndarray):
    """Per-shard top-k of |m| (ties to the lower index) -> (bits uint32, idx uint32)."""
    m = np.ascontiguousarray(m, np.float32)
    P = m.size
    S = shard_k.size
    bits = np.zeros((P + 31) // 32, np.uint32)
    idx = np.zeros(max(int(shard_k.sum()), 1), np.uint32)
    k = np.zeros(1, np.int64)
    rc = _load().oracle_topk_mask(_ptr(m), P, S, _ptr(np.ascontiguousarray(shard_start, np.int64)),
                                  _ptr(np.ascontiguousarray(shard_k, np.int64)),
                                  _ptr(bits), _ptr(idx), _ptr(k))
    if rc != 0:
        raise ValueError("oracle_topk_mask failed")
    return bits, idx[: int(k[0])].copy()


@dataclass
class Hyper:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.95
    eps: float = 1e-8
    weight_decay: float = 0.1


def step(t: int, grads, e, w: np.ndarray, m: np.ndarray, bits: np.ndarray,
         idx: np.ndarray, hp: Hyper):
    """One step under the given mask.  Updates e (list of W arrays), w and m in
    place; returns (pack [W, k] float32, gbar [k] float32)."""
    W = len(grads)
    P = w.size
    dtype = BF16 if grads[0].dtype == np.uint16 else F32
    for g in grads:
        assert g.size == P and g.dtype == (np.uint16 if dtype == BF16 else np.float32)
    k = idx.size
    pack = np.zeros((W, max(k, 1)), np.float32)
    gbar = np.zeros(max(k, 1), np.float32)
    gp = (ctypes.c_void_p * W)(*[_ptr(g) for g in grads])
    ep = (ctypes.c_void_p * W)(*[_ptr(x) for x in e])
    rc = _load().oracle_step(t, P, W, dtype, ctypes.addressof(gp), ctypes.addressof(ep),
                             _ptr(w), _ptr(m), _ptr(bits), _ptr(idx), k,
                             hp.beta1, hp.beta2, hp.lr, hp.eps, hp.weight_decay,
                             _ptr(pack), _ptr(gbar))
    if rc != 0:
        raise ValueError("oracle_step failed")
    return pack[:, :k], gbar[:k]


# variant readings (flags, combinable)
DENSE_OFFMASK = 1   # unselected coordinates take the AdamS update with a zero gradient
MOMENT_SYNC = 2     # the synchronised buffer holds first moments; g is recovered from it


def step_variant(t: int, grads, e, w, m, bits, idx, hp: Hyper, variant: int):
    """step() under a variant reading; returns (pack, synchronised buffer)."""
    W = len(grads)
    P = w.size
    dtype = BF16 if grads[0].dtype == np.uint16 else F32
    k = idx.size
    pack = np.zeros((W, max(k, 1)), np.float32)
    gbar = np.zeros(max(k, 1), np.float32)
    gp = (ctypes.c_void_p * W)(*[_ptr(g) for g in grads])
    ep = (ctypes.c_void_p * W)(*[_ptr(x) for x in e])
    rc = _load().oracle_step_variant(t, P, W, dtype, ctypes.addressof(gp), ctypes.addressof(ep),
                                     _ptr(w), _ptr(m), _ptr(bits), _ptr(idx), k,
                                     hp.beta1, hp.beta2, hp.lr, hp.eps, hp.weight_decay,
                                     int(variant), _ptr(pack), _ptr(gbar))
    if rc != 0:
        raise ValueError("oracle_step_variant failed")
    return pack[:, :k], gbar[:k]


def dense_adams_step(t: int, grads, w, m, hp: Hyper):
    """Dense AdamS on the plain mean of the workers' gradients (no error feedback)."""
    W = len(grads)
    dtype = BF16 if grads[0].dtype == np.uint16 else F32
    gp = (ctypes.c_void_p * W)(*[_ptr(g) for g in grads])
    rc = _load().oracle_dense_adams_step(t, w.size, W, dtype, ctypes.addressof(gp), _ptr(w),
                                         _ptr(m), hp.beta1, hp.beta2, hp.lr, hp.eps,
                                         hp.weight_decay)
    if rc != 0:
        raise ValueError("oracle_dense_adams_step failed")


def adamw_step(t: int, grads, w, m, v, hp: Hyper):
    """Dense AdamW (EMA second moment) on the plain mean of the gradients."""
    W = len(grads)
    dtype = BF16 if grads[0].dtype == np.uint16 else F32
    gp = (ctypes.c_void_p * W)(*[_ptr(g) for g in grads])
    rc = _load().oracle_adamw_step(t, w.size, W, dtype, ctypes.addressof(gp), _ptr(w), _ptr(m),
                                   _ptr(v), hp.beta1, hp.beta2, hp.lr, hp.eps, hp.weight_decay)
    if rc != 0:
        raise ValueError("oracle_adamw_step failed")


def union_k_worker(P: int, sparsity: float) -> int:
    """Coordinates each worker selects over the whole vector (same rounding as
    the shards' k)."""
    ppm = sparsity_ppm(sparsity)
    return (P * (1000000 - ppm) + 999999) // 1000000


def union_topk_step(t: int, grads, e, w, m, k_worker: int, hp: Hyper):
    """Gradient top-k with error feedback and a union mask.  Updates e, w, m
    in place; returns (union bits, idx, pack [W, k_union], gbar)."""
    W = len(grads)
    P = w.size
    dtype = BF16 if grads[0].dtype == np.uint16 else F32
    bits = np.zeros((P + 31) // 32, np.uint32)
    idx = np.zeros(P, np.uint32)
    ku = np.zeros(1, np.int64)
    pack = np.zeros(W * P, np.float32)
    gbar = np.zeros(P, np.float32)
    gp = (ctypes.c_void_p * W)(*[_ptr(g) for g in grads])
    ep = (ctypes.c_void_p * W)(*[_ptr(x) for x in e])
    rc = _load().oracle_union_topk_step(t, P, W, dtype, ctypes.addressof(gp), ctypes.addressof(ep),
                                        _ptr(w), _ptr(m), int(k_worker), hp.beta1, hp.beta2,
                                        hp.lr, hp.eps, hp.weight_decay, _ptr(bits), _ptr(idx),
                                        _ptr(ku), _ptr(pack), _ptr(gbar))
    if rc != 0:
        raise ValueError("oracle_union_topk_step failed")
    k = int(ku[0])
    return bits, idx[:k].copy(), pack[:W * k].reshape(W, k).copy(), gbar[:k].copy()


def dense_mask(P: int):
    """The all-ones mask of step 1 and its index list."""
    bits = np.full((P + 31) // 32, 0xFFFFFFFF, np.uint32)
    if P % 32:
        bits[-1] = np.uint32((1 << (P % 32)) - 1)
    return bits, np.arange(P, dtype=np.uint32)


@dataclass
class State:
    """Optimizer state of one SCAPE instance on the CPU."""
    w: np.ndarray
    m: np.ndarray
    e: list
    shard_start: np.ndarray
    shard_k: np.ndarray
    hp: Hyper
    t: int = 0
    bits: np.ndarray | None = None   # mask to be used by the next step (None: dense)
    idx: np.ndarray | None = None
    history: list = field(default_factory=list)


def new_state(w0: np.ndarray, W: int, sparsity: float, hp: Hyper,
              shard_start=None, shard_k=None) -> State:
    P = w0.size
    if shard_start is None:
        shard_start, shard_k = layout(P, W, sparsity)
    return State(w=np.array(w0, np.float32, copy=True), m=np.zeros(P, np.float32),
                 e=[np.zeros(P, np.float32) for _ in range(W)],
                 shard_start=shard_start, shard_k=shard_k, hp=hp)


def advance(st: State, grads, keep=None, variant: int = 0) -> dict:
    """Step t+1 with the lagged mask, then refresh the mask from the new m."""
    t = st.t + 1
    if st.bits is None:
        used_bits, used_idx = dense_mask(st.w.size)
    else:
        used_bits, used_idx = st.bits, st.idx
    if variant:
        pack, gbar = step_variant(t, grads, st.e, st.w, st.m, used_bits, used_idx, st.hp, variant)
    else:
        pack, gbar = step(t, grads, st.e, st.w, st.m, used_bits, used_idx, st.hp)
    st.t = t
    st.bits, st.idx = topk_mask(st.m, st.shard_start, st.shard_k)
    rec = {"t": t, "used_bits": used_bits, "used_idx": used_idx, "pack": pack,
           "gbar": gbar, "bits": st.bits, "idx": st.idx}
    if keep is None:
        return rec
    return {k: v for k, v in rec.items() if k in keep or k == "t"}

"""ctypes binding of the SCAPE C ABI (include/scape.h): argument marshalling only.

Every step of the optimizer runs in the CUDA kernels of libscape.so; this module
converts Python ints, lists and torch tensors into the pointers and sizes the
C functions take.  Loading fails loudly when the library has not been built:
there is no Python or CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

SCAPE_OK = 0
SCAPE_EINVAL = -1
SCAPE_ECUDA = -2
SCAPE_ESTATE = -4
SCAPE_F32 = 0
SCAPE_BF16 = 1
SCAPE_MAX_WORKERS = 256
SCAPE_NUM_KERNELS = 25

LIB_PATH = _build.LIB


class ScapeError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"SCAPE error {code}: {msg}")
        self.code = code


_lib = None

_vp, _i64, _i32, _f32, _f64 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                               ctypes.c_double)
_PROTOS = {
    "scape_create": (_i32, [ctypes.POINTER(_vp), _i32, _vp, _i32, _f64, _f32, _f32, _f32, _f32,
                            _f32, _i32]),
    "scape_create_range": (_i32, [ctypes.POINTER(_vp), _i32, _vp, _i32, _i32, _i32, _f64, _f32,
                                  _f32, _f32, _f32, _f32, _i32]),
    "scape_get_range": (_i32, [_vp, _vp, _vp, _vp, _vp]),
    "scape_destroy": (None, [_vp]),
    "scape_last_error": (ctypes.c_char_p, [_vp]),
    "scape_get_geometry": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp]),
    "scape_workspace_bytes": (_i32, [_vp, _vp]),
    "scape_bind": (_i32, [_vp, _vp, _vp, _vp, _vp, ctypes.c_size_t]),
    "scape_step": (_i32, [_vp, _vp, _vp]),
    "scape_refresh_mask": (_i32, [_vp, _vp]),
    "scape_set_lr": (_i32, [_vp, _f32]),
    "scape_set_graphs": (_i32, [_vp, _i32]),
    "scape_set_variant": (_i32, [_vp, _i32]),
    "scape_set_fusion": (_i32, [_vp, _i32]),
    "scape_get_fusion": (_i32, [_vp, _vp]),
    "scape_residual_staging_bytes": (_i32, [_vp, _i32, ctypes.POINTER(ctypes.c_size_t)]),
    "scape_set_residual_staging": (_i32, [_vp, _vp, ctypes.c_size_t]),
    "scape_dense_adams_step": (_i32, [_vp, _vp, _vp]),
    "scape_union_workspace_bytes": (_i32, [_vp, _i64, _vp]),
    "scape_union_step": (_i32, [_vp, _vp, _vp, ctypes.c_size_t, _i64, _vp, _vp]),
    "scape_adamw_step": (_i32, [_vp, _vp, _vp, _vp]),
    "scape_get_state": (_i32, [_vp, _vp, _vp, _vp, _vp]),
    "scape_get_buffers": (_i32, [_vp, _vp, _vp, _vp]),
    "scape_set_state": (_i32, [_vp, _i64, _vp, _vp]),
    "scape_step_host": (_i32, [_vp, _vp, _vp, _vp, _vp]),
    "scape_profile_enable": (_i32, [_vp, _i32]),
    "scape_profile_select": (_i32, [_vp, ctypes.c_uint32]),
    "scape_profile_collect": (_i32, [_vp]),
    "scape_profile_read": (_i32, [_vp, _vp, _vp]),
    "scape_profile_reset": (_i32, [_vp]),
    "scape_kernel_name": (ctypes.c_char_p, [_i32]),
    "scape_launch_count": (_i64, [_vp]),
    "scape_topk_mask_static": (_i32, [_vp, _i64, _i32, _f64, _vp, _vp, _vp]),
    "scape_probe_random_access": (_i32, [_vp, _vp]),
    "scape_xc_create": (_i32, [ctypes.POINTER(_vp), _i32, _vp, _i32, _i32, _i32, _f64, _f32, _f32,
                               _f32, _f32, _f32, _i32]),
    "scape_xc_destroy": (None, [_vp]),
    "scape_xc_last_error": (ctypes.c_char_p, [_vp]),
    "scape_xc_layout": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "scape_xc_bind": (_i32, [_vp, _vp, _vp, _vp, _vp, ctypes.c_size_t]),
    "scape_xc_counts": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "scape_xc_buffers": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "scape_xc_pack": (_i32, [_vp, _vp, _vp]),
    "scape_xc_update": (_i32, [_vp, _vp]),
    "scape_xc_refresh": (_i32, [_vp, _vp]),
    "scape_xc_finish": (_i32, [_vp, _vp]),
    "scape_xc_get_state": (_i32, [_vp, _vp, _vp, _vp]),
    "scape_xc_set_state": (_i32, [_vp, _i64, _vp, _vp]),
    "scape_xc_launch_count": (_i64, [_vp]),
}


def load(path: str = LIB_PATH):
    """Load libscape.so; raises if it is missing (build it first)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise ImportError(f"libscape.so not found at {path}: build it with "
                              "`python -m sparse_communication_sharded_gb300.build`")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _PROTOS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def exported_symbols():
    return list(_PROTOS)


def _check(h, rc):
    if rc != SCAPE_OK:
        msg = load().scape_last_error(h)
        raise ScapeError(rc, msg.decode() if msg else "")
    return rc


def _ptr_array(ptrs):
    arr = (ctypes.c_void_p * len(ptrs))(*[int(p) for p in ptrs])
    return arr


# --------------------------------------------------------------- C ABI mirror
def scape_create(layer_numel, W, sparsity, beta1, beta2, lr, eps, weight_decay, grad_dtype):
    lib = load()
    sizes = (ctypes.c_int64 * len(layer_numel))(*[int(n) for n in layer_numel])
    h = ctypes.c_void_p()
    rc = lib.scape_create(ctypes.byref(h), len(layer_numel), ctypes.addressof(sizes), int(W),
                          float(sparsity), beta1, beta2, lr, eps, weight_decay, int(grad_dtype))
    if rc != SCAPE_OK:
        raise ScapeError(rc, lib.scape_last_error(None).decode())
    return h


def scape_create_range(layer_numel, W, shard_begin, shard_end, sparsity, beta1, beta2, lr, eps,
                       weight_decay, grad_dtype):
    lib = load()
    sizes = (ctypes.c_int64 * len(layer_numel))(*[int(n) for n in layer_numel])
    h = ctypes.c_void_p()
    rc = lib.scape_create_range(ctypes.byref(h), len(layer_numel), ctypes.addressof(sizes), int(W),
                                int(shard_begin), int(shard_end), float(sparsity), beta1, beta2,
                                lr, eps, weight_decay, int(grad_dtype))
    if rc != SCAPE_OK:
        raise ScapeError(rc, lib.scape_last_error(None).decode())
    return h


def scape_get_range(h):
    Pg, off = ctypes.c_int64(), ctypes.c_int64()
    a, b = ctypes.c_int(), ctypes.c_int()
    _check(h, load().scape_get_range(h, ctypes.byref(Pg), ctypes.byref(off), ctypes.byref(a),
                                     ctypes.byref(b)))
    return {"P_global": Pg.value, "offset": off.value, "shard_begin": a.value,
            "shard_end": b.value}


def scape_destroy(h):
    load().scape_destroy(h)


def scape_last_error(h):
    return load().scape_last_error(h).decode()


def scape_get_geometry(h):
    P, W, k = ctypes.c_int64(), ctypes.c_int(), ctypes.c_int64()
    _check(h, load().scape_get_geometry(h, ctypes.byref(P), ctypes.byref(W), ctypes.byref(k),
                                        None, None))
    S = scape_get_range(h)["shard_end"] - scape_get_range(h)["shard_begin"]
    start = (ctypes.c_int64 * (S + 1))()
    ks = (ctypes.c_int64 * S)()
    _check(h, load().scape_get_geometry(h, None, None, None, ctypes.addressof(start),
                                        ctypes.addressof(ks)))
    return {"P": P.value, "W": W.value, "k": k.value, "shard_start": list(start),
            "shard_k": list(ks)}


def scape_workspace_bytes(h):
    n = ctypes.c_size_t()
    _check(h, load().scape_workspace_bytes(h, ctypes.byref(n)))
    return n.value


def scape_bind(h, params_ptr, m_ptr, e_ptrs, ws_ptr, ws_bytes):
    arr = _ptr_array(e_ptrs)
    _check(h, load().scape_bind(h, params_ptr, m_ptr, ctypes.addressof(arr), ws_ptr, ws_bytes))


def scape_step(h, grad_ptrs, stream=0):
    arr = _ptr_array(grad_ptrs)
    _check(h, load().scape_step(h, ctypes.addressof(arr), stream))


def scape_refresh_mask(h, stream=0):
    _check(h, load().scape_refresh_mask(h, stream))


SCAPE_VARIANT_PAPER = 0
SCAPE_VARIANT_DENSE_OFFMASK = 1
SCAPE_VARIANT_MOMENT_SYNC = 2


def scape_set_variant(h, flags):
    _check(h, load().scape_set_variant(h, int(flags)))


FUSE_NONE, FUSE_SUM, FUSE_UPDATE = 0, 1, 2


def scape_set_fusion(h, level):
    _check(h, load().scape_set_fusion(h, int(level)))


def scape_get_fusion(h):
    level = ctypes.c_int(0)
    _check(h, load().scape_get_fusion(h, ctypes.byref(level)))
    return level.value


def scape_residual_staging_bytes(h, rows):
    n = ctypes.c_size_t(0)
    _check(h, load().scape_residual_staging_bytes(h, int(rows), ctypes.byref(n)))
    return n.value


def scape_set_residual_staging(h, ptr, nbytes):
    _check(h, load().scape_set_residual_staging(h, ptr, int(nbytes)))


def scape_dense_adams_step(h, grad_ptrs, stream=0):
    arr = _ptr_array(grad_ptrs)
    _check(h, load().scape_dense_adams_step(h, ctypes.addressof(arr), stream))


def scape_adamw_step(h, grad_ptrs, v_ptr, stream=0):
    arr = _ptr_array(grad_ptrs)
    _check(h, load().scape_adamw_step(h, ctypes.addressof(arr), v_ptr, stream))


def scape_union_workspace_bytes(h, capacity):
    n = ctypes.c_size_t()
    _check(h, load().scape_union_workspace_bytes(h, int(capacity), ctypes.byref(n)))
    return n.value


def scape_union_step(h, grad_ptrs, ws_ptr, ws_bytes, capacity, stream=0):
    arr = _ptr_array(grad_ptrs)
    ku = ctypes.c_int64()
    _check(h, load().scape_union_step(h, ctypes.addressof(arr), ws_ptr, ws_bytes, int(capacity),
                                      ctypes.byref(ku), stream))
    return ku.value


def scape_set_graphs(h, on):
    _check(h, load().scape_set_graphs(h, 1 if on else 0))


def scape_set_lr(h, lr):
    _check(h, load().scape_set_lr(h, lr))


def scape_get_state(h):
    t, k = ctypes.c_int64(), ctypes.c_int64()
    bits, idx = ctypes.c_void_p(), ctypes.c_void_p()
    _check(h, load().scape_get_state(h, ctypes.byref(t), ctypes.byref(k), ctypes.byref(bits),
                                     ctypes.byref(idx)))
    return t.value, k.value, bits.value, idx.value


def scape_get_buffers(h):
    pack, stride, gbar = ctypes.c_void_p(), ctypes.c_int64(), ctypes.c_void_p()
    _check(h, load().scape_get_buffers(h, ctypes.byref(pack), ctypes.byref(stride),
                                       ctypes.byref(gbar)))
    return pack.value, stride.value, gbar.value


def scape_set_state(h, t, bits_ptr, stream=0):
    _check(h, load().scape_set_state(h, int(t), bits_ptr, stream))


def scape_step_host(h, host_src_ptrs, dev_grad_ptrs, host_params_out_ptr, stream=0):
    a = _ptr_array(host_src_ptrs)
    b = _ptr_array(dev_grad_ptrs)
    _check(h, load().scape_step_host(h, ctypes.addressof(a), ctypes.addressof(b),
                                     host_params_out_ptr, stream))


def scape_profile_enable(h, on=True):
    _check(h, load().scape_profile_enable(h, 1 if on else 0))


def scape_profile_select(h, names_or_mask):
    """Profile only some kernels: a bit mask, or an iterable of kernel names."""
    if isinstance(names_or_mask, int):
        mask = names_or_mask
    else:
        ids = {scape_kernel_name(i): i for i in range(SCAPE_NUM_KERNELS)}
        mask = 0
        for n in names_or_mask:
            mask |= 1 << ids[n]
    _check(h, load().scape_profile_select(h, mask & 0xFFFFFFFF))


def scape_profile_collect(h):
    _check(h, load().scape_profile_collect(h))


def scape_profile_read(h):
    ms = (ctypes.c_double * SCAPE_NUM_KERNELS)()
    n = (ctypes.c_int64 * SCAPE_NUM_KERNELS)()
    _check(h, load().scape_profile_read(h, ctypes.addressof(ms), ctypes.addressof(n)))
    lib = load()
    return {lib.scape_kernel_name(i).decode(): (ms[i], n[i]) for i in range(SCAPE_NUM_KERNELS)}


def scape_profile_reset(h):
    _check(h, load().scape_profile_reset(h))


def scape_kernel_name(i):
    return load().scape_kernel_name(i).decode()


def scape_launch_count(h):
    return load().scape_launch_count(h)


def scape_probe_random_access(h, stream=0):
    _check(h, load().scape_probe_random_access(h, stream))


SCAPE_STATIC_MAX_P = 1 << 26
SCAPE_STATIC_MAX_WORKERS = 64


def scape_topk_mask_static(m_ptr, P, W, sparsity, bits_ptr, idx_ptr, stream=0):
    """Allocation-free per-shard top-k mask; returns the status code."""
    return load().scape_topk_mask_static(m_ptr, int(P), int(W), float(sparsity), bits_ptr,
                                         idx_ptr, stream)


# ------------------------------------------------------------ several ranks, real exchange
def _xcheck(h, rc):
    if rc != SCAPE_OK:
        msg = load().scape_xc_last_error(h)
        raise ScapeError(rc, msg.decode() if msg else "")
    return rc


def scape_xc_create(layer_numel, W, G, rank, sparsity, beta1, beta2, lr, eps, weight_decay,
                    grad_dtype):
    lib = load()
    sizes = (ctypes.c_int64 * len(layer_numel))(*[int(n) for n in layer_numel])
    h = ctypes.c_void_p()
    rc = lib.scape_xc_create(ctypes.byref(h), len(layer_numel), ctypes.addressof(sizes), int(W),
                             int(G), int(rank), float(sparsity), beta1, beta2, lr, eps,
                             weight_decay, int(grad_dtype))
    if rc != SCAPE_OK:
        raise ScapeError(rc, lib.scape_xc_last_error(None).decode())
    return h


def scape_xc_destroy(h):
    load().scape_xc_destroy(h)


def scape_xc_layout(h):
    P, k, own_b, own_e, own_k = (ctypes.c_int64() for _ in range(5))
    wl = ctypes.c_int()
    ws = ctypes.c_size_t()
    _xcheck(h, load().scape_xc_layout(h, ctypes.byref(P), ctypes.byref(k), ctypes.byref(wl),
                                      ctypes.byref(own_b), ctypes.byref(own_e),
                                      ctypes.byref(own_k), ctypes.byref(ws)))
    return {"P": P.value, "k": k.value, "local_workers": wl.value, "own_begin": own_b.value,
            "own_end": own_e.value, "own_k": own_k.value, "ws_bytes": ws.value}


def scape_xc_bind(h, params_ptr, m_ptr, e_ptrs, ws_ptr, ws_bytes):
    arr = _ptr_array(e_ptrs)
    _xcheck(h, load().scape_xc_bind(h, params_ptr, m_ptr, ctypes.addressof(arr), ws_ptr,
                                    ws_bytes))


def scape_xc_counts(h, G):
    sc = (ctypes.c_int64 * G)()
    rcv = (ctypes.c_int64 * G)()
    ppr = (ctypes.c_int64 * G)()
    mwr = (ctypes.c_int64 * G)()
    ps, ms = ctypes.c_int64(), ctypes.c_int64()
    _xcheck(h, load().scape_xc_counts(h, ctypes.addressof(sc), ctypes.addressof(rcv),
                                      ctypes.addressof(ppr), ctypes.byref(ps),
                                      ctypes.addressof(mwr), ctypes.byref(ms)))
    return {"send": list(sc), "recv": list(rcv), "params": list(ppr), "param_stride": ps.value,
            "mask_words": list(mwr), "mask_stride": ms.value}


def scape_xc_buffers(h):
    ptrs = [ctypes.c_void_p() for _ in range(7)]
    _xcheck(h, load().scape_xc_buffers(h, *[ctypes.byref(p) for p in ptrs]))
    names = ("send", "recv", "param_send", "param_recv", "mask_send", "mask_recv", "global_bits")
    return {n: p.value for n, p in zip(names, ptrs)}


def scape_xc_pack(h, grad_ptrs, stream=0):
    arr = _ptr_array(grad_ptrs)
    _xcheck(h, load().scape_xc_pack(h, ctypes.addressof(arr), stream))


def scape_xc_update(h, stream=0):
    _xcheck(h, load().scape_xc_update(h, stream))


def scape_xc_refresh(h, stream=0):
    _xcheck(h, load().scape_xc_refresh(h, stream))


def scape_xc_finish(h, stream=0):
    _xcheck(h, load().scape_xc_finish(h, stream))


def scape_xc_get_state(h):
    t = ctypes.c_int64()
    bits, idx = ctypes.c_void_p(), ctypes.c_void_p()
    _xcheck(h, load().scape_xc_get_state(h, ctypes.byref(t), ctypes.byref(bits),
                                         ctypes.byref(idx)))
    return t.value, bits.value, idx.value


def scape_xc_set_state(h, t, global_bits_ptr, stream=0):
    _xcheck(h, load().scape_xc_set_state(h, int(t), global_bits_ptr, stream))


def scape_xc_launch_count(h):
    return load().scape_xc_launch_count(h)

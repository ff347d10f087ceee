"""The C-ABI library loads on a host without a GPU, exports every entry point
include/scape.h declares, and its host-only logic (argument validation, shard
layout, k, workspace size, call-order errors) behaves -- no GPU work is done."""
import ctypes
import os
import re

import numpy as np
import pytest

from oracle import oracle as O
from sparse_communication_sharded_gb300 import _scape as C
from sparse_communication_sharded_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return C.load()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(scape_\w+)\s*\(", txt))
    return names


def test_every_declared_symbol_is_exported(lib):
    declared = _declared()
    assert len(declared) >= 19
    for name in declared:
        assert hasattr(lib, name), name
    assert declared == set(C.exported_symbols())


def _create(P=4096, W=4, s=0.9, beta1=0.9, beta2=0.95, lr=1e-3, eps=1e-8, wd=0.1, dt=C.SCAPE_F32):
    return C.scape_create([P] if isinstance(P, int) else P, W, s, beta1, beta2, lr, eps, wd, dt)


@pytest.mark.parametrize("kw", [dict(P=0), dict(W=0), dict(W=C.SCAPE_MAX_WORKERS + 1),
                                dict(s=1.0), dict(s=-0.1), dict(s=0.9999999), dict(beta1=1.0),
                                dict(beta2=-0.5), dict(eps=0.0), dict(wd=-1.0), dict(dt=7),
                                dict(lr=float("nan")), dict(P=[1 << 30, 1 << 30, 1 << 30])])
def test_create_rejects_bad_arguments(lib, kw):
    with pytest.raises(C.ScapeError) as ei:
        _create(**kw)
    assert ei.value.code == C.SCAPE_EINVAL
    assert C.scape_last_error(None) != ""


@pytest.mark.parametrize("P,W,s", [(4096, 4, 0.9), (569570560, 32, 0.99), (354871296, 8, 0.9),
                                   (1364297728, 8, 0.99), (5, 8, 0.5), (1 << 20, 32, 0.999),
                                   (1000, 7, 0.0)])
def test_geometry_matches_oracle_layout(lib, P, W, s):
    h = _create(P=P, W=W, s=s)
    geo = C.scape_get_geometry(h)
    start, ks = O.layout(P, W, s)
    assert geo["shard_start"] == start.tolist()
    assert geo["shard_k"] == ks.tolist()
    assert geo["k"] == int(ks.sum()) and geo["P"] == P and geo["W"] == W
    ws = C.scape_workspace_bytes(h)
    # the W packed buffers dominate the workspace
    assert ws >= 4 * W * geo["k"] + 4 * geo["k"] + (P + 31) // 32 * 4
    C.scape_destroy(h)


def test_layers_concatenate(lib):
    h = C.scape_create([10, 0, 30], 2, 0.5, 0.9, 0.95, 1e-3, 1e-8, 0.1, C.SCAPE_BF16)
    assert C.scape_get_geometry(h)["P"] == 40
    C.scape_destroy(h)


def test_call_order_errors_without_gpu(lib):
    h = _create()
    with pytest.raises(C.ScapeError) as ei:
        C.scape_step(h, [0] * 4)
    assert ei.value.code == C.SCAPE_ESTATE
    with pytest.raises(C.ScapeError) as ei:
        C.scape_refresh_mask(h)
    assert ei.value.code == C.SCAPE_ESTATE
    with pytest.raises(C.ScapeError) as ei:
        C.scape_bind(h, 0, 0, [0] * 4, 0, 0)
    assert ei.value.code == C.SCAPE_EINVAL
    with pytest.raises(C.ScapeError) as ei:
        C.scape_get_buffers(h)
    assert ei.value.code == C.SCAPE_ESTATE
    with pytest.raises(C.ScapeError):
        C.scape_set_lr(h, float("inf"))
    C.scape_set_lr(h, 5e-4)
    t, k, bits, idx = C.scape_get_state(h)
    assert t == 0 and k == 412 and bits is None and idx is None
    assert C.scape_launch_count(h) == 0
    C.scape_destroy(h)


def test_bind_validates_before_any_cuda_call(lib):
    h = _create()
    ws = C.scape_workspace_bytes(h)
    with pytest.raises(C.ScapeError) as ei:        # workspace too small
        C.scape_bind(h, 256, 512, [1024] * 4, 4096, ws - 1)
    assert ei.value.code == C.SCAPE_EINVAL
    with pytest.raises(C.ScapeError) as ei:        # misaligned workspace
        C.scape_bind(h, 256, 512, [1024] * 4, 4096 + 8, ws)
    assert ei.value.code == C.SCAPE_EINVAL
    with pytest.raises(C.ScapeError) as ei:        # misaligned residual
        C.scape_bind(h, 256, 512, [1024, 1028, 2048, 4096], 8192, ws)
    assert ei.value.code == C.SCAPE_EINVAL
    C.scape_destroy(h)


def test_kernel_names(lib):
    names = [C.scape_kernel_name(i) for i in range(C.SCAPE_NUM_KERNELS)]
    assert len(set(names)) == C.SCAPE_NUM_KERNELS and all(names)
    assert C.scape_kernel_name(C.SCAPE_NUM_KERNELS) == ""


def test_missing_library_fails_loudly(lib, monkeypatch):
    monkeypatch.setattr(C, "_lib", None)
    with pytest.raises(ImportError):
        C.load("/nonexistent/libscape.so")


def test_fusion_and_staging_validate_without_gpu(lib):
    h = _create(P=10000, W=8)
    for level in (C.FUSE_NONE, C.FUSE_SUM, C.FUSE_UPDATE):
        C.scape_set_fusion(h, level)
    with pytest.raises(C.ScapeError) as ei:
        C.scape_set_fusion(h, 3)
    assert ei.value.code == C.SCAPE_EINVAL
    # rows are P rounded up to 64 floats
    assert C.scape_residual_staging_bytes(h, 3) == 3 * 10048 * 4
    with pytest.raises(C.ScapeError):
        C.scape_residual_staging_bytes(h, 2)
    with pytest.raises(C.ScapeError) as ei:        # fewer than three rows
        C.scape_set_residual_staging(h, 4096, 2 * 10048 * 4)
    assert ei.value.code == C.SCAPE_EINVAL
    with pytest.raises(C.ScapeError) as ei:        # misaligned
        C.scape_set_residual_staging(h, 4100, 3 * 10048 * 4)
    assert ei.value.code == C.SCAPE_EINVAL
    C.scape_set_residual_staging(h, 4096, 5 * 10048 * 4)
    C.scape_set_residual_staging(h, None, 0)       # back to in place
    C.scape_destroy(h)


@pytest.mark.parametrize("P,W,s,want", [(4096, 4, 0.9, C.FUSE_UPDATE), (4096, 4, 0.99, C.FUSE_SUM),
                                        (4096, 4, 0.0, C.FUSE_SUM), (354871296, 8, 0.9, C.FUSE_UPDATE),
                                        (569570560, 32, 0.99, C.FUSE_SUM),
                                        (1364297728, 8, 0.99, C.FUSE_SUM), (100000, 3, 0.95, C.FUSE_UPDATE),
                                        (100000, 3, 0.96, C.FUSE_SUM), (4096, 1, 0.99, C.FUSE_UPDATE),
                                        (4096, 2, 0.999, C.FUSE_SUM), (4096, 3, 0.99, C.FUSE_SUM),
                                        (1 << 20, 1, 0.0, C.FUSE_SUM)])
def test_default_fusion_follows_density(lib, P, W, s, want):
    """The update goes into the compaction pass from 5% of the coordinates
    selected (20 k >= P; 0.5% with one or two workers), except when every
    coordinate is kept."""
    h = _create(P=P, W=W, s=s)
    k = C.scape_get_geometry(h)["k"]
    fused = 20 * k >= P or (W <= 2 and 200 * k >= P)
    assert (fused and k < P) == (want == C.FUSE_UPDATE)
    assert C.scape_get_fusion(h) == want
    C.scape_set_fusion(h, C.FUSE_NONE)
    assert C.scape_get_fusion(h) == C.FUSE_NONE
    C.scape_destroy(h)


def test_mask_churn_counts_changed_coordinates():
    import torch
    import bench
    a = torch.tensor([0b1011, 0, -1], dtype=torch.int32)     # 3 + 0 + 32 set bits
    assert bench.mask_churn(a, a.clone(), 35) == 0.0
    b = torch.tensor([0b0111, 0, -1], dtype=torch.int32)     # one bit moved
    assert bench.mask_churn(a, b, 35) == 2 / 70
    c = torch.tensor([0, -1, 0], dtype=torch.int32)          # disjoint, 32 set
    assert abs(bench.mask_churn(torch.tensor([0, 0, -1], dtype=torch.int32), c, 32) - 1.0) < 1e-12


def test_algorithmic_bytes_per_step():
    """The per-step byte counts the roofline uses: the sum of each kernel's
    algorithmic bytes; level "none" adds the packed buffers' re-read."""
    import bench
    from sparse_communication_sharded_gb300 import synth
    want = {"gpt345m": (32.21, 33.35), "llama500m": (185.67, 186.40), "llama1p8b": (115.99, 116.43)}
    for name, (gb_sum, gb_none) in want.items():
        wl = synth.WORKLOADS[name]
        _, ks = O.layout(wl.P, wl.W, wl.sparsity)
        k = int(ks.sum())
        a = bench.algorithmic_bytes(wl, k, "sum")
        b = bench.algorithmic_bytes(wl, k, "none")
        assert abs(a["total"] / 1e9 - gb_sum) < 0.01, name
        assert abs(b["total"] / 1e9 - gb_none) < 0.01, name
        assert abs((b["total"] - a["total"]) - 4 * k * wl.W) < 1e-3
        # the compaction dominates the step's bytes (92% at GPT-345M's 10%
        # density, 98.6% at Llama-500M's 1%)
        assert a["ef_compact"] / a["total"] > 0.9

"""The allocation-free mask entry point, scape_topk_mask_static().

It serves callers that cannot call cudaMalloc where they need a mask (code
inside a custom allocator or memory-pool callback, plug-ins handed only their
input and output buffers, loops that cannot take cudaMalloc's implicit device
synchronisation): its scratch is a fixed array inside the library.  These
tests call it through the C ABI twice in a row, on different first moments,
and check each result against the workspace-based scape_refresh_mask() on the
same m and against the CPU oracle's per-shard top-k: the mask and the packed
index list must match exactly (integer outputs, the bar every mask test here
uses).  They also check that a call allocates no device memory.  The file is
collected last so that a run stopping at the first failure has already run
every other test."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from sparse_communication_sharded_gb300 import _scape as C
from tests._harness import make_opt, u32

pytestmark = pytest.mark.gpu


def _reference_mask(dev, m, W, s):
    """Mask and index list from the existing entry point (scape_refresh_mask)."""
    P = m.numel()
    opt = make_opt(torch.zeros(P, device=dev), W, s, torch.float32)
    opt.step([torch.zeros(P, device=dev) for _ in range(W)])
    opt.m.copy_(m)
    opt.refresh_mask()
    torch.cuda.synchronize()
    out = u32(opt.bits()), u32(opt.idx()), opt.k
    opt.close()
    return out


def _static_mask(dev, m, W, s, k):
    P = m.numel()
    bits = torch.full(((P + 31) // 32,), -1, dtype=torch.int32, device=dev)
    idx = torch.full((max(k, 1),), -1, dtype=torch.int32, device=dev)
    rc = C.scape_topk_mask_static(m.data_ptr(), P, W, s, bits.data_ptr(), idx.data_ptr(),
                                  torch.cuda.current_stream().cuda_stream)
    assert rc == C.SCAPE_OK
    torch.cuda.synchronize()
    return u32(bits), u32(idx)[:k]


def _values(kind, gen, P, dev):
    if kind == "gauss":
        return torch.randn(P, device=dev, generator=gen) * 1e-3
    if kind == "levels":      # 256 levels: heavy ties, decided by the index order
        return torch.randint(-128, 128, (P,), device=dev, generator=gen).float() * 2.0 ** -15
    if kind == "signed_zero":  # +0 and -0 are equal keys; a few nonzero values
        z = torch.where(torch.rand(P, device=dev, generator=gen) < 0.5, -0.0, 0.0)
        hot = torch.rand(P, device=dev, generator=gen) < 0.003
        return torch.where(hot, torch.randn(P, device=dev, generator=gen), z)
    raise ValueError(kind)


@pytest.mark.parametrize("P,W,s", [(1_000_003, 8, 0.99), (300_000, 64, 0.9), (4096, 4, 0.999),
                                   (4097, 4, 0.0), (37, 64, 0.9), (2_000_001, 3, 0.5)])
@pytest.mark.parametrize("kinds", [("gauss", "levels"), ("signed_zero", "gauss")])
def test_static_mask_matches_workspace_path_and_oracle_twice(cuda_device, P, W, s, kinds):
    """Two calls in a row (the second on different values, so stale scratch
    would show); sparsity 0 takes the all-kept branch, P < W gives empty
    shards, odd P a ragged last tile."""
    gen = torch.Generator(device=cuda_device).manual_seed(P + W)
    start, ks = O.layout(P, W, s)
    for kind in kinds:
        m = _values(kind, gen, P, cuda_device)
        want_bits, want_idx, k = _reference_mask(cuda_device, m, W, s)
        got_bits, got_idx = _static_mask(cuda_device, m, W, s, k)
        assert np.array_equal(got_bits, want_bits), kind
        assert np.array_equal(got_idx, want_idx), kind
        o_bits, o_idx = O.topk_mask(m.cpu().numpy(), start, ks)
        assert np.array_equal(got_bits, o_bits), kind
        assert np.array_equal(got_idx, o_idx.view(np.uint32)), kind


def test_static_mask_allocates_nothing(cuda_device):
    """After a first call (which looks up the scratch array's address), further
    calls leave the device's free memory and PyTorch's allocator untouched."""
    P, W, s = 3_000_017, 16, 0.99
    gen = torch.Generator(device=cuda_device).manual_seed(5)
    m = _values("gauss", gen, P, cuda_device)
    _, ks = O.layout(P, W, s)
    k = int(ks.sum())
    bits = torch.empty((P + 31) // 32, dtype=torch.int32, device=cuda_device)
    idx = torch.empty(k, dtype=torch.int32, device=cuda_device)
    stream = torch.cuda.current_stream().cuda_stream

    def call():
        return C.scape_topk_mask_static(m.data_ptr(), P, W, s, bits.data_ptr(), idx.data_ptr(),
                                        stream)

    assert call() == C.SCAPE_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_stats().get("num_alloc_retries", 0), torch.cuda.memory_allocated()
    for _ in range(3):
        assert call() == C.SCAPE_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    alloc1 = torch.cuda.memory_stats().get("num_alloc_retries", 0), torch.cuda.memory_allocated()
    assert free1 == free0
    assert alloc1 == alloc0


def test_static_mask_rejects_sizes_beyond_limits(cuda_device):
    m = torch.zeros(16, device=cuda_device)
    out = torch.zeros(16, dtype=torch.int32, device=cuda_device)
    stream = torch.cuda.current_stream().cuda_stream
    for P, W in ((C.SCAPE_STATIC_MAX_P + 1, 8), (16, C.SCAPE_STATIC_MAX_WORKERS + 1), (0, 1)):
        rc = C.scape_topk_mask_static(m.data_ptr(), P, W, 0.9, out.data_ptr(), out.data_ptr(),
                                      stream)
        assert rc == C.SCAPE_EINVAL

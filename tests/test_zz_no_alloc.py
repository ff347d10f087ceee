"""The allocation-free mask entry point, scape_topk_mask_static().

It serves callers that cannot call cudaMalloc where they need a mask (code
inside a custom allocator or memory-pool callback, plug-ins handed only their
input and output buffers, loops that cannot take cudaMalloc's implicit device
synchronisation): its scratch is a fixed array inside the library.  This test
calls it through the C ABI twice in a row, on different first moments, and
checks each result against the workspace-based scape_refresh_mask() on the same
m: the mask and the packed index list must match exactly (integer outputs, the
bar every mask test here uses).  It sits in a file collected last so that a
run stopping at the first failure has already run every other test."""
import numpy as np
import pytest
import torch

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


@pytest.mark.parametrize("P,W,s", [(1_000_003, 8, 0.99), (300_000, 64, 0.9), (4096, 4, 0.999)])
def test_static_mask_matches_workspace_path_twice(cuda_device, P, W, s):
    gen = torch.Generator(device=cuda_device).manual_seed(P)
    ms = [torch.randn(P, device=cuda_device, generator=gen) * 1e-3,
          # second call: 256-level values (heavy ties) so stale scratch would show
          torch.randint(-128, 128, (P,), device=cuda_device, generator=gen).float() * 2.0 ** -15]
    for m in ms:
        want_bits, want_idx, k = _reference_mask(cuda_device, m, W, s)
        bits = torch.full(((P + 31) // 32,), -1, dtype=torch.int32, device=cuda_device)
        idx = torch.full((k,), -1, dtype=torch.int32, device=cuda_device)
        rc = C.scape_topk_mask_static(m.data_ptr(), P, W, s, bits.data_ptr(), idx.data_ptr(),
                                      torch.cuda.current_stream().cuda_stream)
        assert rc == C.SCAPE_OK
        torch.cuda.synchronize()
        assert np.array_equal(u32(bits), want_bits)
        assert np.array_equal(u32(idx), want_idx)


def test_static_mask_rejects_sizes_beyond_limits(cuda_device):
    m = torch.zeros(16, device=cuda_device)
    out = torch.zeros(16, dtype=torch.int32, device=cuda_device)
    stream = torch.cuda.current_stream().cuda_stream
    for P, W in ((C.SCAPE_STATIC_MAX_P + 1, 8), (16, C.SCAPE_STATIC_MAX_WORKERS + 1), (0, 1)):
        rc = C.scape_topk_mask_static(m.data_ptr(), P, W, 0.9, out.data_ptr(), out.data_ptr(),
                                      stream)
        assert rc == C.SCAPE_EINVAL

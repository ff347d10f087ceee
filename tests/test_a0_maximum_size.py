"""The largest problem the library accepts, P = 2^31 - 1, checked on the GPU by
properties that hold at any size (the oracle's sort is too slow there).

This module is collected first (its name sorts first), so that it runs on a
fresh device before any other test has left memory in PyTorch's cache; it
needs about 80 GB and fails, reporting the free memory, rather than skipping.
"""
import pytest
import torch

from sparse_communication_sharded_gb300 import synth
from tests._harness import make_opt

pytestmark = pytest.mark.gpu


def test_maximum_size_properties(cuda_device):
    """P = 2^31 - 1 (the largest accepted), W = 2: too large for the oracle's
    sort, so check what must hold at any size, on the GPU: every shard's mask
    holds exactly k_s coordinates, every selected key beats every unselected one
    (ties to the lower index), the packed buffers are fl(g + e) at the selected
    positions in ascending order, sent + residual == fl(g + e), and unselected
    w and m do not move."""
    P, W, s = (1 << 31) - 1, 2, 0.99
    torch.cuda.empty_cache()
    free, total = torch.cuda.mem_get_info()
    assert free >= 80 << 30, (f"needs ~80 GB of free device memory, {free / 2**30:.1f} GiB of "
                              f"{total / 2**30:.1f} GiB free")
    wl = synth.Workload("max", (("flat", P),), W=W, sparsity=s, steps=2, grad_dtype="bf16")
    gen = synth.GradientStream(wl, seed=12, device=cuda_device)
    params = synth.init_params(P, seed=12, device=cuda_device)
    opt = make_opt(params, W, s, torch.bfloat16)
    bufs = gen.alloc()
    gen.next_into(bufs)
    opt.step(bufs)
    opt.refresh_mask()
    torch.cuda.synchronize()
    # mask: exact k_s per shard and the threshold order
    words = opt.bits()
    sel = ((words.view(-1, 1) >> torch.arange(32, device=cuda_device, dtype=torch.int32))
           & 1).view(-1)[:P].bool()
    keys = opt.m.view(torch.int32) & 0x7FFFFFFF
    for sh in range(W):
        lo, hi = opt.shard_start[sh], opt.shard_start[sh + 1]
        ss, kk = sel[lo:hi], keys[lo:hi]
        assert int(ss.sum()) == opt.shard_k[sh]
        kmin = int(kk[ss].min())
        assert int(kk[~ss].max()) <= kmin
        ties_sel = torch.nonzero(ss & (kk == kmin)).flatten()
        ties_uns = torch.nonzero(~ss & (kk == kmin)).flatten()
        if ties_uns.numel():
            assert int(ties_sel.max()) < int(ties_uns.min())
    del sel, keys
    # one sparse step: compaction, conservation and off-mask invariance at samples
    idx = opt.idx().long()
    e_before = [x.clone() for x in opt.e]
    w_before, m_before = params.clone(), opt.m.clone()
    gen.next_into(bufs)
    opt.step(bufs)
    torch.cuda.synchronize()
    gsel = torch.Generator(device=cuda_device).manual_seed(0)
    js = torch.randint(0, opt.k, (100000,), device=cuda_device, generator=gsel)
    js = torch.cat([js, torch.tensor([0, opt.k - 1], device=cuda_device)])
    ii = idx[js]
    for w in range(W):
        a = bufs[w][ii].float() + e_before[w][ii]
        assert torch.equal(opt.pack()[w][js].view(torch.int32), a.view(torch.int32))
        assert bool((opt.e[w][ii] == 0).all())
    pos = torch.randint(0, P, (200000,), device=cuda_device, generator=gsel)
    pos = torch.cat([pos, torch.tensor([P - 1, P - 2, 0], device=cuda_device)])
    wb = opt.bits()
    unsel = ((wb[pos >> 5] >> (pos & 31).int()) & 1) == 0
    pu = pos[unsel]
    for w in range(W):
        a = bufs[w][pu].float() + e_before[w][pu]
        assert torch.equal(opt.e[w][pu].view(torch.int32), a.view(torch.int32))
    assert torch.equal(params[pu].view(torch.int32), w_before[pu].view(torch.int32))
    assert torch.equal(opt.m[pu].view(torch.int32), m_before[pu].view(torch.int32))
    opt.close()
    del bufs, e_before
    torch.cuda.empty_cache()

"""GPU parity of shard-range handles (scape_create_range): each handle covers
a block of optimizer shards of one problem and steps the slices of all W
workers' gradients there.  Shards are independent ("SCAPE" Sec. II-A, even
partition of the optimizer; "Sintesi Tecnica: SCAPE" Sec. 2, the mask of each
partition is computed from that partition alone), so every handle of a
partition of the shards must reproduce, slice by slice and bit for bit, the
CPU oracle's whole-problem trajectory: the mask bits and index list of its
range, its columns of the packed buffers and of the synchronised buffer at
every step, and w, m and every residual row at the end."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from sparse_communication_sharded_gb300 import Scape, synth
from tests._harness import HP, Report, local_words, u32

pytestmark = pytest.mark.gpu


CASES = [
    # (P, W, sparsity, grad dtype, quantised, shard ranges)
    (100003, 8, 0.99, "bf16", False, [(0, 3), (3, 8)]),
    (70001, 5, 0.9, "f32", False, [(0, 1), (1, 2), (2, 5)]),
    (50000, 32, 0.999, "f32", True, [(0, 7), (7, 32)]),
    (33333, 7, 0.99, "f32", True, [(3, 4), (0, 3), (4, 7)]),
    (6001, 3, 0.0, "bf16", False, [(0, 2), (2, 3)]),
    (20, 8, 0.5, "f32", False, [(0, 5), (5, 8)]),
]


@pytest.mark.parametrize("P,W,s,dtype,quant,ranges", CASES)
def test_range_handles_reproduce_whole_problem(cuda_device, P, W, s, dtype, quant, ranges):
    wl = synth.Workload(f"p{P}", (("flat", P),), W=W, sparsity=s, steps=8, grad_dtype=dtype,
                        quantum=2.0 ** -15 if quant else None)
    gdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    w0 = synth.init_params(P, seed=6)
    gen = synth.GradientStream(wl, seed=6, device="cpu")
    st = O.new_state(w0.numpy(), W, s, HP)
    start, ks = O.layout(P, W, s)
    kofs = np.concatenate([[0], np.cumsum(ks)])
    opts = []
    for a, b in ranges:
        lo, hi = int(start[a]), int(start[b])
        params = w0[lo:hi].clone().to(cuda_device)
        opt = Scape(params, W, s, layer_numel=[P], shard_range=(a, b), lr=HP.lr,
                    beta1=HP.beta1, beta2=HP.beta2, eps=HP.eps, weight_decay=HP.weight_decay,
                    grad_dtype=gdt)
        assert (opt.offset, opt.P, opt.P_global) == (lo, hi - lo, P)
        assert opt.k == int(ks[a:b].sum())
        opts.append((opt, params, lo, hi, a, b))
    rep = Report(f"range handles P={P} W={W} s={s} {ranges}")
    for t in range(1, 9):
        grads = gen.next()
        for opt, _, lo, hi, _, _ in opts:
            opt.step([g[lo:hi].to(cuda_device) for g in grads])
            opt.refresh_mask()
        rec = O.advance(st, [synth.to_numpy_grad(g) for g in grads])
        torch.cuda.synchronize()
        for opt, _, lo, hi, a, b in opts:
            k0, k1 = kofs[a], kofs[b]
            if t >= 2:
                rep.note(np.array_equal(u32(opt.pack()), rec["pack"][:, k0:k1].view(np.uint32)))
                rep.note(np.array_equal(u32(opt.gbar()), rec["gbar"][k0:k1].view(np.uint32)))
            want = local_words(rec["bits"], lo, hi)
            got = u32(opt.bits())
            rep.mask_bits += hi - lo
            rep.flips += int(np.unpackbits((got ^ want).view(np.uint8)).sum())
            rep.note(np.array_equal(got, want))
            rep.note(np.array_equal(u32(opt.idx()), rec["idx"][k0:k1] - np.uint32(lo)))
    for opt, params, lo, hi, _, _ in opts:
        rep.note(np.array_equal(u32(params), st.w[lo:hi].view(np.uint32)))
        rep.note(np.array_equal(u32(opt.m), st.m[lo:hi].view(np.uint32)))
        for w in range(W):
            rep.note(np.array_equal(u32(opt.e[w]), st.e[w][lo:hi].view(np.uint32)))
        opt.close()
    assert rep.exact, f"{rep.flips} mask flips"


def test_range_handle_rejects_a_wrong_slice(cuda_device):
    with pytest.raises(ValueError):
        Scape(torch.zeros(10, device=cuda_device), 4, 0.9, layer_numel=[100], shard_range=(0, 1),
              grad_dtype=torch.float32)
    with pytest.raises(ValueError):
        Scape(torch.zeros(25, device=cuda_device), 4, 0.9, shard_range=(0, 1),
              grad_dtype=torch.float32)

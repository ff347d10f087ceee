"""Helpers for the GPU parity tests: run the CUDA path and the CPU oracle on the
same seeded inputs and compare them."""
from __future__ import annotations

import numpy as np
import torch

from oracle import oracle as O
from sparse_communication_sharded_gb300 import Scape, synth

HP = O.Hyper(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
RTOL, ATOL = 1e-5, 1e-7          # float states after the trajectory
MAX_FLIP_FRACTION = 1e-4         # threshold-boundary mask flips


def u32(t: torch.Tensor) -> np.ndarray:
    a = t.detach().cpu().contiguous().numpy()
    return a.view(np.uint32)


def bits_to_bool(bits: np.ndarray, lo: int, hi: int) -> np.ndarray:
    i = np.arange(lo, hi)
    return ((bits[i // 32] >> (i % 32).astype(np.uint32)) & 1).astype(bool)


def make_opt(params, W, s, grad_dtype, **kw):
    return Scape(params, W, s, lr=HP.lr, beta1=HP.beta1, beta2=HP.beta2, eps=HP.eps,
                 weight_decay=HP.weight_decay, grad_dtype=grad_dtype, **kw)


def assert_close_f32(got: np.ndarray, want: np.ndarray, what: str):
    got = np.asarray(got, np.float32)
    want = np.asarray(want, np.float32)
    bad = ~np.isclose(got, want, rtol=RTOL, atol=ATOL)
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside rtol={RTOL} atol={ATOL}; "
                           f"max abs diff {np.abs(got - want).max():.3e}")


# every Report made during the session, for the flip-fraction summary that
# conftest.py prints at the end of the run
REPORTS = []


class Report:
    """Per-run parity facts the tests assert on and print: whether every
    compared value was bit-identical, and how many mask bits differ from the
    oracle's (threshold-boundary flips) out of how many compared."""

    def __init__(self, name=""):
        self.name = name
        self.flips = 0
        self.mask_bits = 0
        self.exact = True
        REPORTS.append(self)

    def note(self, equal: bool):
        self.exact = self.exact and bool(equal)

    @property
    def flip_fraction(self):
        return self.flips / self.mask_bits if self.mask_bits else 0.0


_POPC8 = np.array([bin(v).count("1") for v in range(256)], np.int64)


def popcount(words: np.ndarray) -> int:
    return int(_POPC8[np.ascontiguousarray(words).view(np.uint8)].sum())


def local_words(g: np.ndarray, lo: int, hi: int) -> np.ndarray:
    """Bits [lo, hi) of the global bitmap g (uint32 words) as a bitmap of their
    own starting at bit 0, with the bits past hi - lo cleared."""
    n = hi - lo
    nw = (n + 31) // 32
    w0, sh = lo // 32, lo % 32
    a = g[w0:w0 + nw].astype(np.uint64)
    b = np.zeros(nw, np.uint64)
    nxt = g[w0 + 1:w0 + 1 + nw].astype(np.uint64)
    b[:nxt.size] = nxt
    out = (((a >> np.uint64(sh)) | (b << np.uint64(32 - sh))) & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    if n % 32:
        out[-1] &= np.uint32((1 << (n % 32)) - 1)
    return out


def run_full_trajectory(wl: synth.Workload, device, steps: int, seed: int = 0,
                        grad_offset_elems: int = 0, variant: int = 0, fusion=None,
                        graphs=None):
    """Whole problem on both sides (small sizes): compare every step."""
    P, W, s = wl.P, wl.W, wl.sparsity
    gdt = torch.bfloat16 if wl.grad_dtype == "bf16" else torch.float32
    w0 = synth.init_params(P, seed=seed)
    gen = synth.GradientStream(wl, seed=seed, device="cpu")
    params = w0.to(device)
    opt = make_opt(params, W, s, gdt)
    if variant:
        opt.set_variant(variant)
    if fusion is not None:
        opt.set_fusion(fusion)
    if graphs is not None:
        opt.set_graphs(graphs)
    st = O.new_state(w0.numpy(), W, s, HP)
    rep = Report(f"{wl.name} W={W} s={s} x {steps} steps")
    # optional misaligned gradient buffers (scalar path)
    dev_bufs = [torch.empty(P + grad_offset_elems, dtype=gdt, device=device) for _ in range(W)]
    for t in range(1, steps + 1):
        grads = gen.next()
        dg = []
        for buf, g in zip(dev_bufs, grads):
            view = buf[grad_offset_elems:grad_offset_elems + P]
            view.copy_(g.to(device))
            dg.append(view)
        opt.step(dg)
        rec = O.advance(st, [synth.to_numpy_grad(g) for g in grads], variant=variant)
        if t >= 2:
            torch.cuda.synchronize()
            pack = u32(opt.pack())
            gbar = u32(opt.gbar())
            assert pack.shape == rec["pack"].shape
            rep.note(np.array_equal(pack, rec["pack"].view(np.uint32)))
            rep.note(np.array_equal(gbar, rec["gbar"].view(np.uint32)))
        opt.refresh_mask()
        torch.cuda.synchronize()
        gb = u32(opt.bits())
        flips = int(np.unpackbits((gb ^ rec["bits"]).view(np.uint8)).sum())
        rep.flips += flips
        rep.mask_bits += P
        if flips == 0:
            assert np.array_equal(u32(opt.idx()), rec["idx"].view(np.uint32)), "idx mismatch"
        rep.note(flips == 0)
    torch.cuda.synchronize()
    assert_close_f32(params.cpu().numpy(), st.w, "w")
    assert_close_f32(opt.m.cpu().numpy(), st.m, "m")
    for w in range(W):
        assert_close_f32(opt.e[w].cpu().numpy(), st.e[w], f"e[{w}]")
    rep.note(np.array_equal(u32(params), st.w.view(np.uint32)))
    rep.note(np.array_equal(u32(opt.m), st.m.view(np.uint32)))
    for w in range(W):
        rep.note(np.array_equal(u32(opt.e[w]), st.e[w].view(np.uint32)))
    assert rep.flips <= MAX_FLIP_FRACTION * rep.mask_bits, f"{rep.flips} mask flips"
    opt.close()
    return rep


def run_sampled_shards(wl: synth.Workload, device, steps: int, shards, seed: int = 0,
                       fusion=None):
    """Full-size problem on the GPU; the oracle runs each sampled shard as an
    independent sub-problem (shards share nothing but the step count), one
    process per shard in parallel (oracle.pool).  Every step compares the
    shard's mask bits, index list, packed buffers and synchronised buffer; the
    end compares w, m and the first and last workers' residuals."""
    from oracle.pool import ShardOracles

    P, W, s = wl.P, wl.W, wl.sparsity
    gdt = torch.bfloat16 if wl.grad_dtype == "bf16" else torch.float32
    w0 = synth.init_params(P, seed=seed, device=device)
    gen = synth.GradientStream(wl, seed=seed, device=device)
    params = w0.clone()
    opt = make_opt(params, W, s, gdt)
    if fusion is not None:
        opt.set_fusion(fusion)
    start, ks = opt.shard_start, opt.shard_k
    kofs = np.concatenate([[0], np.cumsum(ks)])
    spec = [(start[sh], start[sh + 1], ks[sh]) for sh in shards]
    rep = Report(f"{wl.name} shards {tuple(shards)} x {steps} steps")
    with ShardOracles(spec, W, wl.grad_dtype, HP, lambda lo, hi: w0[lo:hi].cpu().numpy(),
                      dump_rows=(0, W - 1)) as pool:
        del w0
        bufs = gen.alloc()
        for t in range(1, steps + 1):
            gen.next_into(bufs)
            for j, (lo, hi, _) in enumerate(spec):
                host = torch.from_numpy(pool.grads(j).view(
                    np.int16 if wl.grad_dtype == "bf16" else np.float32))
                for w in range(W):
                    src = bufs[w][lo:hi]
                    host[w].copy_(src.view(torch.int16) if wl.grad_dtype == "bf16" else src,
                                  non_blocking=True)
            opt.step(bufs)
            opt.refresh_mask()
            torch.cuda.synchronize()
            pool.step()
            gbits = u32(opt.bits())
            gidx = u32(opt.idx())
            for j, sh in enumerate(shards):
                lo, hi, _ = spec[j]
                out = pool.out(j)
                got = local_words(gbits, lo, hi)
                flips = popcount(got ^ out["bits"])
                rep.flips += flips
                rep.mask_bits += hi - lo
                rep.note(flips == 0)
                k0, k1 = kofs[sh], kofs[sh + 1]
                if flips == 0:
                    rep.note(np.array_equal(gidx[k0:k1] - np.uint32(lo), out["idx"]))
                if t >= 2:
                    pk = u32(opt.pack()[:, k0:k1])
                    gb = u32(opt.gbar()[k0:k1])
                    rep.note(np.array_equal(pk, out["pack"].view(np.uint32)))
                    rep.note(np.array_equal(gb, out["gbar"].view(np.uint32)))
        del bufs
        final = pool.dump()
        for j, sh in enumerate(shards):
            lo, hi, _ = spec[j]
            f = final[j]
            assert_close_f32(params[lo:hi].cpu().numpy(), f["w"], f"w shard {sh}")
            assert_close_f32(opt.m[lo:hi].cpu().numpy(), f["m"], f"m shard {sh}")
            rep.note(np.array_equal(u32(params[lo:hi]), f["w"].view(np.uint32)))
            rep.note(np.array_equal(u32(opt.m[lo:hi]), f["m"].view(np.uint32)))
            for r, w in enumerate((0, W - 1)):
                assert_close_f32(opt.e[w][lo:hi].cpu().numpy(), f["e"][r], f"e[{w}] shard {sh}")
                rep.note(np.array_equal(u32(opt.e[w][lo:hi]), f["e"][r].view(np.uint32)))
        del final, f
    assert rep.flips <= MAX_FLIP_FRACTION * rep.mask_bits, f"{rep.flips} mask flips"
    opt.close()
    return rep

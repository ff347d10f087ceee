"""The shard-parallel oracle runner (oracle/pool.py) against the whole-problem
oracle, on the CPU.

Optimizer shards are independent ("SCAPE" Sec. II-A, even partition of the
optimizer state; "Sintesi Tecnica: SCAPE" Sec. 2, each worker selects its mask
only inside its own partition), so running every shard as its own one-shard
problem in its own process must reproduce the whole problem bit for bit:
masks, index lists, packed buffers, synchronised buffer, w, m and residuals.
The full-size GPU parity tests rely on this to compare sampled shards."""
import numpy as np
import pytest

from oracle import oracle as O
from oracle.pool import ShardOracles
from sparse_communication_sharded_gb300 import synth
from tests._harness import HP, bits_to_bool, local_words, popcount


@pytest.mark.parametrize("P,W,s,dtype,quant", [(50003, 4, 0.9, "bf16", False),
                                                (20011, 5, 0.99, "f32", True)])
def test_pool_of_all_shards_equals_whole_problem(P, W, s, dtype, quant):
    wl = synth.Workload("t", (("flat", P),), W=W, sparsity=s, steps=5, grad_dtype=dtype,
                        quantum=2.0 ** -15 if quant else None)
    gen = synth.GradientStream(wl, seed=13, device="cpu")
    w0 = synth.init_params(P, seed=13).numpy()
    st = O.new_state(w0, W, s, HP)
    start, ks = O.layout(P, W, s)
    kofs = np.concatenate([[0], np.cumsum(ks)])
    spec = [(start[j], start[j + 1], ks[j]) for j in range(W)]
    with ShardOracles(spec, W, dtype, HP, lambda lo, hi: w0[lo:hi], dump_rows=range(W),
                      pin=False) as pool:
        for t in range(1, 6):
            grads = [synth.to_numpy_grad(g) for g in gen.next()]
            for j, (lo, hi, _) in enumerate(spec):
                for w in range(W):
                    pool.grads(j)[w] = grads[w][lo:hi]
            times = pool.step()
            assert len(times) == W and min(times) >= 0.0
            rec = O.advance(st, grads)
            for j, (lo, hi, _) in enumerate(spec):
                out = pool.out(j)
                assert np.array_equal(local_words(rec["bits"], lo, hi), out["bits"])
                assert np.array_equal(rec["idx"][kofs[j]:kofs[j + 1]] - np.uint32(lo), out["idx"])
                if t >= 2:
                    k0, k1 = kofs[j], kofs[j + 1]
                    assert np.array_equal(rec["pack"][:, k0:k1].view(np.uint32),
                                          out["pack"].view(np.uint32))
                    assert np.array_equal(rec["gbar"][k0:k1].view(np.uint32),
                                          out["gbar"].view(np.uint32))
        final = pool.dump()
        for j, (lo, hi, _) in enumerate(spec):
            assert np.array_equal(final[j]["w"].view(np.uint32), st.w[lo:hi].view(np.uint32))
            assert np.array_equal(final[j]["m"].view(np.uint32), st.m[lo:hi].view(np.uint32))
            for w in range(W):
                assert np.array_equal(final[j]["e"][w].view(np.uint32),
                                      st.e[w][lo:hi].view(np.uint32))


def test_local_words_matches_bit_by_bit_extraction():
    r = np.random.default_rng(3)
    g = r.integers(0, 2 ** 32, 40, dtype=np.uint64).astype(np.uint32)
    P = 40 * 32
    for lo, hi in ((0, 32), (0, 1), (5, 70), (31, 33), (32, 1280), (17, 1280), (700, 701)):
        got = local_words(g, lo, hi)
        want = np.packbits(bits_to_bool(g, lo, hi), bitorder="little")
        want = np.concatenate([want, np.zeros((-want.size) % 4, np.uint8)]).view(np.uint32)
        assert np.array_equal(got, want), (lo, hi)
        assert popcount(got) == int(bits_to_bool(g, lo, hi).sum())
    assert hi <= P

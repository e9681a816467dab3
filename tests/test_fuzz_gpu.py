"""Seeded fuzz of the GEMVs and the verify kernels against the oracle: shapes
drawn at random (fast and plain GEMV paths, ragged row tiles, every stream
count, stream-K splits with one or several CTAs per tile), the oracle's bars
(|err| <= 1e-5 * sum |w x| per output; argmax, matches and accepted lengths
bit-exact).  The draws are fixed by the seed, so a failure reproduces."""
import numpy as np
import pytest
import torch

import oracle
import pti_synth
import stream_quantized_gemv_gb300 as pti

pytestmark = pytest.mark.gpu

TOL = 1e-5
RNG = np.random.default_rng(20261202)
Q8_CASES = [(int(RNG.integers(1, 3000)), int(RNG.integers(1, 48)) * 32, int(RNG.integers(1, 5)), s)
            for s in range(24)]
TWIN_CASES = [(int(RNG.integers(1, 2000)), int(RNG.integers(1, 40)) * 32, int(RNG.integers(1, 3)), s)
              for s in range(12)]
VERIFY_CASES = [(int(RNG.integers(0, 40)), int(RNG.integers(1, 5)), int(RNG.integers(1, 70000)), s)
                for s in range(10)]


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def check(y, ref, bound, what):
    err = np.abs(np.asarray(y, dtype=np.float64) - ref)
    bad = err > TOL * bound
    assert not bad.any(), f"{what}: {bad.sum()} outputs off, max err/bound {np.max(err / np.maximum(bound, 1e-300)):.3g}"


@pytest.mark.parametrize("rows,cols,n,seed", Q8_CASES)
def test_q8_fuzz(rows, cols, n, seed):
    w = pti_synth.q8_matrix(rows, cols, seed=100 + seed)
    x = pti_synth.activations(n, cols, seed=100 + seed, tensor_id=5)
    y = pti.q8_gemv_nstream(dev(w), rows, cols, dev(x)).cpu().numpy()
    ref, bound = oracle.q8_gemv(w, rows, cols, x)
    check(y, ref, bound, f"q8 {rows}x{cols} n={n}")


@pytest.mark.parametrize("rows,cols,per_model,seed", TWIN_CASES)
def test_twin_fuzz(rows, cols, per_model, seed):
    w = pti_synth.twin_matrix(rows, cols, seed=200 + seed)
    xa = pti_synth.activations(per_model, cols, seed=200 + seed, tensor_id=6)
    xb = pti_synth.activations(per_model, cols, seed=200 + seed, tensor_id=7)
    ra, rb, ba, bb = [], [], [], []
    for s in range(per_model):
        a_, b_, c_, d_ = oracle.twin_gemv(w, rows, cols, xa[s], xb[s])
        ra.append(a_); rb.append(b_); ba.append(c_); bb.append(d_)
    if per_model == 1:
        ya, yb = pti.ssq_twin_gemv(dev(w), rows, cols, dev(xa[0]), dev(xb[0]))
    else:
        ya, yb = pti.ssq_twin_gemv_nstream(dev(w), rows, cols, dev(xa), dev(xb))
    check(ya.cpu().numpy().reshape(per_model, rows), np.array(ra), np.array(ba), f"twin A {rows}x{cols}")
    check(yb.cpu().numpy().reshape(per_model, rows), np.array(rb), np.array(bb), f"twin B {rows}x{cols}")


@pytest.mark.parametrize("steps,n,vocab,seed", VERIFY_CASES)
def test_verify_fuzz(steps, n, vocab, seed):
    lg, gs, _ = pti_synth.verify_batch(steps, n, vocab, 0.5, seed=300 + seed)
    a, m, c = pti.verify_greedy(dev(lg), dev(gs))
    ra, rm, rc = oracle.verify_greedy(lg, gs)
    assert np.array_equal(a.cpu().numpy(), ra)
    assert np.array_equal(c.cpu().numpy(), rc)
    if n > 1:
        assert np.array_equal(m.cpu().numpy(), rm)

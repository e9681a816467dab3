"""GPU sampling-mode verify against the oracle.

The draw is the inverse-CDF token of softmax(logits / T) for a supplied
uniform number u.  The kernel computes the CDF in fp32, the oracle in fp64, so
the two may disagree only where u lies within rounding of an interval edge.
The bar, derived from the arithmetic: each fp32 partial sum of the kernel
holds at most a few hundred terms (one lane's share of a warp's segment, then
a 16-way and a 512-way combine), so its relative error is below
300 * 2^-24 ~ 2e-5, and exp2f adds a few ulp per term.  Hence
  * where the oracle's margin (distance of u from the drawn interval's edges)
    exceeds EPS = 5e-5 the tokens are equal;
  * everywhere the kernel's token v has mass and satisfies
    CDF(v - 1) - EPS <= u < CDF(v) + EPS in fp64;
  * match flags and accepted-prefix lengths are exactly those the kernel's
    own tokens imply (bit-exact), and equal the oracle's where every token of
    the step agrees;
  * the collision probability sum p^2 is within 1e-4 relative of the oracle.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import pti_synth
import stream_quantized_gemv_gb300 as pti

pytestmark = pytest.mark.gpu

EPS = 5e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    pti.build()
    pti.lib()
    yield
    assert pti.device_error() == 0


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run(logits, guess, uniform, temperature):
    t, m, a, c = pti.verify_sample(dev(logits), dev(guess), dev(uniform), temperature)
    return t.cpu().numpy(), m.cpu().numpy(), a.cpu().numpy(), c.cpu().numpy()


def cdf64(logits, temperature):
    lg = logits.astype(np.float64)
    top = np.max(lg, axis=-1, keepdims=True)
    e = np.exp((lg - top) / temperature)
    p = e / e.sum(axis=-1, keepdims=True)
    return p, np.cumsum(p, axis=-1)


def implied_match(guess, token):
    steps, n = token.shape
    match = (guess[:, 1:] == token[:, :-1]).astype(np.uint8)
    accept = np.zeros(steps, np.int32)
    for t in range(steps):
        k = 0
        while k < n - 1 and match[t, k]:
            k += 1
        accept[t] = k
    return match, accept


def check(logits, guess, uniform, temperature, out):
    tok, match, accept, col = out
    steps, n, vocab = logits.shape
    r_tok, r_match, r_acc, r_col, r_margin = oracle.verify_sample(logits, guess, uniform, temperature)
    assert tok.dtype == np.int32 and np.all((tok >= 0) & (tok < vocab))
    sure = r_margin > EPS
    assert np.array_equal(tok[sure], r_tok[sure]), np.argwhere(sure & (tok != r_tok))[:5]
    p, cdf = cdf64(logits, temperature)
    pv = np.take_along_axis(p, tok[..., None], 2)[..., 0]
    hi = np.take_along_axis(cdf, tok[..., None], 2)[..., 0]
    lo = hi - pv
    u = uniform.astype(np.float64)
    assert np.all(pv > 0.0)
    assert np.all(lo - EPS <= u) and np.all(u < hi + EPS)
    i_match, i_acc = implied_match(guess, tok)
    if n > 1:
        assert np.array_equal(match, i_match)
    assert np.array_equal(accept, i_acc)
    same = np.all(tok == r_tok, axis=1)
    if n > 1:
        assert np.array_equal(match[same], r_match[same])
    assert np.array_equal(accept[same], r_acc[same])
    assert np.allclose(col, r_col, rtol=1e-4, atol=0.0)
    return r_tok, sure


def planted_guesses(r_tok, vocab, p, seed):
    """guess[t][s+1] = the oracle's draw of stream s with probability p, else
    the next token: accept chains of every length occur."""
    steps, n = r_tok.shape
    keep = pti_synth.uniform_f32(seed, 99, steps * n).reshape(steps, n) < p
    guess = np.zeros((steps, n), np.int32)
    guess[:, 0] = pti_synth.index_uniform(seed, 98, steps, vocab)
    if n > 1:
        guess[:, 1:] = np.where(keep[:, 1:], r_tok[:, :-1], (r_tok[:, :-1] + 1) % vocab)
    return guess


@pytest.mark.parametrize("n", [1, 2, 3, 4])
@pytest.mark.parametrize("vocab", [1, 2, 5, 63, 64, 1000, 1001, 4099, 40000, 151936])
def test_sample_matches_oracle(n, vocab):
    steps = 37 if vocab < 100000 else 9
    temperature = 0.7 + 0.1 * n
    logits, uniform = pti_synth.sample_batch(steps, n, vocab, seed=vocab + 10 * n)
    r_tok, _, _, _, _ = oracle.verify_sample(logits, np.zeros((steps, n), np.int32), uniform, temperature)
    guess = planted_guesses(r_tok, vocab, 0.7, seed=vocab)
    out = run(logits, guess, uniform, temperature)
    _, sure = check(logits, guess, uniform, temperature, out)
    assert sure.mean() > 0.25  # a good share of the draws is compared exactly


@pytest.mark.parametrize("temperature", [1e-20, 0.05, 1.0, 25.0, 1e6])
def test_sample_temperatures(temperature):
    steps, n, vocab = 16, 4, 5000
    logits, uniform = pti_synth.sample_batch(steps, n, vocab, seed=11)
    guess = np.zeros((steps, n), np.int32)
    check(logits, guess, uniform, temperature, run(logits, guess, uniform, temperature))


def test_tiny_temperature_draws_among_tied_maxima():
    """T -> 0 leaves the tied maxima equally likely: with k ties the draw is
    the floor(u k)-th of them (u kept away from the interval edges)."""
    vocab, k = 3000, 5
    ties = np.array([7, 100, 1500, 2998, 2999])
    us = np.array([0.03, 0.25, 0.41, 0.77, 0.95], np.float32)
    logits = np.full((len(us), 1, vocab), -3.0, np.float32)
    logits[:, :, ties] = 4.0
    logits[:, :, 50] = 3.999
    tok, _, _, col = run(logits, np.zeros((len(us), 1), np.int32), us[:, None], 1e-30)
    assert np.array_equal(tok[:, 0], ties[np.floor(us * k).astype(int)])
    assert np.allclose(col, 1.0 / k, rtol=1e-6)


@pytest.mark.parametrize("masked", [0.5, 0.99])
def test_masked_tokens_are_never_drawn(masked):
    steps, n, vocab = 24, 4, 6001
    logits, uniform = pti_synth.sample_batch(steps, n, vocab, seed=12, masked=masked)
    guess = np.zeros((steps, n), np.int32)
    out = run(logits, guess, uniform, 1.0)
    check(logits, guess, uniform, 1.0, out)
    assert np.all(np.isfinite(np.take_along_axis(logits, out[0][..., None], 2)))


def test_u_zero_draws_the_first_token_with_mass():
    """u = 0 is exact: the draw is the first token whose logit is finite."""
    steps, n, vocab = 8, 4, 9000
    logits, _ = pti_synth.sample_batch(steps, n, vocab, seed=13)
    first = pti_synth.index_uniform(13, 50, steps * n, vocab).reshape(steps, n)
    for t in range(steps):
        for s in range(n):
            logits[t, s, :first[t, s]] = -np.inf
    tok, _, _, _ = run(logits, np.zeros((steps, n), np.int32), np.zeros((steps, n), np.float32), 0.9)
    assert np.array_equal(tok, first.astype(np.int32))


def test_u_near_one_draws_a_late_token():
    steps, n, vocab = 8, 2, 2048
    logits, _ = pti_synth.sample_batch(steps, n, vocab, seed=14, sigma=0.1)
    u = np.full((steps, n), np.float32(1.0 - 2.0 ** -24))
    guess = np.zeros((steps, n), np.int32)
    out = run(logits, guess, u, 1.0)
    check(logits, guess, u, 1.0, out)
    assert np.all(out[0] >= vocab - 8)


def test_stratified_draws_follow_p():
    """K draws with u = (k + 1/2) / K from one row: an exact inverse CDF draws
    each token K p(v) times, +-1.  The grid spacing 1/K is above 2 EPS, so
    rounding can move at most one grid point across each of a token's two
    interval edges: the bound is 3."""
    K, vocab, temperature = 8192, 600, 0.8
    row, _ = pti_synth.sample_batch(1, 1, vocab, seed=15, sigma=1.5)
    logits = np.repeat(row, K, axis=0)
    u = ((np.arange(K) + 0.5) / K).astype(np.float32)[:, None]
    tok, _, _, _ = run(logits, np.zeros((K, 1), np.int32), u, temperature)
    counts = np.bincount(tok[:, 0], minlength=vocab)
    p, _ = cdf64(row[0, 0], temperature)
    assert np.all(np.abs(counts - K * p) <= 3.0)


def test_misaligned_and_ragged_rows_take_the_scalar_path():
    steps, n, vocab = 12, 3, 2051
    logits, uniform = pti_synth.sample_batch(steps, n, vocab, seed=16)
    buf = torch.empty(steps * n * vocab + 1, dtype=torch.float32, device="cuda")
    buf[1:] = dev(logits).reshape(-1)
    view = buf[1:].view(steps, n, vocab)
    guess = np.zeros((steps, n), np.int32)
    t, m, a, c = pti.verify_sample(view, dev(guess), dev(uniform), 1.1)
    check(logits, guess, uniform, 1.1, (t.cpu().numpy(), m.cpu().numpy(), a.cpu().numpy(), c.cpu().numpy()))


def test_sample_deterministic_and_collision_optional():
    steps, n, vocab = 64, 4, 30000
    logits, uniform = pti_synth.sample_batch(steps, n, vocab, seed=17)
    lg, un, gs = dev(logits), dev(uniform), dev(np.zeros((steps, n), np.int32))
    a = pti.verify_sample(lg, gs, un, 0.9)
    b = pti.verify_sample(lg, gs, un, 0.9, collision=False)
    assert b[3] is None
    for x, y in zip(a[:3], b[:3]):
        assert torch.equal(x, y)


def test_empty_batch():
    lg = torch.empty((0, 4, 100), dtype=torch.float32, device="cuda")
    t, m, a, c = pti.verify_sample(lg, torch.empty((0, 4), dtype=torch.int32, device="cuda"),
                                   torch.empty((0, 4), dtype=torch.float32, device="cuda"), 1.0)
    assert t.numel() == 0 and a.numel() == 0


def test_full_size_batch_sampled_rows_and_acceptance_rate():
    """The 4096 steps x 4 streams x 151936 batch in the benchmark's launch
    configuration: sampled steps against the oracle, and the pages' rule as a
    property at full size: a guess that is an independent draw from the same
    distribution is accepted at the mean collision probability (within 4
    standard errors)."""
    steps, n, vocab, temperature = 4096, 4, 151936, 1.0
    logits, uniform = pti_synth.sample_batch_device(steps, n, vocab, seed=3)
    _, u2 = pti_synth.sample_batch_device(steps, n, 1, seed=4)
    zeros = torch.zeros((steps, n), dtype=torch.int32, device="cuda")
    tok2, _, _, _ = pti.verify_sample(logits, zeros, u2, temperature)  # independent draws
    guess = torch.zeros_like(zeros)
    guess[:, 1:] = tok2[:, :-1]
    tok, match, accept, col = pti.verify_sample(logits, guess, uniform, temperature)
    torch.cuda.synchronize()
    pick = [0, 1, 2047, 4095]
    lg = logits[pick].cpu().numpy()
    out = tuple(x[pick].cpu().numpy() for x in (tok, match, accept, col))
    check(lg, guess[pick].cpu().numpy(), uniform[pick].cpu().numpy(), temperature, out)
    q = col[:, :-1].double().cpu().numpy().reshape(-1)
    rate = match.double().cpu().numpy().reshape(-1)
    se = math.sqrt(float(np.mean(q * (1 - q))) / q.size)
    assert abs(rate.mean() - q.mean()) <= 4 * se, (rate.mean(), q.mean(), se)
    m_np, a_np = implied_match(guess.cpu().numpy(), tok.cpu().numpy())
    assert np.array_equal(match.cpu().numpy(), m_np) and np.array_equal(accept.cpu().numpy(), a_np)

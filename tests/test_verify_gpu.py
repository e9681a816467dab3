"""GPU greedy verify against the oracle: argmax, match flags and accepted-prefix
length are compared bit for bit; at the full 4096 x 4 x 151936 batch the
planted maxima and guesses fix every output and a Monte-Carlo mean is checked
against 1 + p + p^2 + p^3."""
import math

import numpy as np
import pytest
import torch

import oracle
import pti_synth
import stream_quantized_gemv_gb300 as pti

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    pti.build()
    pti.lib()
    yield
    assert pti.device_error() == 0


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run(logits, guess):
    a, m, c = pti.verify_greedy(dev(logits), dev(guess))
    return a.cpu().numpy(), m.cpu().numpy(), c.cpu().numpy()


@pytest.mark.parametrize("n", [1, 2, 3, 4])
@pytest.mark.parametrize("vocab", [1, 2, 5, 1000, 1001, 151936])
def test_verify_matches_oracle(n, vocab):
    steps = 37 if vocab < 100000 else 9
    logits, guess, planted = pti_synth.verify_batch(steps, n, vocab, 0.6, seed=vocab + n)
    a_ref, m_ref, c_ref = oracle.verify_greedy(logits, guess)
    a, m, c = run(logits, guess)
    assert np.array_equal(a, a_ref) and np.array_equal(a, planted)
    assert np.array_equal(m, m_ref)
    assert np.array_equal(c, c_ref)


def test_verify_ties_and_infinities():
    v = 4099    # odd vocabulary: scalar path
    rows = []
    for pos in ([0, v - 1], [3, 9, v - 1], [v - 1], [2048, 2049], [4000, 17]):
        r = np.full(v, -2.0, np.float32)
        r[pos] = 1.5
        rows.append(r)
    r = np.zeros(v, np.float32)
    r[4] = -0.0
    rows.append(r)
    rows.append(np.full(v, -np.inf, np.float32))
    r = np.zeros(v, np.float32)
    r[[700, 12]] = np.inf
    rows.append(r)
    logits = np.stack(rows)[:, None, :]
    guess = np.zeros((len(rows), 1), np.int32)
    a_ref, _, _ = oracle.verify_greedy(logits, guess)
    a, _, _ = run(logits, guess)
    assert a[:, 0].tolist() == a_ref[:, 0].tolist() == [0, 3, v - 1, 2048, 17, 0, 0, 12]
    # vector path (vocabulary multiple of 4, aligned rows)
    v4 = 4096
    lg = np.full((3, 1, v4), -1.0, np.float32)
    lg[0, 0, [4095, 5, 2000]] = 7.0
    lg[1, 0, [1, 2, 3, 0]] = 7.0
    lg[2, 0, :] = 0.0
    a, _, _ = run(lg, np.zeros((3, 1), np.int32))
    assert a[:, 0].tolist() == [5, 0, 0]


def test_verify_empty_batch_is_a_no_op():
    logits = torch.empty((0, 4, 10), dtype=torch.float32, device="cuda")
    guess = torch.empty((0, 4), dtype=torch.int32, device="cuda")
    a, m, c = pti.verify_greedy(logits, guess)
    assert a.numel() == 0 and m.numel() == 0 and c.numel() == 0


def test_greedy_self_speculation_accepts_everything_on_gpu():
    """Toy deterministic model (bigram logits table); greedy rollouts supply the
    guesses, so every guess is accepted: accept_len == N - 1 on every step."""
    vocab, n, steps = 64, 4, 512
    table = pti_synth.normal_f32(7, 0, vocab * vocab).reshape(vocab, vocab)
    confirmed = pti_synth.index_uniform(7, 1, steps, vocab)
    logits = np.empty((steps, n, vocab), np.float32)
    guess = np.empty((steps, n), np.int32)
    for t in range(steps):
        tok = int(confirmed[t])
        for s in range(n):
            guess[t, s] = tok
            logits[t, s] = table[tok]
            tok = int(np.argmax(table[tok]))
    _, _, c = run(logits, guess)
    assert np.all(c == n - 1)


@pytest.mark.parametrize("p", [1.0, 0.75, 0.6, 0.4])
def test_full_batch_4096x4x151936(p):
    """The full verify batch: N(0, 3) logits with planted maxima, guesses planted
    at rate p.  Every argmax equals the planted index, every accept length equals
    the leading run of planted matches, sampled steps equal the oracle bit for
    bit, and mean tokens/step is within 4 standard errors of 1+p+p^2+p^3."""
    steps, n, vocab = 4096, 4, 151936
    logits, guess, planted = pti_synth.verify_batch_device(steps, n, vocab, p, seed=11, tensor_id=int(p * 100))
    a, m, c = pti.verify_greedy(logits, guess)
    torch.cuda.synchronize()
    assert torch.equal(a, planted)
    want_m = (guess[:, 1:] == planted[:, :-1]).to(torch.int32)
    assert torch.equal(m.to(torch.int32), want_m)
    run_len = torch.cumprod(want_m, dim=1).sum(dim=1).to(torch.int32)
    assert torch.equal(c, run_len)
    sample = torch.tensor([0, 1, 2047, 4095], device="cuda")
    lg = logits[sample].cpu().numpy()
    gs = guess[sample].cpu().numpy()
    a_ref, m_ref, c_ref = oracle.verify_greedy(lg, gs)
    assert np.array_equal(a[sample].cpu().numpy(), a_ref)
    assert np.array_equal(m[sample].cpu().numpy(), m_ref)
    assert np.array_equal(c[sample].cpu().numpy(), c_ref)
    emitted = (1 + c.double()).cpu().numpy()
    probs = np.array([p ** k * (1 - p) for k in range(n - 1)] + [p ** (n - 1)])
    vals = np.arange(1, n + 1, dtype=np.float64)
    mean = float(probs @ vals)
    se = math.sqrt(float(probs @ (vals - mean) ** 2) / steps)
    assert abs(emitted.mean() - (1 + p + p * p + p ** 3)) <= 4 * se + 1e-12
    del logits
    torch.cuda.empty_cache()

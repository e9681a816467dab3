"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test names what fixes the expected value: a library routine on a special
case (numpy's binary16 decode, exact integer matrix products), a closed form,
an invariant the pages state, a fixture holding the pages' printed values, or
brute force on tiny inputs.  They are chosen so that a plausible slip in the
oracle (wrong byte for the scale, swapped high/low byte, transposed operand,
dropped scale, off-by-one in the payload offset, wrong tie rule, wrong
acceptance chaining) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest

import oracle
import pti_synth

# --------------------------------------------------------------------------
# binary16 decode
# --------------------------------------------------------------------------


def test_f16_decode_matches_numpy_for_all_patterns():
    """Every binary16 pattern decodes like numpy's float16 -> float64 routine."""
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


@pytest.mark.parametrize("bits,value", [
    (0x3C00, 1.0), (0xC000, -2.0), (0x7BFF, 65504.0), (0x0001, 2.0 ** -24),
    (0x0400, 2.0 ** -14), (0x3555, 0.333251953125), (0x0000, 0.0), (0x3800, 0.5),
])
def test_f16_decode_textbook_values(bits, value):
    assert oracle.f16_to_f64(bits) == value


def test_f16_negative_zero_and_inf():
    assert math.copysign(1.0, oracle.f16_to_f64(0x8000)) == -1.0
    assert oracle.f16_to_f64(0x7C00) == math.inf
    assert oracle.f16_to_f64(0xFC00) == -math.inf
    assert math.isnan(oracle.f16_to_f64(0x7E00))


# --------------------------------------------------------------------------
# Q8 GEMV
# --------------------------------------------------------------------------

def _q8_fields(w, rows, cols):
    """Scales (via numpy float16) and int8 payload (via numpy int8 view) of a Q8 buffer."""
    blk = w.reshape(rows, cols // 32, 34)
    scales = blk[:, :, 0:2].copy().view("<f2").astype(np.float64).reshape(rows, cols // 32)
    q = blk[:, :, 2:].copy().view(np.int8).reshape(rows, cols)
    return scales, q


def test_q8_one_hot_picks_single_weight():
    """x = e_j gives y[r] = d(r, j // 32) * q[r][j] (the scale times one int8)."""
    rows, cols = 7, 96          # rows != cols so a transposed operand fails
    w = pti_synth.q8_matrix(rows, cols, seed=11)
    scales, q = _q8_fields(w, rows, cols)
    x = np.eye(cols, dtype=np.float32)          # cols streams, one per column
    y, bound = oracle.q8_gemv(w, rows, cols, x)
    expect = (scales[:, np.arange(cols) // 32] * q).T   # [stream j][row r]
    assert np.array_equal(y, expect)
    assert np.array_equal(bound, np.abs(expect))


def test_q8_integer_case_equals_integer_matmul():
    """Scales 1.0 and integer x in [-4, 4]: y is the exact integer product q @ x."""
    rows, cols = 33, 256
    w = pti_synth.q8_matrix(rows, cols, seed=3).reshape(-1, 34).copy()
    w[:, 0] = 0x00
    w[:, 1] = 0x3C                   # binary16 1.0 little-endian
    w = w.reshape(-1)
    _, q = _q8_fields(w, rows, cols)
    rng = np.random.default_rng(5)
    xi = rng.integers(-4, 5, size=(3, cols))
    y, _ = oracle.q8_gemv(w, rows, cols, xi.astype(np.float32))
    expect = (q.astype(np.int64) @ xi.T).T
    assert np.array_equal(y, expect.astype(np.float64))


def test_q8_zero_weights_give_zero():
    rows, cols = 5, 64
    w = pti_synth.q8_matrix(rows, cols, seed=2).reshape(-1, 34).copy()
    w[:, 2:] = 0
    y, bound = oracle.q8_gemv(w.reshape(-1), rows, cols, pti_synth.activations(2, cols, 1))
    assert not y.any() and not bound.any()


def test_q8_linearity():
    """y(2 x1 + x2) = 2 y(x1) + y(x2), with x chosen so the float32 sum is exact."""
    rows, cols = 9, 128
    w = pti_synth.q8_matrix(rows, cols, seed=4)
    rng = np.random.default_rng(0)
    x1 = (rng.integers(-64, 65, size=cols) / 8.0).astype(np.float32)
    x2 = (rng.integers(-64, 65, size=cols) / 8.0).astype(np.float32)
    y1, b1 = oracle.q8_gemv(w, rows, cols, x1)
    y2, b2 = oracle.q8_gemv(w, rows, cols, x2)
    y3, _ = oracle.q8_gemv(w, rows, cols, 2 * x1 + x2)
    tol = 1e-13 * (2 * b1 + b2)
    assert np.all(np.abs(y3 - (2 * y1 + y2)) <= tol)


def test_q8_rows_and_streams_are_independent():
    rows, cols = 12, 160
    w = pti_synth.q8_matrix(rows, cols, seed=6)
    x = pti_synth.activations(4, cols, 6)
    y, _ = oracle.q8_gemv(w, rows, cols, x)
    idx = np.array([11, 0, 5], dtype=np.int64)
    ys, _ = oracle.q8_gemv(w, rows, cols, x, rows_idx=idx)
    assert np.array_equal(ys, y[:, idx])
    for s in range(4):
        y1, _ = oracle.q8_gemv(w, rows, cols, x[s:s + 1])
        assert np.array_equal(y1[0], y[s])


def test_q8_block_permutation_invariance():
    """Permuting the blocks of every row together with the matching x segments keeps y."""
    rows, cols = 6, 256
    nb = cols // 32
    w = pti_synth.q8_matrix(rows, cols, seed=8)
    x = pti_synth.activations(2, cols, 8)
    perm = np.random.default_rng(1).permutation(nb)
    wp = w.reshape(rows, nb, 34)[:, perm, :].reshape(-1).copy()
    xp = x.reshape(2, nb, 32)[:, perm, :].reshape(2, cols).copy()
    y, b = oracle.q8_gemv(w, rows, cols, x)
    yp, _ = oracle.q8_gemv(wp, rows, cols, xp)
    assert np.all(np.abs(y - yp) <= 1e-13 * b)


def test_q8_bound_dominates_and_is_tight_for_nonnegative_terms():
    rows, cols = 8, 96
    w = pti_synth.q8_matrix(rows, cols, seed=9)
    x = pti_synth.activations(2, cols, 9)
    y, b = oracle.q8_gemv(w, rows, cols, x)
    assert np.all(b >= np.abs(y))
    blk = w.reshape(-1, 34).copy()
    blk[:, 2:] = blk[:, 2:].view(np.int8).__abs__().view(np.uint8)
    yp, bp = oracle.q8_gemv(blk.reshape(-1), rows, cols, np.abs(x))
    assert np.allclose(yp, bp, rtol=1e-14, atol=0)


def test_q8_rejects_bad_shapes():
    w = pti_synth.q8_matrix(2, 64, seed=0)
    with pytest.raises(ValueError):
        oracle.q8_gemv(w, 2, 64, np.zeros((1, 63), np.float32))
    with pytest.raises(ValueError):
        oracle.q8_gemv(w, 2, 64, np.zeros((1, 64), np.float32), rows_idx=[2])


# --------------------------------------------------------------------------
# SSQ twin format and twin GEMV
# --------------------------------------------------------------------------

def _read_fixture(golden_dir):
    facts, examples = {}, []
    with open(os.path.join(golden_dir, "ssq_twin_block.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            if parts[0] == "example":
                examples.append((int(parts[1], 16), int(parts[2], 16), int(parts[3], 16),
                                 float(parts[4]), float(parts[5])))
            else:
                facts[parts[0]] = int(parts[1])
    return facts, examples


def test_twin_block_size_is_two_q8_blocks(golden_dir):
    facts, _ = _read_fixture(golden_dir)
    assert facts["block_bytes"] == oracle.TWIN_BLOCK_BYTES == 2 * facts["q8_block_bytes"]
    assert facts["q8_block_bytes"] == oracle.Q8_BLOCK_BYTES
    assert facts["positions"] == oracle.BLOCK_COLS


def test_twin_weight_extraction_matches_page_examples(golden_dir):
    """The pages' rule wa = (int8)(pw >> 8), wb = (int8)(pw & 0xFF) on worked slots."""
    _, examples = _read_fixture(golden_dir)
    assert examples
    for pw, sa, sb, wa_ref, wb_ref in examples:
        blk = np.zeros(68, dtype=np.uint8)
        blk[0:2] = [sa & 0xFF, sa >> 8]
        blk[2:4] = [sb & 0xFF, sb >> 8]
        pos = 5
        blk[4 + 2 * pos] = pw & 0xFF          # little-endian uint16 at slot 5
        blk[5 + 2 * pos] = pw >> 8
        wa, wb = oracle.twin_weight(blk, 32, 0, pos)
        assert (wa, wb) == (wa_ref, wb_ref), hex(pw)


def test_twin_pack_unpack_exhaustive_payload():
    """All 65536 uint16 payload values and all 65536 scale patterns round-trip."""
    n_blocks = 65536 // 32
    twin = np.zeros((n_blocks, 68), dtype=np.uint8)
    pw = np.arange(65536, dtype="<u2").reshape(n_blocks, 32)
    twin[:, 4:] = pw.view(np.uint8).reshape(n_blocks, 64)
    scales = np.arange(65536, dtype="<u2")
    twin[:, 0:2] = scales[:n_blocks].view(np.uint8).reshape(n_blocks, 2)
    twin[:, 2:4] = scales[n_blocks:2 * n_blocks].view(np.uint8).reshape(n_blocks, 2)
    qa, qb = oracle.twin_unpack(twin.reshape(-1))
    qa = qa.reshape(n_blocks, 34)
    qb = qb.reshape(n_blocks, 34)
    assert np.array_equal(qa[:, 2:], (pw >> 8).astype(np.uint8))     # high byte -> A
    assert np.array_equal(qb[:, 2:], (pw & 0xFF).astype(np.uint8))   # low byte -> B
    assert np.array_equal(qa[:, 0:2].copy().view("<u2").ravel(), scales[:n_blocks])
    assert np.array_equal(qb[:, 0:2].copy().view("<u2").ravel(), scales[n_blocks:2 * n_blocks])
    assert np.array_equal(oracle.twin_pack(qa, qb), twin.reshape(-1))
    # all 65536 scale patterns in both fields
    for field in (0, 2):
        t = np.zeros((65536, 68), dtype=np.uint8)
        t[:, field:field + 2] = scales.view(np.uint8).reshape(65536, 2)
        a, b = oracle.twin_unpack(t.reshape(-1))
        assert np.array_equal(oracle.twin_pack(a, b), t.reshape(-1))


def test_twin_pack_random_round_trip_and_byte_multiset():
    rows, cols = 5, 128
    qa = pti_synth.q8_matrix(rows, cols, seed=21)
    qb = pti_synth.q8_matrix(rows, cols, seed=22)
    t = oracle.twin_pack(qa, qb)
    assert t.size == qa.size + qb.size
    a, b = oracle.twin_unpack(t)
    assert np.array_equal(a, qa) and np.array_equal(b, qb)
    for blk in range(t.size // 68):
        tb = np.sort(t[68 * blk:68 * (blk + 1)])
        ab = np.sort(np.concatenate([qa[34 * blk:34 * (blk + 1)], qb[34 * blk:34 * (blk + 1)]]))
        assert np.array_equal(tb, ab)


def test_twin_gemv_equals_two_q8_gemvs_on_unpacked_models():
    rows, cols = 11, 192
    t = pti_synth.twin_matrix(rows, cols, seed=31)
    xa, xb = pti_synth.activations(2, cols, 31)
    ya, yb, ba, bb = oracle.twin_gemv(t, rows, cols, xa, xb)
    qa, qb = oracle.twin_unpack(t)
    ra, rba = oracle.q8_gemv(qa, rows, cols, xa)
    rb, rbb = oracle.q8_gemv(qb, rows, cols, xb)
    assert np.array_equal(ya, ra[0]) and np.array_equal(yb, rb[0])
    assert np.array_equal(ba, rba[0]) and np.array_equal(bb, rbb[0])


def test_twin_one_hot_uses_high_byte_for_a_and_low_byte_for_b():
    rows, cols = 3, 64
    t = pti_synth.twin_matrix(rows, cols, seed=41)
    blk = t.reshape(rows, cols // 32, 68)
    sa = blk[:, :, 0:2].copy().view("<f2").astype(np.float64).reshape(rows, -1)
    sb = blk[:, :, 2:4].copy().view("<f2").astype(np.float64).reshape(rows, -1)
    hi = blk[:, :, 5::2].copy().view(np.int8).reshape(rows, cols)
    lo = blk[:, :, 4::2].copy().view(np.int8).reshape(rows, cols)
    for j in (0, 31, 32, 63):
        e = np.zeros(cols, np.float32)
        e[j] = 1.0
        ya, yb, _, _ = oracle.twin_gemv(t, rows, cols, e, 2 * e)
        assert np.array_equal(ya, sa[:, j // 32] * hi[:, j])
        assert np.array_equal(yb, 2 * sb[:, j // 32] * lo[:, j])


def test_identical_twins_give_identical_outputs():
    rows, cols = 13, 256
    t = pti_synth.twin_matrix(rows, cols, seed=51, identical=True)
    x = pti_synth.activations(1, cols, 51)[0]
    ya, yb, ba, bb = oracle.twin_gemv(t, rows, cols, x, x)
    assert np.array_equal(ya, yb) and np.array_equal(ba, bb)


# --------------------------------------------------------------------------
# Greedy verify
# --------------------------------------------------------------------------

def _brute_argmax(row):
    m = max(row)
    return min(i for i, v in enumerate(row) if v == m)


def test_verify_argmax_brute_force_tiny_vocab():
    """Exhaustive small-value rows for vocab 1, 2, 5 against max/first-index."""
    vals = np.array([-1.0, 0.0, 2.0], dtype=np.float32)
    for vocab in (1, 2, 5):
        grid = np.array(np.meshgrid(*([vals] * vocab), indexing="ij")).reshape(vocab, -1).T
        logits = grid.reshape(-1, 1, vocab).astype(np.float32)
        guess = np.zeros((logits.shape[0], 1), np.int32)
        a, _, acc = oracle.verify_greedy(logits, guess)
        ref = [_brute_argmax(list(r)) for r in grid]
        assert a[:, 0].tolist() == ref
        assert not acc.any()


def test_verify_ties_go_to_lowest_index():
    v = 17
    rows = []
    for pos in ([0, 16], [3, 9, 16], [16], [5, 6]):
        r = np.full(v, -2.0, np.float32)
        r[pos] = 1.5
        rows.append(r)
    r = np.zeros(v, np.float32)
    r[4] = -0.0                     # -0.0 ties with +0.0: index 0 wins
    rows.append(r)
    r = np.full(v, -np.inf, np.float32)
    rows.append(r)
    r = np.zeros(v, np.float32)
    r[[7, 12]] = np.inf
    rows.append(r)
    logits = np.stack(rows)[:, None, :]
    a, _, _ = oracle.verify_greedy(logits, np.zeros((len(rows), 1), np.int32))
    assert a[:, 0].tolist() == [0, 3, 16, 5, 0, 0, 7]


def test_verify_planted_argmax_and_extreme_rates():
    for n in (1, 2, 3, 4):
        for p, expect in ((1.0, n - 1), (0.0, 0)):
            logits, guess, planted = pti_synth.verify_batch(64, n, 997, p, seed=n)
            a, m, acc = oracle.verify_greedy(logits, guess)
            assert np.array_equal(a, planted)
            assert np.all(acc == expect)
            assert m.shape == (64, n - 1)


def test_verify_accept_is_leading_run_of_matches():
    """accept counts matches only up to the first mismatch (brute force on all patterns)."""
    n, vocab = 4, 8
    patterns = np.array(np.meshgrid(*([[0, 1]] * (n - 1)), indexing="ij")).reshape(n - 1, -1).T
    steps = patterns.shape[0]
    logits = np.zeros((steps, n, vocab), np.float32)
    tok = np.arange(steps * n).reshape(steps, n) % vocab
    logits[np.arange(steps)[:, None], np.arange(n)[None, :], tok] = 1.0
    guess = np.zeros((steps, n), np.int32)
    for t in range(steps):
        for s in range(n - 1):
            guess[t, s + 1] = tok[t, s] if patterns[t, s] else (tok[t, s] + 1) % vocab
    _, m, acc = oracle.verify_greedy(logits, guess)
    assert np.array_equal(m, patterns.astype(np.uint8))
    for t in range(steps):
        run = 0
        while run < n - 1 and patterns[t, run]:
            run += 1
        assert acc[t] == run


def test_greedy_self_speculation_accepts_everything():
    """A deterministic toy model (bigram logits table) rolled out greedily from the
    confirmed token supplies the guesses; under greedy decoding the same model
    always agrees with itself, so every guess is accepted (the pages' 100%)."""
    vocab, n, steps = 64, 4, 200
    table = pti_synth.normal_f32(7, 0, vocab * vocab).reshape(vocab, vocab)
    rng = np.random.default_rng(3)
    confirmed = rng.integers(0, vocab, size=steps)
    logits = np.empty((steps, n, vocab), np.float32)
    guess = np.empty((steps, n), np.int32)
    for t in range(steps):
        tok = int(confirmed[t])
        for s in range(n):
            guess[t, s] = tok
            logits[t, s] = table[tok]
            tok = int(np.argmax(table[tok]))     # greedy rollout supplies the next guess
    _, _, acc = oracle.verify_greedy(logits, guess)
    assert np.all(acc == n - 1)


def _read_tokens_table(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "expected_tokens_per_step.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                p, e = line.split()
                rows.append((float(p), float(e)))
    return rows


def test_expected_tokens_closed_form_matches_page_table(golden_dir):
    for p, printed in _read_tokens_table(golden_dir):
        assert abs((1 + p + p ** 2 + p ** 3) - printed) <= 0.025


def test_monte_carlo_acceptance_matches_closed_form(golden_dir):
    """4096 steps per p: mean(1 + accept) within 4 standard errors of 1+p+p^2+p^3."""
    n, steps, vocab = 4, 4096, 151
    for i, (p, _) in enumerate(_read_tokens_table(golden_dir)):
        logits, guess, _ = pti_synth.verify_batch(steps, n, vocab, p, seed=100 + i)
        _, _, acc = oracle.verify_greedy(logits, guess)
        emitted = 1 + acc.astype(np.float64)
        probs = np.array([p ** k * (1 - p) for k in range(n - 1)] + [p ** (n - 1)])
        values = np.arange(1, n + 1, dtype=np.float64)
        mean = float(probs @ values)
        var = float(probs @ (values - mean) ** 2)
        assert mean == pytest.approx(1 + p + p ** 2 + p ** 3, abs=1e-12)
        se = math.sqrt(var / steps)
        assert abs(emitted.mean() - mean) <= 4 * se + 1e-12


# --------------------------------------------------------------------------
# Gated-MLP layer of the decode weight pass
# --------------------------------------------------------------------------

def _diag_q8(n, q_diag, scale_bits=0x3C00, perm=None):
    """An n x n Q8 matrix with q_diag on the (permuted) diagonal and a fixed scale."""
    q = np.zeros((n, n), dtype=np.int8)
    cols = np.arange(n) if perm is None else perm
    q[np.arange(n), cols] = q_diag
    blk = np.zeros((n, n // 32, 34), dtype=np.uint8)
    blk[:, :, 0] = scale_bits & 0xFF
    blk[:, :, 1] = scale_bits >> 8
    blk[:, :, 2:] = q.view(np.uint8).reshape(n, n // 32, 32)
    return blk.reshape(-1)


def test_mlp_layer_with_identity_like_weights():
    """Wg = I, Wu = 2I, Wd = a permutation P: h = norm(SiLU(x) * 2x), x_out = norm(P h)."""
    d = 64
    x = pti_synth.activations(2, d, 61).astype(np.float64)
    perm = np.random.default_rng(2).permutation(d)
    wg = _diag_q8(d, 1)
    wu = _diag_q8(d, 2)
    wd = _diag_q8(d, 1, perm=perm)
    eps = 1e-6
    x_out, h = oracle.mlp_layer(wg, wu, wd, d, d, x, eps)
    hh = x / (1.0 + np.exp(-x)) * (2.0 * x)
    hh = hh / np.sqrt(np.mean(hh ** 2, axis=1, keepdims=True) + eps)
    assert np.allclose(h, hh, rtol=1e-13, atol=0)
    xo = hh[:, perm]
    xo = xo / np.sqrt(np.mean(xo ** 2, axis=1, keepdims=True) + eps)
    assert np.allclose(x_out, xo, rtol=1e-13, atol=0)


def test_mlp_layer_rms_invariants():
    hidden, ffn = 64, 96
    wg = pti_synth.q8_matrix(ffn, hidden, seed=71, tensor_id=0)
    wu = pti_synth.q8_matrix(ffn, hidden, seed=71, tensor_id=1)
    wd = pti_synth.q8_matrix(hidden, ffn, seed=71, tensor_id=2)
    x = pti_synth.activations(3, hidden, 71)
    x_out, h = oracle.mlp_layer(wg, wu, wd, hidden, ffn, x, 1e-6)
    assert np.allclose(np.mean(h ** 2, axis=1), 1.0, rtol=1e-4)
    assert np.allclose(np.mean(x_out ** 2, axis=1), 1.0, rtol=1e-4)


def test_mlp_layer_zero_weights_give_zero():
    d = 32
    z = _diag_q8(d, 0)
    x_out, h = oracle.mlp_layer(z, z, z, d, d, pti_synth.activations(1, d, 1))
    assert not x_out.any() and not h.any()# ---------------------------------------------------------------------------
# Sampling-mode verify ([PTI-readme] §接受机制如何工作, temperature > 0)
# ---------------------------------------------------------------------------
def _one_row(logits, u, temperature):
    lg = np.asarray(logits, np.float32)[None, None, :]
    tok, _, _, col, margin = oracle.verify_sample(lg, np.zeros((1, 1), np.int32),
                                                  np.array([[u]], np.float32), temperature)
    return int(tok[0, 0]), float(col[0, 0]), float(margin[0, 0])


def test_sample_uniform_logits_is_floor_u_v():
    """Equal logits: p = 1/V, the draw is floor(u V) and the collision 1/V."""
    for vocab in (1, 2, 7, 1000, 151936):
        for u in (0.0, 0.1234, 0.5 + 0.25 / vocab, 0.9999):
            tok, col, _ = _one_row(np.full(vocab, 3.5), u, 0.7)
            assert tok == min(vocab - 1, math.floor(np.float32(u) * vocab)), (vocab, u, tok)
            assert abs(col - 1.0 / vocab) <= 1e-12


def test_sample_two_tokens_closed_form():
    """Two tokens: p0 = 1 / (1 + exp((b - a) / T)); the draw is 0 iff u < p0 and
    the collision p0^2 + (1 - p0)^2."""
    for a, b, temp in ((0.0, 1.0, 1.0), (2.0, -1.0, 0.5), (1.0, 1.0, 3.0), (-4.0, 4.0, 2.0)):
        p0 = 1.0 / (1.0 + math.exp((b - a) / temp))
        for u in (0.05, p0 - 1e-4, p0 + 1e-4, 0.95):
            if not 0.0 <= u < 1.0:
                continue
            tok, col, _ = _one_row([a, b], u, temp)
            assert tok == (0 if np.float32(u) < p0 else 1)
            assert abs(col - (p0 * p0 + (1 - p0) ** 2)) <= 1e-12


def test_sample_low_temperature_is_argmax():
    rng = np.random.default_rng(4)
    for _ in range(20):
        row = rng.normal(0, 1, 500).astype(np.float32)
        for u in (1e-3, 0.5, 0.999):  # u = 0 would pick the first token with any (tiny) mass
            tok, col, _ = _one_row(row, u, 1e-4)
            assert tok == int(np.argmax(row)) and col > 1 - 1e-9


def test_sample_stratified_grid_reproduces_p():
    """Inverse-CDF draws at u_k = (k + 1/2) / K hit token v exactly K p(v) times,
    up to one at each interval edge."""
    logits = np.array([0.3, -1.2, 2.0, 0.0, 1.1, -0.4, 0.9], np.float32)
    temp, K = 0.8, 4000
    e = np.exp((logits.astype(np.float64) - logits.max()) / temp)
    p = e / e.sum()
    u = ((np.arange(K) + 0.5) / K).astype(np.float32)
    lg = np.broadcast_to(logits, (K, 1, logits.size)).copy()
    tok, _, _, col, margin = oracle.verify_sample(lg, np.zeros((K, 1), np.int32), u[:, None], temp)
    counts = np.bincount(tok[:, 0], minlength=logits.size)
    assert np.all(np.abs(counts - K * p) <= 1.0 + 1e-9), (counts, K * p)
    assert np.all(margin >= 0.0)
    assert np.allclose(col, np.sum(p * p), rtol=0, atol=1e-14)


def test_sample_temperature_scaling_invariance():
    """Doubling the logits and the temperature changes nothing (exact in fp32)."""
    rng = np.random.default_rng(5)
    lg = rng.normal(0, 2, (6, 3, 300)).astype(np.float32)
    u = rng.random((6, 3)).astype(np.float32)
    g = np.zeros((6, 3), np.int32)
    a = oracle.verify_sample(lg, g, u, 0.6)
    b = oracle.verify_sample(lg * np.float32(2.0), g, u, 1.2)
    assert np.array_equal(a[0], b[0])
    assert np.allclose(a[3], b[3], rtol=1e-12, atol=0)


def test_sample_acceptance_is_the_collision_probability():
    """The pages' rule: a guess drawn from the same distribution as the stream's
    own draw is accepted with probability sum_x p(x)^2.  Monte Carlo over rows of
    various entropies: the accept rate of stream 0's draw against an independent
    draw from an identical row lies within 4 standard errors of the mean
    collision probability."""
    rng = np.random.default_rng(6)
    steps, vocab = 6000, 40
    lg = np.empty((steps, 2, vocab), np.float32)
    base = rng.normal(0, 1.5, (steps, vocab)).astype(np.float32)
    lg[:, 0], lg[:, 1] = base, base
    u = rng.random((steps, 2)).astype(np.float32)
    # the guess for stream 1 is an independent draw from the same row
    g_tok, _, _, _, _ = oracle.verify_sample(lg[:, 1:2].copy(), np.zeros((steps, 1), np.int32), u[:, 1:2].copy(), 0.9)
    guess = np.zeros((steps, 2), np.int32)
    guess[:, 1] = g_tok[:, 0]
    tok, match, accept, col, _ = oracle.verify_sample(lg, guess, u, 0.9)
    rate = match[:, 0].mean()
    q = col[:, 0]
    se = math.sqrt(float(np.mean(q * (1 - q))) / steps)
    assert abs(rate - q.mean()) <= 4 * se + 1e-12, (rate, q.mean(), se)
    assert np.array_equal(accept, match[:, 0].astype(np.int32))


def test_sample_accept_chain_and_margins():
    """Guesses planted equal to the draws are all accepted; a mismatch at stream
    s stops the run there; every draw lies inside its CDF interval."""
    rng = np.random.default_rng(7)
    steps, n, vocab = 50, 4, 64
    lg = rng.normal(0, 2, (steps, n, vocab)).astype(np.float32)
    u = rng.random((steps, n)).astype(np.float32)
    tok, _, _, _, margin = oracle.verify_sample(lg, np.zeros((steps, n), np.int32), u, 1.3)
    guess = np.zeros((steps, n), np.int32)
    guess[:, 1:] = tok[:, :-1]
    _, match, accept, _, _ = oracle.verify_sample(lg, guess, u, 1.3)
    assert np.all(match == 1) and np.all(accept == n - 1)
    guess[:, 2] = (tok[:, 1] + 1) % vocab
    _, match, accept, _, _ = oracle.verify_sample(lg, guess, u, 1.3)
    assert np.all(accept == 1) and np.all(match[:, 1] == 0) and np.all(match[:, 2] == 1)
    e = np.exp((lg.astype(np.float64) - lg.max(axis=2, keepdims=True)) / 1.3)
    cdf = np.cumsum(e / e.sum(axis=2, keepdims=True), axis=2)
    hi = np.take_along_axis(cdf, tok[..., None], 2)[..., 0]
    lo = hi - np.take_along_axis(e / e.sum(axis=2, keepdims=True), tok[..., None], 2)[..., 0]
    assert np.all(lo <= u + 1e-12) and np.all(u < hi + 1e-12) and np.all(margin >= 0)


def test_sample_rejects_bad_temperature():
    lg = np.zeros((1, 1, 4), np.float32)
    for temp in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(ValueError):
            oracle.verify_sample(lg, np.zeros((1, 1), np.int32), np.zeros((1, 1), np.float32), temp)




"""The seeded input generator: determinism, ranges and distributions."""
import numpy as np

import pti_synth


def test_streams_are_deterministic_and_distinct():
    a = pti_synth.draws(0, 0, 0, 1000)
    assert np.array_equal(a, pti_synth.draws(0, 0, 0, 1000))
    assert np.array_equal(a[100:200], pti_synth.draws(0, 0, 100, 100))
    assert not np.array_equal(a, pti_synth.draws(1, 0, 0, 1000))
    assert not np.array_equal(a, pti_synth.draws(0, 1, 0, 1000))


def test_splitmix64_reference_sequence():
    """With base 0 the stream is Vigna's splitmix64 seeded with 0; its first
    output is the published 0xE220A8397B1DCDAF."""
    i = np.array([1], dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = pti_synth._mix(i * pti_synth.GAMMA)
    assert int(z[0]) == 0xE220A8397B1DCDAF


def test_int8_range_and_balance():
    q = pti_synth.int8_uniform(0, 0, 1 << 20)
    assert q.min() == -127 and q.max() == 127
    counts = np.bincount(q.astype(np.int64) + 127, minlength=255)
    assert counts.min() > 0.8 * counts.mean()
    assert abs(q.astype(np.float64).mean()) < 0.2


def test_scales_are_normal_binary16_in_range():
    s = pti_synth.f16_scales(0, 1, 100000).view(np.float16).astype(np.float64)
    lo = np.float16(0.5 / 127)
    hi = np.float16(2.0 / 127)
    assert s.min() >= lo and s.max() <= hi
    assert np.all(s >= 2.0 ** -14)           # normal binary16


def test_normal_moments():
    z = pti_synth.normal_f32(0, 2, 1 << 20).astype(np.float64)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01


def test_layouts_have_the_documented_sizes():
    assert pti_synth.q8_matrix(3, 64, 0).size == 3 * 2 * 34
    assert pti_synth.twin_matrix(3, 64, 0).size == 3 * 2 * 68
    t = pti_synth.twin_matrix(2, 64, 0, identical=True).reshape(-1, 68)
    assert np.array_equal(t[:, 0:2], t[:, 2:4])
    assert np.array_equal(t[:, 4::2], t[:, 5::2])


def test_verify_batch_plants_a_unique_maximum():
    logits, guess, planted = pti_synth.verify_batch(16, 4, 301, 0.5, seed=9)
    for t in range(16):
        for s in range(4):
            row = logits[t, s]
            assert np.sum(row == row.max()) == 1
            assert row[planted[t, s]] == row.max()
    assert guess.dtype == np.int32 and guess.min() >= 0 and guess.max() < 301


def test_uniform_f32_is_on_the_half_open_unit_interval():
    u = pti_synth.uniform_f32(0, 3, 1 << 20)
    assert u.dtype == np.float32 and u.min() >= 0.0 and u.max() < 1.0
    assert np.all(u * np.float32(2 ** 24) == np.floor(u * np.float32(2 ** 24)))   # 24-bit grid
    assert abs(float(u.astype(np.float64).mean()) - 0.5) < 0.002


def test_sample_batch_masks_but_keeps_token_zero():
    logits, u = pti_synth.sample_batch(6, 4, 500, seed=2, masked=0.9)
    assert logits.shape == (6, 4, 500) and u.shape == (6, 4)
    assert np.all(np.isfinite(logits[:, :, 0]))
    frac = np.isinf(logits).mean()
    assert 0.85 < frac < 0.95 and np.all(logits[np.isinf(logits)] < 0)
    plain, u2 = pti_synth.sample_batch(6, 4, 500, seed=2)
    assert np.array_equal(u, u2) and np.all(np.isfinite(plain))

"""GPU parity of the N-stream Q8 GEMV and the SSQ twin GEMV against the fp64 oracle.

Bar (per output element): |y_gpu - y_oracle| <= 1e-5 * sum_k |w_k x_k|, the
oracle's exact bound.  Special cases whose result is exact in fp32 (one-hot x,
integer weights and activations, zero weights, identical twins) are checked
bit for bit.  Inputs come from the seeded generator (pti_synth) only.
"""
import contextlib

import numpy as np
import pytest
import torch

import oracle
import pti_synth
import stream_quantized_gemv_gb300 as pti

pytestmark = pytest.mark.gpu

TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    pti.build()
    pti.lib()
    yield
    assert pti.device_error() == 0


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_parity(y_gpu, y_ref, bound, what=""):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(y_gpu - y_ref)
    bad = err > TOL * bound
    if bad.any():
        ratio = np.max(err / np.maximum(bound, 1e-300))
        raise AssertionError(f"{what}: {bad.sum()} outputs off, max err/bound {ratio:.3g}")


@contextlib.contextmanager
def all_cores():
    """The oracle's OpenMP build for the full-size checks (rows are independent,
    so its results equal the single-threaded build's bit for bit)."""
    oracle.use_all_cores(True)
    try:
        yield
    finally:
        oracle.use_all_cores(False)


def tile_sample_rows(rows, rng):
    """One row per 128-row tile (at a varying offset), plus the matrix ends."""
    idx = {0, rows - 1}
    for rb in range((rows + 127) // 128):
        idx.add(min(rows - 1, rb * 128 + (rb * 37) % 128))
    idx.update(rng.integers(0, rows, size=8).tolist())
    return np.array(sorted(idx), dtype=np.int64)


# ---------------------------------------------------------------------------
# Q8, small and ragged shapes (fast path: cols % 256 == 0; plain path otherwise)
# ---------------------------------------------------------------------------
Q8_SHAPES = [(256, 512), (1, 256), (33, 256), (200, 768), (129, 1024), (1000, 2048),
             (300, 96), (17, 544), (5, 32)]


@pytest.mark.parametrize("rows,cols", Q8_SHAPES)
@pytest.mark.parametrize("n", [1, 2, 3, 4])
def test_q8_small_shapes_match_oracle(rows, cols, n):
    w = pti_synth.q8_matrix(rows, cols, seed=rows * 7 + cols, tensor_id=n)
    x = pti_synth.activations(n, cols, seed=rows + cols, tensor_id=n)
    y_ref, bound = oracle.q8_gemv(w, rows, cols, x)
    y = pti.q8_gemv_nstream(dev(w), rows, cols, dev(x)).cpu().numpy()
    assert y.shape == (n, rows)
    assert_parity(y, y_ref, bound, f"q8 {rows}x{cols} n={n}")


def test_q8_is_bit_reproducible():
    rows, cols = 1000, 2048
    w = dev(pti_synth.q8_matrix(rows, cols, seed=1))
    x = dev(pti_synth.activations(4, cols, seed=1))
    a = pti.q8_gemv_nstream(w, rows, cols, x).clone()
    b = pti.q8_gemv_nstream(w, rows, cols, x).clone()
    assert torch.equal(a, b)


def test_q8_one_hot_is_exact():
    """x = e_j: every output is the single product d*q, exact in fp32."""
    rows, cols = 300, 512
    w = pti_synth.q8_matrix(rows, cols, seed=5)
    for j in (0, 1, 31, 32, 255, 256, 511):
        x = np.zeros((4, cols), np.float32)
        x[0, j] = 1.0
        x[1, (j + 1) % cols] = -1.0
        x[2, j] = 2.0
        x[3, (j + 100) % cols] = 0.5
        y_ref, _ = oracle.q8_gemv(w, rows, cols, x)
        y = pti.q8_gemv_nstream(dev(w), rows, cols, dev(x)).cpu().numpy().astype(np.float64)
        assert np.array_equal(y, y_ref), j


def test_q8_integer_case_is_exact():
    """Scales 1.0, integer x in [-4, 4]: |y| < 2^24 so any order is exact."""
    rows, cols = 257, 1024
    w = pti_synth.q8_matrix(rows, cols, seed=9).reshape(-1, 34).copy()
    w[:, 0], w[:, 1] = 0x00, 0x3C
    w = w.reshape(-1)
    xi = np.random.default_rng(2).integers(-4, 5, size=(4, cols)).astype(np.float32)
    y_ref, _ = oracle.q8_gemv(w, rows, cols, xi)
    y = pti.q8_gemv_nstream(dev(w), rows, cols, dev(xi)).cpu().numpy().astype(np.float64)
    assert np.array_equal(y, y_ref)


def test_q8_extreme_bytes_and_zero_weights():
    rows, cols = 130, 512
    w = pti_synth.q8_matrix(rows, cols, seed=3).reshape(-1, 34).copy()
    w[0::3, 2:] = 0x80           # q = -128 (representable, outside the generator's range)
    w[1::3, 2:] = 0x7F           # q = 127
    w[2::3, 2:] = 0x00           # q = 0
    w = w.reshape(-1)
    x = pti_synth.activations(3, cols, seed=3)
    y_ref, bound = oracle.q8_gemv(w, rows, cols, x)
    y = pti.q8_gemv_nstream(dev(w), rows, cols, dev(x)).cpu().numpy()
    assert_parity(y, y_ref, bound, "extreme bytes")


# ---------------------------------------------------------------------------
# Q8 at the configured full sizes, in the launch configuration the bench uses
# ---------------------------------------------------------------------------
@pytest.fixture(scope="module")
def full_q8():
    mats = {}
    for rows, cols in ((17408, 5120), (5120, 17408)):
        mats[(rows, cols)] = pti_synth.q8_matrix(rows, cols, seed=0, tensor_id=rows)
    return mats


@pytest.mark.parametrize("rows,cols", [(17408, 5120), (5120, 17408)])
def test_q8_full_size_matches_oracle_on_every_row(full_q8, rows, cols):
    w_np = full_q8[(rows, cols)]
    w = dev(w_np)
    for n in (1, 2, 3, 4):
        x = pti_synth.activations(n, cols, seed=0, tensor_id=100 + n)
        y = pti.q8_gemv_nstream(w, rows, cols, dev(x)).cpu().numpy()
        assert np.isfinite(y).all()
        with all_cores():
            y_ref, bound = oracle.q8_gemv(w_np, rows, cols, x)
        assert_parity(y, y_ref, bound, f"q8 {rows}x{cols} n={n}")


def test_q8_streams_are_independent_at_full_size(full_q8):
    """Stream s of an N-stream call equals the 1-stream call on x[s] within the bar."""
    rows, cols = 17408, 5120
    w_np = full_q8[(rows, cols)]
    w = dev(w_np)
    x = dev(pti_synth.activations(4, cols, seed=5))
    y4 = pti.q8_gemv_nstream(w, rows, cols, x).cpu().numpy()
    idx = np.arange(0, rows, 97)
    for s in range(4):
        y1 = pti.q8_gemv_nstream(w, rows, cols, x[s:s + 1].contiguous()).cpu().numpy()
        _, bound = oracle.q8_gemv(w_np, rows, cols, x[s:s + 1].cpu().numpy(), rows_idx=idx)
        assert np.all(np.abs(y4[s, idx].astype(np.float64) - y1[0, idx]) <= 2 * TOL * bound[0])


def test_q8_pdl_chain_reads_each_finished_output(full_q8):
    """y1 = W1 x, then y2 = W2 y1 and y3 = W1 y2 launched with FLAG_PDL: each
    may start while its predecessor still runs (prefetching weights), yet must
    read the predecessor's finished output and share its workspace safely."""
    a, b = full_q8[(17408, 5120)], full_q8[(5120, 17408)]
    wa, wb = dev(a), dev(b)
    x = dev(pti_synth.activations(4, 5120, seed=9))
    y1 = pti.q8_gemv_nstream(wa, 17408, 5120, x)
    y2 = pti.q8_gemv_nstream(wb, 5120, 17408, y1, flags=pti.FLAG_PDL)
    y3 = pti.q8_gemv_nstream(wa, 17408, 5120, y2, flags=pti.FLAG_PDL)
    torch.cuda.synchronize()
    y1n, y2n, y3n = y1.cpu().numpy(), y2.cpu().numpy(), y3.cpu().numpy()
    idx2 = tile_sample_rows(5120, np.random.default_rng(2))
    r2, b2 = oracle.q8_gemv(b, 5120, 17408, y1n, rows_idx=idx2)
    assert_parity(y2n[:, idx2], r2, b2, "pdl chain step 2")
    idx3 = tile_sample_rows(17408, np.random.default_rng(3))
    r3, b3 = oracle.q8_gemv(a, 17408, 5120, y2n, rows_idx=idx3)
    assert_parity(y3n[:, idx3], r3, b3, "pdl chain step 3")


# ---------------------------------------------------------------------------
# Q8 on the tensor core (PTI_FLAG_TENSOR_CORES): the same bar
# ---------------------------------------------------------------------------
TC = pti.FLAG_TENSOR_CORES
TC_SHAPES = [(256, 512), (1, 256), (33, 256), (200, 768), (129, 1024), (1000, 2048), (4096, 5120)]


@pytest.mark.parametrize("rows,cols", TC_SHAPES)
@pytest.mark.parametrize("n", [1, 2, 3, 4])
def test_tc_small_shapes_match_oracle(rows, cols, n):
    w = pti_synth.q8_matrix(rows, cols, seed=rows * 5 + cols, tensor_id=n)
    x = pti_synth.activations(n, cols, seed=rows + 3 * cols, tensor_id=n)
    y_ref, bound = oracle.q8_gemv(w, rows, cols, x)
    y = pti.q8_gemv_nstream(dev(w), rows, cols, dev(x), flags=TC).cpu().numpy()
    assert_parity(y, y_ref, bound, f"tc {rows}x{cols} n={n}")


def test_cuda_core_flag_is_the_default_path():
    """PTI_FLAG_CUDA_CORES selects the default consumer: bit-identical results."""
    rows, cols = 1000, 2048
    w = dev(pti_synth.q8_matrix(rows, cols, seed=13))
    for n in (1, 4):
        x = dev(pti_synth.activations(n, cols, seed=13, tensor_id=n))
        a = pti.q8_gemv_nstream(w, rows, cols, x).clone()
        b = pti.q8_gemv_nstream(w, rows, cols, x, flags=pti.FLAG_CUDA_CORES).clone()
        assert torch.equal(a, b)


def test_tc_exact_cases():
    """One-hot x, integer x with unit scales, extreme bytes: results exact in
    fp32 on the tensor core too (every product and partial sum is)."""
    rows, cols = 300, 512
    w = pti_synth.q8_matrix(rows, cols, seed=5)
    for j in (0, 1, 31, 32, 255, 256, 511):
        x = np.zeros((4, cols), np.float32)
        x[0, j], x[1, (j + 1) % cols], x[2, j], x[3, (j + 100) % cols] = 1.0, -1.0, 2.0, 0.5
        y_ref, _ = oracle.q8_gemv(w, rows, cols, x)
        y = pti.q8_gemv_nstream(dev(w), rows, cols, dev(x), flags=TC).cpu().numpy().astype(np.float64)
        assert np.array_equal(y, y_ref), j
    rows, cols = 257, 1024
    wi = pti_synth.q8_matrix(rows, cols, seed=9).reshape(-1, 34).copy()
    wi[:, 0], wi[:, 1] = 0x00, 0x3C
    wi[0::5, 2:] = 0x80
    wi[1::5, 2:] = 0x7F
    wi = wi.reshape(-1)
    xi = np.random.default_rng(2).integers(-4, 5, size=(4, cols)).astype(np.float32)
    y_ref, _ = oracle.q8_gemv(wi, rows, cols, xi)
    y = pti.q8_gemv_nstream(dev(wi), rows, cols, dev(xi), flags=TC).cpu().numpy().astype(np.float64)
    assert np.array_equal(y, y_ref)


def test_tc_activation_range():
    """The activation pieces are scaled per (block, stream): blocks of very
    different magnitude, spreads of 2^20 inside a block, zeros and
    subnormals stay within the bar."""
    rows, cols = 512, 2048
    w = pti_synth.q8_matrix(rows, cols, seed=11)
    x = pti_synth.activations(4, cols, seed=11).astype(np.float64)
    rng = np.random.default_rng(11)
    x[0] *= np.repeat(2.0 ** rng.integers(-60, 60, cols // 32), 32)    # block magnitudes 2^-60 .. 2^60
    x[1] *= 2.0 ** rng.integers(-20, 1, cols)                            # spread inside each block
    x[2, ::3] = 0.0
    x[2, 1::7] = 1e-40                                                   # fp32 subnormals
    x[3, :64] = 0.0                                                      # all-zero blocks
    x = x.astype(np.float32)
    y_ref, bound = oracle.q8_gemv(w, rows, cols, x)
    y = pti.q8_gemv_nstream(dev(w), rows, cols, dev(x), flags=TC).cpu().numpy()
    assert_parity(y, y_ref, bound, "tc activation range")


@pytest.mark.parametrize("rows,cols", [(17408, 5120), (5120, 17408)])
def test_tc_full_size_matches_oracle_on_every_row(full_q8, rows, cols):
    w_np = full_q8[(rows, cols)]
    w = dev(w_np)
    for n in (2, 4):
        x = pti_synth.activations(n, cols, seed=0, tensor_id=200 + n)
        y = pti.q8_gemv_nstream(w, rows, cols, dev(x), flags=TC).cpu().numpy()
        with all_cores():
            y_ref, bound = oracle.q8_gemv(w_np, rows, cols, x)
        assert_parity(y, y_ref, bound, f"tc {rows}x{cols} n={n}")


def test_tc_pdl_chain_and_bit_reproducible(full_q8):
    a, b = full_q8[(17408, 5120)], full_q8[(5120, 17408)]
    wa, wb = dev(a), dev(b)
    x = dev(pti_synth.activations(4, 5120, seed=19))
    y1 = pti.q8_gemv_nstream(wa, 17408, 5120, x, flags=TC)
    y2 = pti.q8_gemv_nstream(wb, 5120, 17408, y1, flags=TC | pti.FLAG_PDL)
    y2b = pti.q8_gemv_nstream(wb, 5120, 17408, y1, flags=TC | pti.FLAG_PDL)
    torch.cuda.synchronize()
    assert torch.equal(y2, y2b)
    idx2 = tile_sample_rows(5120, np.random.default_rng(4))
    r2, b2 = oracle.q8_gemv(b, 5120, 17408, y1.cpu().numpy(), rows_idx=idx2)
    assert_parity(y2.cpu().numpy()[:, idx2], r2, b2, "tc pdl chain")


# ---------------------------------------------------------------------------
# SSQ twin GEMV
# ---------------------------------------------------------------------------
def test_twin_256x512_seed0_matches_oracle():
    """The 256 x 512 twin case (16 blocks per row, 68 bytes each), seed 0."""
    rows, cols = 256, 512
    w = pti_synth.twin_matrix(rows, cols, seed=0)
    xa, xb = pti_synth.activations(2, cols, seed=0, tensor_id=1)
    ya_ref, yb_ref, ba, bb = oracle.twin_gemv(w, rows, cols, xa, xb)
    ya, yb = pti.ssq_twin_gemv(dev(w), rows, cols, dev(xa), dev(xb))
    assert_parity(ya.cpu().numpy(), ya_ref, ba, "twin A")
    assert_parity(yb.cpu().numpy(), yb_ref, bb, "twin B")


@pytest.mark.parametrize("rows,cols", [(1, 128), (3, 128), (130, 384), (129, 2048), (64, 96), (7, 224)])
def test_twin_small_shapes_match_oracle(rows, cols):
    w = pti_synth.twin_matrix(rows, cols, seed=rows + cols, tensor_id=2)
    xa, xb = pti_synth.activations(2, cols, seed=cols, tensor_id=3)
    ya_ref, yb_ref, ba, bb = oracle.twin_gemv(w, rows, cols, xa, xb)
    ya, yb = pti.ssq_twin_gemv(dev(w), rows, cols, dev(xa), dev(xb))
    assert_parity(ya.cpu().numpy(), ya_ref, ba, f"twin A {rows}x{cols}")
    assert_parity(yb.cpu().numpy(), yb_ref, bb, f"twin B {rows}x{cols}")


def test_twin_one_hot_is_exact_and_uses_high_byte_for_a():
    rows, cols = 200, 256
    w = pti_synth.twin_matrix(rows, cols, seed=4)
    for j in (0, 1, 30, 31, 32, 127, 128, 255):
        e = np.zeros(cols, np.float32)
        e[j] = 1.0
        f = np.zeros(cols, np.float32)
        f[(j + 5) % cols] = -2.0
        ya_ref, yb_ref, _, _ = oracle.twin_gemv(w, rows, cols, e, f)
        ya, yb = pti.ssq_twin_gemv(dev(w), rows, cols, dev(e), dev(f))
        assert np.array_equal(ya.cpu().numpy().astype(np.float64), ya_ref), j
        assert np.array_equal(yb.cpu().numpy().astype(np.float64), yb_ref), j


@pytest.fixture(scope="module")
def full_twin():
    return {(r, c): pti_synth.twin_matrix(r, c, seed=0, tensor_id=r) for r, c in ((17408, 5120), (5120, 17408))}


@pytest.mark.parametrize("rows,cols", [(17408, 5120), (5120, 17408)])
def test_twin_full_size_matches_oracle_on_every_row(full_twin, rows, cols):
    w_np = full_twin[(rows, cols)]
    xa, xb = pti_synth.activations(2, cols, seed=0, tensor_id=200)
    ya, yb = pti.ssq_twin_gemv(dev(w_np), rows, cols, dev(xa), dev(xb))
    with all_cores():
        ya_ref, yb_ref, ba, bb = oracle.twin_gemv(w_np, rows, cols, xa, xb)
    assert_parity(ya.cpu().numpy(), ya_ref, ba, "twin A full")
    assert_parity(yb.cpu().numpy(), yb_ref, bb, "twin B full")


def test_twin_pdl_chain_reads_each_finished_output(full_twin):
    """(y_A, y_B) of a 17408 x 5120 twin GEMV feed a 5120 x 17408 twin GEMV
    launched with FLAG_PDL."""
    a, b = full_twin[(17408, 5120)], full_twin[(5120, 17408)]
    xa, xb = pti_synth.activations(2, 5120, seed=0, tensor_id=300)
    ya, yb = pti.ssq_twin_gemv(dev(a), 17408, 5120, dev(xa), dev(xb))
    za, zb = pti.ssq_twin_gemv(dev(b), 5120, 17408, ya, yb, flags=pti.FLAG_PDL)
    torch.cuda.synchronize()
    idx = tile_sample_rows(5120, np.random.default_rng(4))
    ra, rb, ba, bb = oracle.twin_gemv(b, 5120, 17408, ya.cpu().numpy(), yb.cpu().numpy(), rows_idx=idx)
    assert_parity(za.cpu().numpy()[idx], ra, ba, "twin pdl chain A")
    assert_parity(zb.cpu().numpy()[idx], rb, bb, "twin pdl chain B")


@pytest.mark.parametrize("rows,cols", [(17408, 5120), (5120, 17408)])
def test_identical_twins_give_identical_outputs(rows, cols):
    """A == B and x_A == x_B: y_A == y_B bit for bit, and both match the oracle."""
    w_np = pti_synth.twin_matrix(rows, cols, seed=1, tensor_id=7, identical=True)
    x = pti_synth.activations(1, cols, seed=1, tensor_id=8)[0]
    xd = dev(x)
    ya, yb = pti.ssq_twin_gemv(dev(w_np), rows, cols, xd, xd)
    assert torch.equal(ya, yb)
    idx = np.arange(0, rows, 211)
    ya_ref, _, ba, _ = oracle.twin_gemv(w_np, rows, cols, x, x, rows_idx=idx)
    assert_parity(ya.cpu().numpy()[idx], ya_ref, ba, "identical twins")


@pytest.mark.parametrize("rows,cols", [(1, 128), (130, 384), (256, 512), (1000, 2048), (7, 224)])
@pytest.mark.parametrize("n", [1, 2])
def test_twin_nstream_matches_oracle(rows, cols, n):
    """n streams per model: every stream of A and of B matches the oracle's twin
    GEMV on that stream pair (fast path for cols % 128 == 0, plain otherwise)."""
    w = pti_synth.twin_matrix(rows, cols, seed=rows + n)
    xa = pti_synth.activations(n, cols, seed=rows + n, tensor_id=1)
    xb = pti_synth.activations(n, cols, seed=rows + n, tensor_id=2)
    ya, yb = pti.ssq_twin_gemv_nstream(dev(w), rows, cols, dev(xa), dev(xb))
    ya, yb = ya.cpu().numpy(), yb.cpu().numpy()
    for s in range(n):
        ra, rb, ba, bb = oracle.twin_gemv(w, rows, cols, xa[s], xb[s])
        assert_parity(ya[s], ra, ba, f"A stream {s}")
        assert_parity(yb[s], rb, bb, f"B stream {s}")


@pytest.mark.parametrize("rows,cols", [(17408, 5120), (5120, 17408)])
def test_twin_two_streams_per_model_full_size(full_twin, rows, cols):
    """Four tokens per weight load: two streams of each twin at full size,
    every row checked; stream 0 equals the one-stream call within the bar."""
    w_np = full_twin[(rows, cols)]
    w = dev(w_np)
    xa = pti_synth.activations(2, cols, seed=0, tensor_id=400)
    xb = pti_synth.activations(2, cols, seed=0, tensor_id=401)
    ya, yb = pti.ssq_twin_gemv_nstream(w, rows, cols, dev(xa), dev(xb))
    ya, yb = ya.cpu().numpy(), yb.cpu().numpy()
    for s in range(2):
        with all_cores():
            ra, rb, ba, bb = oracle.twin_gemv(w_np, rows, cols, xa[s], xb[s])
        assert_parity(ya[s], ra, ba, f"A stream {s}")
        assert_parity(yb[s], rb, bb, f"B stream {s}")
    idx = tile_sample_rows(rows, np.random.default_rng(rows + 2))
    y1a, y1b = pti.ssq_twin_gemv(w, rows, cols, dev(xa[0]), dev(xb[0]))
    _, _, ba, bb = oracle.twin_gemv(w_np, rows, cols, xa[0], xb[0], rows_idx=idx)
    assert np.all(np.abs(ya[0, idx].astype(np.float64) - y1a.cpu().numpy()[idx]) <= 2 * TOL * ba)
    assert np.all(np.abs(yb[0, idx].astype(np.float64) - y1b.cpu().numpy()[idx]) <= 2 * TOL * bb)


def test_twin_two_streams_identical_twins_and_streams():
    """A == B and x_A[s] == x_B[s]: y_A[s] == y_B[s] bit for bit for both streams."""
    rows, cols = 1000, 2048
    w = pti_synth.twin_matrix(rows, cols, seed=3, tensor_id=9, identical=True)
    x = pti_synth.activations(2, cols, seed=3, tensor_id=10)
    ya, yb = pti.ssq_twin_gemv_nstream(dev(w), rows, cols, dev(x), dev(x))
    assert torch.equal(ya, yb)


def test_twin_matches_q8_on_unpacked_models():
    """Cross-kernel: twin(T, x_a, x_b) agrees with the Q8 GEMV of each unpacked model."""
    rows, cols = 520, 1024
    t = pti_synth.twin_matrix(rows, cols, seed=12)
    qa, qb = oracle.twin_unpack(t)
    xa, xb = pti_synth.activations(2, cols, seed=12)
    ya, yb = pti.ssq_twin_gemv(dev(t), rows, cols, dev(xa), dev(xb))
    ra = pti.q8_gemv_nstream(dev(qa), rows, cols, dev(xa[None])).cpu().numpy()[0]
    rb = pti.q8_gemv_nstream(dev(qb), rows, cols, dev(xb[None])).cpu().numpy()[0]
    _, _, ba, bb = oracle.twin_gemv(t, rows, cols, xa, xb)
    assert np.all(np.abs(ya.cpu().numpy().astype(np.float64) - ra) <= 2 * TOL * ba)
    assert np.all(np.abs(yb.cpu().numpy().astype(np.float64) - rb) <= 2 * TOL * bb)


def test_workspace_needs_no_initialisation():
    """The workspace is scratch: three calls in a row on one workspace filled
    with 0xFF bytes (NaN patterns) all match the oracle."""
    rows, cols = 1000, 2048
    need = pti.q8_gemv_workspace_bytes(rows, cols, 4)
    ws = torch.full((need,), 255, dtype=torch.uint8, device="cuda")
    w_np = pti_synth.q8_matrix(rows, cols, seed=2)
    w = dev(w_np)
    for k in range(3):
        x = pti_synth.activations(4, cols, seed=20 + k)
        y = pti.q8_gemv_nstream(w, rows, cols, dev(x), ws=ws).cpu().numpy()
        y_ref, bound = oracle.q8_gemv(w_np, rows, cols, x)
        assert_parity(y, y_ref, bound, f"call {k}")


def test_one_workspace_serves_every_shape_and_stream_count():
    """One workspace shared, in turn, by Q8 calls of different shapes and stream
    counts and by twin calls: every call matches the oracle."""
    ws = torch.full((pti.q8_gemv_workspace_bytes(5120, 17408, 4),), 255, dtype=torch.uint8, device="cuda")
    cases = [("q8", 1000, 2048, 4), ("q8", 520, 1024, 1), ("twin", 520, 1024, 2), ("q8", 1000, 2048, 2),
             ("twin", 1000, 2048, 2), ("q8", 520, 1024, 3), ("q8", 1000, 2048, 1)]
    for k, (kind, rows, cols, n) in enumerate(cases):
        if kind == "q8":
            w = pti_synth.q8_matrix(rows, cols, seed=40 + k)
            x = pti_synth.activations(n, cols, seed=40 + k)
            y = pti.q8_gemv_nstream(dev(w), rows, cols, dev(x), ws=ws).cpu().numpy()
            y_ref, bound = oracle.q8_gemv(w, rows, cols, x)
            assert_parity(y, y_ref, bound, f"case {k}")
        else:
            w = pti_synth.twin_matrix(rows, cols, seed=40 + k)
            xa, xb = pti_synth.activations(2, cols, seed=40 + k)
            ya, yb = pti.ssq_twin_gemv(dev(w), rows, cols, dev(xa), dev(xb), ws=ws)
            ra, rb, ba, bb = oracle.twin_gemv(w, rows, cols, xa, xb)
            assert_parity(ya.cpu().numpy(), ra, ba, f"case {k} A")
            assert_parity(yb.cpu().numpy(), rb, bb, f"case {k} B")


def test_unaligned_activations_take_the_plain_path():
    """x offset by 4 bytes (not 16-byte aligned): still correct."""
    rows, cols = 300, 1024
    w = pti_synth.q8_matrix(rows, cols, seed=77)
    x = pti_synth.activations(2, cols, seed=77)
    buf = torch.empty(2 * cols + 1, dtype=torch.float32, device="cuda")
    xv = buf[1:].view(2, cols)
    xv.copy_(dev(x))
    y = pti.q8_gemv_nstream(dev(w), rows, cols, xv).cpu().numpy()
    y_ref, bound = oracle.q8_gemv(w, rows, cols, x)
    assert_parity(y, y_ref, bound, "unaligned x")

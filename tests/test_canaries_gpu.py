"""Guard canaries: every output buffer sits between two guard regions filled
with a known byte pattern, and no call may write outside its documented
extent (fast and plain GEMV paths, twin GEMV, both verify kernels, the
decode pass, the self-speculative loop with a token capacity smaller than
what it confirms)."""
import numpy as np
import pytest
import torch

import pti_synth
import stream_quantized_gemv_gb300 as pti

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side
PATTERN = 0xA5


def guarded(shape, dtype):
    """A tensor of `shape` inside a byte buffer with GUARD canary bytes before
    and after it (the tensor starts 256-byte aligned)."""
    n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
    buf = torch.full((GUARD + n + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
    t = buf[GUARD:GUARD + n].view(dtype).view(*shape)
    return buf, t


def intact(buf):
    torch.cuda.synchronize()
    g = torch.cat([buf[:GUARD], buf[-GUARD:]]).cpu().numpy()
    return bool(np.all(g == PATTERN))


def up(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("rows,cols,n", [(384, 1024, 4), (17, 512, 3), (100, 96, 2)])
def test_q8_gemv_writes_only_y(rows, cols, n):
    w = up(pti_synth.q8_matrix(rows, cols, seed=3))
    x = up(pti_synth.activations(n, cols, seed=3))
    buf, y = guarded((n, rows), torch.float32)
    pti.q8_gemv_nstream(w, rows, cols, x, y=y)
    assert intact(buf)
    assert torch.isfinite(y).all()


def test_twin_gemv_writes_only_ya_yb():
    rows, cols = 256, 512
    w = up(pti_synth.twin_matrix(rows, cols, seed=0))
    xa, xb = (up(v) for v in pti_synth.activations(2, cols, seed=0, tensor_id=1))
    ba, ya = guarded((rows,), torch.float32)
    bb, yb = guarded((rows,), torch.float32)
    pti.ssq_twin_gemv(w, rows, cols, xa, xb, y_a=ya, y_b=yb)
    assert intact(ba) and intact(bb)


def test_verify_kernels_write_only_their_outputs():
    steps, n, vocab = 8, 4, 1000
    lg, gs, _ = pti_synth.verify_batch(steps, n, vocab, 0.6, seed=2)
    b1, a = guarded((steps, n), torch.int32)
    b2, m = guarded((steps, n - 1), torch.uint8)
    b3, c = guarded((steps,), torch.int32)
    pti.verify_greedy(up(lg), up(gs), argmax=a, match=m, accept=c)
    assert intact(b1) and intact(b2) and intact(b3)
    lg2, u = pti_synth.sample_batch(steps, n, vocab, seed=4)
    b4, t = guarded((steps, n), torch.int32)
    b5, m2 = guarded((steps, n - 1), torch.uint8)
    b6, c2 = guarded((steps,), torch.int32)
    pti.verify_sample(up(lg2), up(gs), up(u), 0.8, token=t, match=m2, accept=c2)
    assert intact(b4) and intact(b5) and intact(b6)


def test_decode_pass_writes_only_x_out():
    hidden, ffn, n = 256, 512, 4
    wg, wu = up(pti_synth.q8_matrix(ffn, hidden, 5, 0)), up(pti_synth.q8_matrix(ffn, hidden, 5, 1))
    wd = up(pti_synth.q8_matrix(hidden, ffn, 5, 2))
    x = up(pti_synth.activations(n, hidden, 5, 1000))
    buf, xo = guarded((n, hidden), torch.float32)
    pti.mlp_decode_pass(pti.DecodeWeights([wg], [wu], [wd]), hidden, ffn, x, x_out=xo)
    assert intact(buf)


def test_selfspec_stops_at_its_token_capacity():
    V, H, F, n, steps, cap = 512, 256, 256, 4, 12, 7
    m = pti_synth.toy_model(V, H, F, seed=11)
    dev = {k: up(m[k]) for k in ("embedding", "w_gate", "w_up", "w_down", "w_head")}
    bt, tokens = guarded((cap,), torch.int32)
    bc, count = guarded((1,), torch.int32)
    ba, accept = guarded((steps,), torch.int32)
    pti.selfspec_greedy(dev["embedding"], dev["w_gate"], dev["w_up"], dev["w_down"], dev["w_head"], V, H, F, n,
                        13, steps, capacity=cap, out=(tokens, count, accept))
    assert intact(bt) and intact(bc) and intact(ba)
    assert int(count.item()) >= steps > cap   # more confirmed than stored

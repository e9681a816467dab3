"""The C-ABI library builds, loads and exports every entry point of include/pti.h,
and its host-side argument checks reject bad calls before touching a GPU.

Every call here fails validation, so no kernel is ever launched (safe with or
without a GPU; fake pointer values are never dereferenced).
"""
import ctypes
import os
import re

import pytest

import stream_quantized_gemv_gb300 as pti

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    pti.build()
    return pti.lib()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "pti.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pti_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_documented_entry_points():
    names = _declared_functions()
    for required in ("pti_q8_gemv_nstream", "pti_ssq_twin_gemv", "pti_verify_greedy", "pti_verify_sample",
                     "pti_status_string", "pti_device_error"):
        assert required in names


def test_library_exports_every_declared_symbol(L):
    for name in _declared_functions():
        assert hasattr(L, name), name


def test_status_strings(L):
    for code, name in pti.STATUS_NAMES.items():
        assert L.pti_status_string(code).decode().startswith(name)
    assert L.pti_status_string(99).decode() == "PTI_ERR_UNKNOWN"


def test_workspace_queries(L):
    # fast paths need a workspace, plain paths do not, invalid shapes report 0
    assert L.pti_q8_gemv_workspace_bytes(17408, 5120, 4) > 0
    assert L.pti_q8_gemv_workspace_bytes(5120, 17408, 1) > 0
    assert L.pti_q8_gemv_workspace_bytes(100, 96, 2) == 0
    assert L.pti_q8_gemv_workspace_bytes(100, 256, 5) == 0
    assert L.pti_q8_gemv_workspace_bytes(0, 256, 1) == 0
    assert L.pti_ssq_twin_gemv_workspace_bytes(256, 512) > 0
    assert L.pti_ssq_twin_gemv_workspace_bytes(256, 96) == 0
    assert L.pti_q8_gemv_workspace_bytes(17408, 5120, 4) % 256 == 0


FAKE = 0x7F0000000000  # 256-byte aligned, never dereferenced


def _q8(L, w=FAKE, rows=128, cols=512, n=2, x=FAKE + (1 << 30), y=FAKE + (2 << 30),
        ws=FAKE + (3 << 30), ws_bytes=1 << 24):
    return L.pti_q8_gemv_nstream(w, rows, cols, n, x, y, ws, ws_bytes, None)


def test_q8_validation(L):
    assert _q8(L, w=None) == 1 and _q8(L, x=None) == 1 and _q8(L, y=None) == 1
    assert _q8(L, rows=0) == 2 and _q8(L, cols=0) == 2 and _q8(L, cols=48) == 2
    assert _q8(L, cols=16) == 2 and _q8(L, rows=1 << 32) == 2
    assert _q8(L, n=0) == 3 and _q8(L, n=5) == 3
    assert _q8(L, w=FAKE + 8) == 4 and _q8(L, x=FAKE + (1 << 30) + 2) == 4
    assert _q8(L, y=FAKE + 4) == 5                      # y overlaps w
    assert _q8(L, y=FAKE + (1 << 30) + 64) == 5          # y overlaps x
    assert _q8(L, ws=None) == 7 and _q8(L, ws_bytes=16) == 7
    assert _q8(L, ws=FAKE + (3 << 30) + 16) == 4
    assert _q8(L, ws=FAKE + 256) == 5                    # workspace overlaps w


def _twin(L, w=FAKE, rows=128, cols=512, xa=FAKE + (1 << 30), xb=FAKE + (1 << 30),
          ya=FAKE + (2 << 30), yb=FAKE + (2 << 30) + 4096, ws=FAKE + (3 << 30), ws_bytes=1 << 24):
    return L.pti_ssq_twin_gemv(w, rows, cols, xa, xb, ya, yb, ws, ws_bytes, None)


def test_twin_validation(L):
    assert _twin(L, w=None) == 1 and _twin(L, xb=None) == 1 and _twin(L, ya=None) == 1
    assert _twin(L, rows=-1) == 2 and _twin(L, cols=33) == 2
    assert _twin(L, w=FAKE + 4) == 4 and _twin(L, yb=FAKE + (2 << 30) + 4098) == 4
    assert _twin(L, yb=FAKE + (2 << 30) + 8) == 5       # y_a and y_b overlap
    assert _twin(L, ya=FAKE + 1024) == 5                # y_a overlaps w
    assert _twin(L, ws=None) == 7


def _verify(L, logits=FAKE, guess=FAKE + (1 << 34), steps=4, n=4, vocab=1000,
            am=FAKE + (2 << 34), m=FAKE + (3 << 34), acc=FAKE + (4 << 34)):
    return L.pti_verify_greedy(logits, guess, steps, n, vocab, am, m, acc, None)


def test_verify_validation(L):
    assert _verify(L, n=0) == 3 and _verify(L, n=5) == 3
    assert _verify(L, steps=-1) == 2 and _verify(L, vocab=0) == 2 and _verify(L, vocab=1 << 31) == 2
    assert _verify(L, logits=None) == 1 and _verify(L, m=None) == 1 and _verify(L, acc=None) == 1
    assert _verify(L, logits=FAKE + 2) == 4 and _verify(L, am=FAKE + (2 << 34) + 1) == 4
    assert _verify(L, am=FAKE + 64) == 5                 # argmax overlaps logits
    assert _verify(L, acc=FAKE + (2 << 34) + 4) == 5     # accept overlaps argmax


def _sample(L, logits=FAKE, guess=FAKE + (1 << 34), uniform=FAKE + (11 << 34), steps=4, n=4, vocab=1000,
            temperature=0.8, tok=FAKE + (2 << 34), m=FAKE + (3 << 34), acc=FAKE + (4 << 34),
            col=FAKE + (12 << 34)):
    return L.pti_verify_sample(logits, guess, uniform, steps, n, vocab, temperature, tok, m, acc, col, None)


def test_verify_sample_validation(L):
    """Every call below fails validation, so nothing is launched."""
    assert _sample(L, n=0) == 3 and _sample(L, n=5) == 3
    assert _sample(L, steps=-1) == 2 and _sample(L, vocab=0) == 2 and _sample(L, vocab=1 << 31) == 2
    for bad in (0.0, -1.0, float("inf"), float("nan"), 1e-45):
        assert _sample(L, temperature=bad) == 8, bad
    assert _sample(L, temperature=0.0, steps=0) == 8      # scalars are checked even for no steps
    assert _sample(L, uniform=None) == 1 and _sample(L, tok=None) == 1 and _sample(L, m=None) == 1
    assert _sample(L, acc=None) == 1 and _sample(L, logits=None) == 1 and _sample(L, guess=None) == 1
    assert _sample(L, uniform=FAKE + (11 << 34) + 2) == 4 and _sample(L, col=FAKE + (12 << 34) + 1) == 4
    assert _sample(L, tok=FAKE + 64) == 5                  # token overlaps logits
    assert _sample(L, col=FAKE + (11 << 34) + 8) == 5      # collision overlaps uniform
    assert _sample(L, m=FAKE + (2 << 34) + 8) == 5         # match overlaps token
    assert _sample(L, acc=FAKE + (12 << 34) + 4) == 5      # accept overlaps collision


def _ptrs(*vals):
    return (ctypes.c_void_p * len(vals))(*vals)


GATE, UP, DOWN = FAKE + (5 << 34), FAKE + (6 << 34), FAKE + (7 << 34)


def _decode(L, gate=None, up=None, down=None, layers=2, hidden=512, ffn=1024, n=4, eps=1e-6,
            x_in=FAKE + (8 << 34), x_out=FAKE + (9 << 34), ws=FAKE + (10 << 34), ws_bytes=1 << 26):
    gate = _ptrs(GATE, GATE + (1 << 30)) if gate is None else gate
    up = _ptrs(UP, UP + (1 << 30)) if up is None else up
    down = _ptrs(DOWN, DOWN + (1 << 30)) if down is None else down
    return L.pti_mlp_decode_pass(gate, up, down, layers, hidden, ffn, n, eps, x_in, x_out, ws, ws_bytes, None)


def test_decode_pass_workspace_query(L):
    need = L.pti_mlp_decode_pass_workspace_bytes(5120, 17408, 4)
    # stream-K partials, h, the raw layer output and the sums of squares
    assert need >= 320 * 2 * 4 * 128 * 4 + 4 * 17408 * 4 + 4 * 5120 * 4 and need % 256 == 0
    assert L.pti_mlp_decode_pass_workspace_bytes(5120, 17408, 1) < need
    assert L.pti_mlp_decode_pass_workspace_bytes(5000, 17408, 4) == 0      # hidden % 256
    assert L.pti_mlp_decode_pass_workspace_bytes(5120, 100, 4) == 0
    assert L.pti_mlp_decode_pass_workspace_bytes(5120, 17408, 5) == 0


def test_decode_pass_validation(L):
    """Every call below fails validation, so nothing is launched."""
    ok_bytes = L.pti_mlp_decode_pass_workspace_bytes(512, 1024, 4)
    assert ok_bytes > 0
    assert _decode(L, x_in=None) == 1 and _decode(L, x_out=None) == 1
    assert _decode(L, gate=_ptrs(GATE, None)) == 1
    assert L.pti_mlp_decode_pass(None, _ptrs(UP), _ptrs(DOWN), 1, 512, 1024, 4, 1e-6,
                                 FAKE, FAKE + (1 << 30), FAKE + (2 << 30), 1 << 26, None) == 1
    assert _decode(L, layers=0) == 2 and _decode(L, hidden=500) == 2 and _decode(L, ffn=1000) == 2
    assert _decode(L, hidden=128) == 2
    assert _decode(L, n=0) == 3 and _decode(L, n=5) == 3
    assert _decode(L, eps=-1.0) == 8 and _decode(L, eps=float("nan")) == 8 and _decode(L, eps=float("inf")) == 8
    assert _decode(L, down=_ptrs(DOWN, DOWN + 8)) == 4          # weight not 16-byte aligned
    assert _decode(L, x_in=FAKE + (8 << 34) + 4) == 4           # x_in needs 16 bytes
    assert _decode(L, x_out=FAKE + (9 << 34) + 2) == 4
    assert _decode(L, ws=None) == 7 and _decode(L, ws_bytes=ok_bytes - 1) == 7
    assert _decode(L, ws=FAKE + (10 << 34) + 16) == 4
    assert _decode(L, x_out=GATE + (1 << 30) + 64) == 5         # x_out inside layer 1's gate matrix
    assert _decode(L, ws=UP) == 5                                # workspace overlaps a weight matrix
    assert _decode(L, ws=FAKE + (8 << 34) - 256) == 5           # workspace overlaps x_in


def test_ex_entry_points_reject_unknown_flags(L):
    """The _ex variants validate like the plain ones and reject unknown flag bits."""
    args = (FAKE, 128, 512, 2, FAKE + (1 << 30), FAKE + (2 << 30), FAKE + (3 << 30), 1 << 24, None)
    assert L.pti_q8_gemv_nstream_ex(*args, 8) == 8 and L.pti_q8_gemv_nstream_ex(*args, 0x80000000) == 8
    # the two consumer choices exclude each other
    assert L.pti_q8_gemv_nstream_ex(*args, pti.FLAG_CUDA_CORES | pti.FLAG_TENSOR_CORES) == 8
    assert L.pti_q8_gemv_nstream_ex(None, *args[1:], pti.FLAG_TENSOR_CORES) == 1
    assert L.pti_q8_gemv_nstream_ex(None, *args[1:], 1) == 1
    assert L.pti_q8_gemv_nstream_ex(FAKE, 128, 48, *args[3:], 1) == 2
    targs = (FAKE, 128, 512, FAKE + (1 << 30), FAKE + (1 << 30), FAKE + (2 << 30), FAKE + (2 << 30) + 4096,
             FAKE + (3 << 30), 1 << 24, None)
    assert L.pti_ssq_twin_gemv_ex(*targs, 8) == 8
    # the twin GEMV has one consumer: the core choice is a Q8 flag
    assert L.pti_ssq_twin_gemv_ex(*targs, pti.FLAG_CUDA_CORES) == 8
    assert L.pti_ssq_twin_gemv_ex(*targs, pti.FLAG_TENSOR_CORES) == 8
    assert L.pti_ssq_twin_gemv_ex(None, *targs[1:], 1) == 1


def test_decode_pass_layer_count(L):
    ok_bytes = L.pti_mlp_decode_pass_workspace_bytes(512, 1024, 4)
    gate, up, down = _ptrs(GATE), _ptrs(UP), _ptrs(DOWN)
    args = (512, 1024, 4, 1e-6, FAKE + (8 << 34), FAKE + (9 << 34), FAKE + (10 << 34), ok_bytes, None)
    assert L.pti_mlp_decode_pass(gate, up, down, 0, *args) == 2
    assert L.pti_mlp_decode_pass(gate, up, down, 4097, *args) == 2


def test_stall_hook_validation(L):
    """The testing hook checks its arguments like the GEMV (nothing launched)."""
    x, y, ws = FAKE + (1 << 30), FAKE + (2 << 30), FAKE + (3 << 30)

    def call(w=FAKE, rows=1024, cols=512, n=2, x=x, y=y, ws=ws, ws_bytes=1 << 24, stall=8, wait=10 ** 6, flags=0):
        return L.pti_test_q8_gemv_stall(w, rows, cols, n, x, y, ws, ws_bytes, None, stall, wait, flags)

    assert call(w=None) == 1 and call(ws=None) == 1
    assert call(cols=96) == 2 and call(cols=128) == 2           # the hook needs the fast path
    assert call(n=5) == 3
    assert call(x=x + 4) == 4 and call(ws=ws + 16) == 4
    assert call(ws_bytes=256) == 7
    assert call(wait=999) == 8 and call(wait=3 * 10 ** 9) == 8
    assert call(flags=pti.FLAG_CUDA_CORES | pti.FLAG_TENSOR_CORES) == 8 and call(flags=pti.FLAG_PDL) == 8


def test_twin_nstream_validation(L):
    args = (FAKE, 128, 512)
    xa, xb, ya, yb = FAKE + (1 << 30), FAKE + (1 << 30) + 4096, FAKE + (2 << 30), FAKE + (2 << 30) + 8192
    assert L.pti_ssq_twin_gemv_nstream(*args, 0, xa, xb, ya, yb, FAKE + (3 << 30), 1 << 24, None, 0) == 3
    assert L.pti_ssq_twin_gemv_nstream(*args, 3, xa, xb, ya, yb, FAKE + (3 << 30), 1 << 24, None, 0) == 3
    assert L.pti_ssq_twin_gemv_nstream(*args, 2, xa, xb, ya, yb, FAKE + (3 << 30), 1 << 24, None, 8) == 8
    assert L.pti_ssq_twin_gemv_nstream(*args, 2, xa, xb, ya, ya + 512, FAKE + (3 << 30), 1 << 24, None, 0) == 5
    assert L.pti_ssq_twin_gemv_nstream(*args, 2, xa, xb, ya, yb, None, 0, None, 0) == 7
    assert L.pti_ssq_twin_gemv_nstream_workspace_bytes(128, 512, 2) > L.pti_ssq_twin_gemv_nstream_workspace_bytes(128, 512, 1)
    assert L.pti_ssq_twin_gemv_nstream_workspace_bytes(128, 512, 3) == 0


def _toy(emb=FAKE, gate=FAKE + (1 << 30), up=FAKE + (2 << 30), down=FAKE + (3 << 30), head=FAKE + (4 << 30),
         vocab=512, hidden=256, ffn=256, eps=1e-6):
    return pti.ToyModel(emb, gate, up, down, head, vocab, hidden, ffn, eps)


def test_selfspec_validation(L):
    """The self-speculative loop validates everything before its first launch."""
    need = L.pti_selfspec_greedy_workspace_bytes(512, 256, 256, 4)
    assert need > 0 and need % 256 == 0
    assert L.pti_selfspec_greedy_workspace_bytes(1, 256, 256, 4) == 0
    assert L.pti_selfspec_greedy_workspace_bytes(512, 100, 256, 4) == 0
    assert L.pti_selfspec_greedy_workspace_bytes(512, 256, 256, 5) == 0
    out, cnt, acc, ws = FAKE + (8 << 34), FAKE + (9 << 34), FAKE + (10 << 34), FAKE + (11 << 34)

    def call(model=None, n=4, first=3, steps=8, tokens=out, cap=32, count=cnt, accept=acc, w=ws, wb=need):
        m = _toy() if model is None else model
        return L.pti_selfspec_greedy(ctypes.byref(m), n, first, steps, tokens, cap, count, accept, w, wb, None)

    assert L.pti_selfspec_greedy(None, 4, 3, 8, out, 32, cnt, acc, ws, need, None) == 1
    assert call(model=_toy(emb=None)) == 1 and call(model=_toy(head=None)) == 1
    assert call(count=None) == 1 and call(w=None) == 1 and call(tokens=None) == 1
    assert call(n=0) == 3 and call(n=5) == 3
    assert call(steps=-1) == 2 and call(steps=(1 << 28) + 1) == 2 and call(cap=-1) == 2
    assert call(model=_toy(vocab=1)) == 2 and call(model=_toy(hidden=100)) == 2
    assert call(first=-1) == 8 and call(first=512) == 8
    assert call(model=_toy(eps=-1.0)) == 8 and call(model=_toy(eps=float("nan"))) == 8
    assert call(model=_toy(emb=FAKE + 4)) == 4 and call(model=_toy(down=FAKE + (3 << 30) + 8)) == 4
    assert call(w=ws + 16) == 4 and call(count=cnt + 2) == 4
    assert call(wb=need - 1) == 7
    assert call(w=FAKE + (4 << 30)) == 5                  # workspace over the LM head
    assert call(tokens=FAKE + 64) == 5                     # tokens inside the embedding table
    assert call(count=out + 8) == 5                        # count inside the token buffer

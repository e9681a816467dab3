"""Plain fp64 CPU oracle for the Packed Twin Inference hot path.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product path (``stream_quantized_gemv_gb300``) never imports it, and this
package never imports the product path: the two share no code.

The arithmetic lives in ``pti_oracle.c`` (plain C99, double precision); this
module compiles it with gcc and wraps it with ctypes, converting numpy arrays
to pointers.  Every function cites the passage it follows in the C source.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_SOURCES = [os.path.join(_HERE, "pti_oracle.c")]
_HEADERS = [os.path.join(_HERE, "pti_oracle.h")]

_lib = None
_lock = threading.Lock()

Q8_BLOCK_BYTES = 34
TWIN_BLOCK_BYTES = 68
BLOCK_COLS = 32


_OMP_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_omp.so")


def _stale_lib(path: str) -> bool:
    if not os.path.exists(path):
        return True
    built = os.path.getmtime(path)
    return any(os.path.getmtime(p) > built for p in _SOURCES + _HEADERS)


def _compile(path: str, extra: list[str]) -> None:
    os.makedirs(_BUILD_DIR, exist_ok=True)
    tmp = path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-Wall", "-Wextra", *extra,
           "-o", tmp] + _SOURCES + ["-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, path)


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (plain gcc, -O2),
    and, where gcc supports OpenMP, the same source with the row loops split
    over the host's cores into ``liboracle_omp.so`` (used only to time the
    CPU baseline on all cores)."""
    if force or _stale_lib(_LIB_PATH):
        _compile(_LIB_PATH, ["-Wno-unknown-pragmas"])
    if force or _stale_lib(_OMP_LIB_PATH):
        try:
            _compile(_OMP_LIB_PATH, ["-fopenmp"])
        except (subprocess.CalledProcessError, OSError):
            pass
    return _LIB_PATH


def has_all_cores() -> bool:
    """True when the OpenMP build of the oracle exists."""
    build()
    return os.path.exists(_OMP_LIB_PATH)


def use_all_cores(on: bool) -> None:
    """Route every following oracle call to the OpenMP build (on=True) or the
    plain single-threaded build (on=False, the default)."""
    global _lib, _use_omp
    with _lock:
        if on != _use_omp:
            _use_omp = on
            _lib = None


_use_omp = False


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_OMP_LIB_PATH if _use_omp and os.path.exists(_OMP_LIB_PATH) else _LIB_PATH)
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            I = ctypes.c_int
            lib.pti_or_f16_to_f64.restype = ctypes.c_double
            lib.pti_or_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.pti_or_q8_weight.restype = ctypes.c_double
            lib.pti_or_q8_weight.argtypes = [P, I64, I64, I64]
            lib.pti_or_twin_weight.restype = None
            lib.pti_or_twin_weight.argtypes = [P, I64, I64, I64, P, P]
            lib.pti_or_twin_pack.restype = I
            lib.pti_or_twin_pack.argtypes = [P, P, I64, P]
            lib.pti_or_twin_unpack.restype = I
            lib.pti_or_twin_unpack.argtypes = [P, I64, P, P]
            lib.pti_or_q8_gemv_rows.restype = I
            lib.pti_or_q8_gemv_rows.argtypes = [P, I64, I64, I, P, P, I64, P, P]
            lib.pti_or_twin_gemv_rows.restype = I
            lib.pti_or_twin_gemv_rows.argtypes = [P, I64, I64, P, P, P, I64, P, P, P, P]
            lib.pti_or_verify_greedy.restype = I
            lib.pti_or_verify_greedy.argtypes = [P, P, I64, I, I64, P, P, P]
            lib.pti_or_verify_sample.restype = I
            lib.pti_or_verify_sample.argtypes = [P, P, P, I64, I, I64, ctypes.c_double, P, P, P, P, P]
            lib.pti_or_mlp_layer.restype = I
            lib.pti_or_mlp_layer.argtypes = [P, P, P, I64, I64, I, ctypes.c_double, P, P, P]
            lib.pti_or_selfspec_greedy.restype = I
            lib.pti_or_selfspec_greedy.argtypes = [P, I64, I, ctypes.c_int32, I64, P, I64,
                                                   ctypes.POINTER(ctypes.c_int64), P]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    if not a.flags["C_CONTIGUOUS"]:
        raise ValueError("oracle arrays must be C-contiguous")
    return ctypes.c_void_p(a.ctypes.data)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what}: bad argument")


def f16_to_f64(h: int) -> float:
    """Decode one IEEE-754 binary16 bit pattern exactly."""
    return _load().pti_or_f16_to_f64(int(h) & 0xFFFF)


def q8_weight(w: np.ndarray, cols: int, row: int, col: int) -> float:
    return _load().pti_or_q8_weight(_ptr(w), cols, row, col)


def twin_weight(w: np.ndarray, cols: int, row: int, col: int) -> tuple[float, float]:
    a = ctypes.c_double()
    b = ctypes.c_double()
    _load().pti_or_twin_weight(_ptr(w), cols, row, col, ctypes.byref(a), ctypes.byref(b))
    return a.value, b.value


def twin_pack(qa: np.ndarray, qb: np.ndarray) -> np.ndarray:
    """Two Q8 block streams (uint8, 34 bytes per block) -> one twin stream."""
    qa = np.ascontiguousarray(qa, dtype=np.uint8).reshape(-1)
    qb = np.ascontiguousarray(qb, dtype=np.uint8).reshape(-1)
    if qa.size != qb.size or qa.size % Q8_BLOCK_BYTES:
        raise ValueError("twin_pack: mismatched or partial blocks")
    n_blocks = qa.size // Q8_BLOCK_BYTES
    out = np.empty(n_blocks * TWIN_BLOCK_BYTES, dtype=np.uint8)
    _check(_load().pti_or_twin_pack(_ptr(qa), _ptr(qb), n_blocks, _ptr(out)), "twin_pack")
    return out


def twin_unpack(twin: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    twin = np.ascontiguousarray(twin, dtype=np.uint8).reshape(-1)
    if twin.size % TWIN_BLOCK_BYTES:
        raise ValueError("twin_unpack: partial block")
    n_blocks = twin.size // TWIN_BLOCK_BYTES
    qa = np.empty(n_blocks * Q8_BLOCK_BYTES, dtype=np.uint8)
    qb = np.empty(n_blocks * Q8_BLOCK_BYTES, dtype=np.uint8)
    _check(_load().pti_or_twin_unpack(_ptr(twin), n_blocks, _ptr(qa), _ptr(qb)), "twin_unpack")
    return qa, qb


def q8_gemv(w: np.ndarray, rows: int, cols: int, x: np.ndarray, rows_idx=None):
    """fp64 N-stream Q8 GEMV.  ``x`` is [n][cols] float32.

    Returns ``(y, bound)``, both float64 [n][len(rows_idx)].
    """
    w = np.ascontiguousarray(w, dtype=np.uint8).reshape(-1)
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim == 1:
        x = x[None, :]
    n = x.shape[0]
    if x.shape[1] != cols:
        raise ValueError("q8_gemv: x has the wrong length")
    if w.size != rows * (cols // BLOCK_COLS) * Q8_BLOCK_BYTES:
        raise ValueError("q8_gemv: weight buffer has the wrong size")
    idx = (np.arange(rows, dtype=np.int64) if rows_idx is None
           else np.ascontiguousarray(rows_idx, dtype=np.int64))
    y = np.empty((n, idx.size), dtype=np.float64)
    bound = np.empty((n, idx.size), dtype=np.float64)
    _check(_load().pti_or_q8_gemv_rows(_ptr(w), rows, cols, n, _ptr(x), _ptr(idx), idx.size,
                                       _ptr(y), _ptr(bound)), "q8_gemv")
    return y, bound


def twin_gemv(w: np.ndarray, rows: int, cols: int, xa: np.ndarray, xb: np.ndarray, rows_idx=None):
    """fp64 twin GEMV.  Returns ``(ya, yb, bound_a, bound_b)``."""
    w = np.ascontiguousarray(w, dtype=np.uint8).reshape(-1)
    xa = np.ascontiguousarray(xa, dtype=np.float32).reshape(-1)
    xb = np.ascontiguousarray(xb, dtype=np.float32).reshape(-1)
    if xa.size != cols or xb.size != cols:
        raise ValueError("twin_gemv: x has the wrong length")
    if w.size != rows * (cols // BLOCK_COLS) * TWIN_BLOCK_BYTES:
        raise ValueError("twin_gemv: weight buffer has the wrong size")
    idx = (np.arange(rows, dtype=np.int64) if rows_idx is None
           else np.ascontiguousarray(rows_idx, dtype=np.int64))
    out = [np.empty(idx.size, dtype=np.float64) for _ in range(4)]
    _check(_load().pti_or_twin_gemv_rows(_ptr(w), rows, cols, _ptr(xa), _ptr(xb), _ptr(idx), idx.size,
                                         *[_ptr(o) for o in out]), "twin_gemv")
    return tuple(out)


def verify_greedy(logits: np.ndarray, guess: np.ndarray):
    """Greedy verify.  ``logits`` [steps][n][vocab] float32, ``guess`` [steps][n] int32.

    Returns ``(argmax [steps][n] int32, match [steps][n-1] uint8, accept [steps] int32)``.
    """
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    guess = np.ascontiguousarray(guess, dtype=np.int32)
    steps, n, vocab = logits.shape
    if guess.shape != (steps, n):
        raise ValueError("verify_greedy: guess has the wrong shape")
    argmax = np.empty((steps, n), dtype=np.int32)
    match = np.empty((steps, max(n - 1, 0)), dtype=np.uint8)
    accept = np.empty(steps, dtype=np.int32)
    match_ptr = _ptr(match) if n > 1 else None
    _check(_load().pti_or_verify_greedy(_ptr(logits), _ptr(guess), steps, n, vocab,
                                        _ptr(argmax), match_ptr, _ptr(accept)), "verify_greedy")
    return argmax, match, accept


def verify_sample(logits: np.ndarray, guess: np.ndarray, uniform: np.ndarray, temperature: float):
    """Sampling-mode verify.  ``logits`` [steps][n][vocab] float32, ``guess``
    [steps][n] int32, ``uniform`` [steps][n] float32 in [0, 1).

    Returns ``(token, match, accept, collision, margin)``: the inverse-CDF draws
    [steps][n] int32, match [steps][n-1] uint8, accept [steps] int32, the
    collision probabilities and the draws' margins [steps][n] float64.
    """
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    guess = np.ascontiguousarray(guess, dtype=np.int32)
    uniform = np.ascontiguousarray(uniform, dtype=np.float32)
    steps, n, vocab = logits.shape
    if guess.shape != (steps, n) or uniform.shape != (steps, n):
        raise ValueError("verify_sample: guess or uniform has the wrong shape")
    token = np.empty((steps, n), dtype=np.int32)
    match = np.empty((steps, max(n - 1, 0)), dtype=np.uint8)
    accept = np.empty(steps, dtype=np.int32)
    collision = np.empty((steps, n), dtype=np.float64)
    margin = np.empty((steps, n), dtype=np.float64)
    _check(_load().pti_or_verify_sample(_ptr(logits), _ptr(guess), _ptr(uniform), steps, n, vocab,
                                        float(temperature), _ptr(token), _ptr(match), _ptr(accept),
                                        _ptr(collision), _ptr(margin)), "verify_sample")
    return token, match, accept, collision, margin


def mlp_layer(wg, wu, wd, hidden: int, ffn: int, x: np.ndarray, eps: float = 1e-6):
    """One fp64 layer of the decode weight pass.  ``x`` [n][hidden] (any float dtype).

    Returns ``(x_out [n][hidden] float64, h [n][ffn] float64 normalised)``.
    """
    wg = np.ascontiguousarray(wg, dtype=np.uint8).reshape(-1)
    wu = np.ascontiguousarray(wu, dtype=np.uint8).reshape(-1)
    wd = np.ascontiguousarray(wd, dtype=np.uint8).reshape(-1)
    x = np.ascontiguousarray(x, dtype=np.float64)
    if x.ndim == 1:
        x = x[None, :]
    n = x.shape[0]
    if wg.size != ffn * (hidden // BLOCK_COLS) * Q8_BLOCK_BYTES or wu.size != wg.size:
        raise ValueError("mlp_layer: gate/up buffers have the wrong size")
    if wd.size != hidden * (ffn // BLOCK_COLS) * Q8_BLOCK_BYTES:
        raise ValueError("mlp_layer: down buffer has the wrong size")
    x_out = np.empty((n, hidden), dtype=np.float64)
    h = np.empty((n, ffn), dtype=np.float64)
    _check(_load().pti_or_mlp_layer(_ptr(wg), _ptr(wu), _ptr(wd), hidden, ffn, n, eps,
                                    _ptr(x), _ptr(x_out), _ptr(h)), "mlp_layer")
    return x_out, h


def selfspec_greedy(next_token: np.ndarray, n: int, first: int, steps: int):
    """Greedy self-speculative decoding over the greedy next-token table
    ``next_token`` [vocab] (pti_oracle.c, pti_or_selfspec_greedy).

    Returns ``(tokens, accept)``: the confirmed tokens after ``first``
    (int32 [count]) and the accepted length of every step (int32 [steps]).
    """
    nxt = np.ascontiguousarray(next_token, dtype=np.int32)
    cap = steps * n
    tokens = np.zeros(max(cap, 1), dtype=np.int32)
    accept = np.zeros(max(steps, 1), dtype=np.int32)
    count = ctypes.c_int64(0)
    _check(_load().pti_or_selfspec_greedy(_ptr(nxt), nxt.size, n, first, steps, _ptr(tokens), cap,
                                          ctypes.byref(count), _ptr(accept)), "selfspec_greedy")
    return tokens[:count.value].copy(), accept[:steps].copy()


def toy_logits(embedding, wg, wu, wd, wh, vocab: int, hidden: int, ffn: int, tokens, eps: float = 1e-6):
    """fp64 logits [len(tokens)][vocab] of the toy model of the self-speculative
    loop: x = embedding[token] (an fp32 table [vocab][hidden]), one decode
    layer (``mlp_layer``), logits = W_head x (``q8_gemv``, vocab rows)."""
    emb = np.asarray(embedding, dtype=np.float32).reshape(vocab, hidden)
    x = emb[np.asarray(tokens, dtype=np.int64)]
    xo, _ = mlp_layer(wg, wu, wd, hidden, ffn, x, eps)
    # the C GEMV takes fp32 activations: split the fp64 layer output into an
    # fp32 head and tail (x = hi + lo to about 2^-48 relative) and add the two
    # fp64 products
    hi = xo.astype(np.float32)
    lo = (xo - hi.astype(np.float64)).astype(np.float32)
    y, _ = q8_gemv(wh, vocab, hidden, np.concatenate([hi, lo]))
    return y[:x.shape[0]] + y[x.shape[0]:]


def greedy_next_table(logits: np.ndarray):
    """The greedy next token (argmax, lowest index on ties) of each row of
    ``logits`` [vocab][vocab] and its margin over the runner-up."""
    lg = np.asarray(logits, dtype=np.float64)
    nxt = np.argmax(lg, axis=1).astype(np.int32)
    top = lg[np.arange(lg.shape[0]), nxt]
    rest = lg.copy()
    rest[np.arange(lg.shape[0]), nxt] = -np.inf
    return nxt, top - rest.max(axis=1)

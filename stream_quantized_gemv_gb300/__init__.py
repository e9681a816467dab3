"""Packed Twin Inference hot path on GB300: Python binding of ``libpti.so``.

The compute lives in hand-written sm_103a CUDA kernels behind the C ABI of
``include/pti.h``.  This module only marshals arguments: it turns torch device
tensors into pointers, passes torch's current CUDA stream, allocates the
(reusable scratch) workspace the fast paths need, and raises ``PTIError``
on a non-OK status.  There is no fallback: if ``libpti.so`` has not been built
the import of the native library fails loudly.

Functions (same names as the C ABI, without the ``pti_`` prefix):

* ``q8_gemv_nstream(w, rows, cols, x)``      -> y [n][rows]
* ``ssq_twin_gemv(w, rows, cols, x_a, x_b)``  -> (y_a, y_b)
* ``ssq_twin_gemv_nstream(w, rows, cols, x_a, x_b)`` -> (y_a [n][rows], y_b [n][rows])
* ``verify_greedy(logits, guess)``            -> (argmax, match, accept_len)
* ``verify_sample(logits, guess, uniform, temperature)`` -> (token, match, accept_len, collision)
* ``mlp_decode_pass(w_gate, w_up, w_down, hidden, ffn, x)`` -> x after the layers
* ``device_error()``                          -> device error word (0 = none)
* ``lib()``                                   -> the ctypes handle of the C ABI
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libpti.so")

PTI_OK = 0
STATUS_NAMES = {
    0: "PTI_OK", 1: "PTI_ERR_NULL", 2: "PTI_ERR_SHAPE", 3: "PTI_ERR_NSTREAMS",
    4: "PTI_ERR_ALIGN", 5: "PTI_ERR_ALIAS", 6: "PTI_ERR_CUDA", 7: "PTI_ERR_WORKSPACE",
    8: "PTI_ERR_VALUE",
}


class PTIError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")


_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compiles libpti.so in-tree (nvcc, sm_103a)."""
    from . import _build
    return _build.build(force=force)


def lib() -> ctypes.CDLL:
    """The C ABI, with argument types declared.  Raises if the library is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"libpti.so is not built ({LIB_PATH}); run "
                                  "stream_quantized_gemv_gb300.build() first")
            L = ctypes.CDLL(LIB_PATH)
            P, I64, I, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
            L.pti_status_string.restype = ctypes.c_char_p
            L.pti_status_string.argtypes = [I]
            L.pti_q8_gemv_workspace_bytes.restype = SZ
            L.pti_q8_gemv_workspace_bytes.argtypes = [I64, I64, I]
            L.pti_q8_gemv_nstream.restype = I
            L.pti_q8_gemv_nstream.argtypes = [P, I64, I64, I, P, P, P, SZ, P]
            L.pti_q8_gemv_nstream_ex.restype = I
            L.pti_q8_gemv_nstream_ex.argtypes = [P, I64, I64, I, P, P, P, SZ, P, ctypes.c_uint32]
            L.pti_ssq_twin_gemv_ex.restype = I
            L.pti_ssq_twin_gemv_ex.argtypes = [P, I64, I64, P, P, P, P, P, SZ, P, ctypes.c_uint32]
            L.pti_ssq_twin_gemv_nstream.restype = I
            L.pti_ssq_twin_gemv_nstream.argtypes = [P, I64, I64, I, P, P, P, P, P, SZ, P, ctypes.c_uint32]
            L.pti_ssq_twin_gemv_nstream_workspace_bytes.restype = SZ
            L.pti_ssq_twin_gemv_nstream_workspace_bytes.argtypes = [I64, I64, I]
            L.pti_ssq_twin_gemv_workspace_bytes.restype = SZ
            L.pti_ssq_twin_gemv_workspace_bytes.argtypes = [I64, I64]
            L.pti_ssq_twin_gemv.restype = I
            L.pti_ssq_twin_gemv.argtypes = [P, I64, I64, P, P, P, P, P, SZ, P]
            L.pti_verify_greedy.restype = I
            L.pti_verify_greedy.argtypes = [P, P, I64, I, I64, P, P, P, P]
            L.pti_verify_sample.restype = I
            L.pti_verify_sample.argtypes = [P, P, P, I64, I, I64, ctypes.c_float, P, P, P, P, P]
            L.pti_q8_gemv_noalloc_max_scratch_bytes.restype = SZ
            L.pti_q8_gemv_noalloc_max_scratch_bytes.argtypes = []
            L.pti_q8_gemv_nstream_noalloc.restype = I
            L.pti_q8_gemv_nstream_noalloc.argtypes = [P, I64, I64, I, P, P, P]
            L.pti_mlp_decode_pass_workspace_bytes.restype = SZ
            L.pti_mlp_decode_pass_workspace_bytes.argtypes = [I64, I64, I]
            L.pti_mlp_decode_pass.restype = I
            L.pti_mlp_decode_pass.argtypes = [P, P, P, I, I64, I64, I, ctypes.c_double, P, P, P, SZ, P]
            L.pti_selfspec_greedy_workspace_bytes.restype = SZ
            L.pti_selfspec_greedy_workspace_bytes.argtypes = [I64, I64, I64, I]
            L.pti_selfspec_greedy.restype = I
            L.pti_selfspec_greedy.argtypes = [ctypes.POINTER(ToyModel), I, ctypes.c_int32, I, P, I64, P, P, P, SZ, P]
            L.pti_test_q8_gemv_stall.restype = I
            L.pti_test_q8_gemv_stall.argtypes = [P, I64, I64, I, P, P, P, SZ, P, I64, ctypes.c_uint64,
                                                 ctypes.c_uint32]
            L.pti_device_error.restype = I
            L.pti_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
            _lib = L
    return _lib


def _check(status: int, what: str) -> None:
    if status != PTI_OK:
        raise PTIError(status, what)


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def _stream(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


_ws_cache: dict = {}


def workspace(nbytes: int, device):
    """A device scratch buffer of at least ``nbytes`` bytes, reused across calls
    on the same device (the library needs no initialisation of it)."""
    import torch
    if nbytes == 0:
        return None
    dev = torch.device(device)
    key = (dev.type, dev.index if dev.index is not None else torch.cuda.current_device())
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.zeros(max(nbytes, 1 << 20), dtype=torch.uint8, device=dev)
        _ws_cache[key] = buf
    return buf


def q8_gemv_workspace_bytes(rows: int, cols: int, n_streams: int) -> int:
    return lib().pti_q8_gemv_workspace_bytes(rows, cols, n_streams)


def ssq_twin_gemv_workspace_bytes(rows: int, cols: int) -> int:
    return lib().pti_ssq_twin_gemv_workspace_bytes(rows, cols)


FLAG_PDL = 0x1
FLAG_CUDA_CORES = 0x2
FLAG_TENSOR_CORES = 0x4


def q8_gemv_nstream(w, rows: int, cols: int, x, y=None, ws=None, stream=None, flags: int = 0):
    """y[s] = W x[s] for the n = x.shape[0] streams (1..4).  ``w``: uint8 Q8 bytes.
    ``flags=FLAG_PDL`` lets the kernel start while the previous kernel in the
    stream runs (that kernel must not write ``w``); ``FLAG_CUDA_CORES`` or
    ``FLAG_TENSOR_CORES`` picks the fast path's consumer (default: CUDA
    cores)."""
    import torch
    if x.dim() == 1:
        x = x.unsqueeze(0)
    n = x.shape[0]
    if y is None:
        y = torch.empty((n, rows), dtype=torch.float32, device=x.device)
    need = q8_gemv_workspace_bytes(rows, cols, n)
    if ws is None:
        ws = workspace(need, x.device)
    _check(lib().pti_q8_gemv_nstream_ex(_ptr(w), rows, cols, n, _ptr(x), _ptr(y), _ptr(ws),
                                        0 if ws is None else ws.numel() * ws.element_size(),
                                        _stream(stream), flags), "pti_q8_gemv_nstream")
    return y


def ssq_twin_gemv(w, rows: int, cols: int, x_a, x_b, y_a=None, y_b=None, ws=None, stream=None, flags: int = 0):
    """(y_A, y_B) = (W_A x_A, W_B x_B) from one packed twin matrix ``w`` (uint8)."""
    import torch
    if y_a is None:
        y_a = torch.empty(rows, dtype=torch.float32, device=x_a.device)
    if y_b is None:
        y_b = torch.empty(rows, dtype=torch.float32, device=x_a.device)
    need = ssq_twin_gemv_workspace_bytes(rows, cols)
    if ws is None:
        ws = workspace(need, x_a.device)
    _check(lib().pti_ssq_twin_gemv_ex(_ptr(w), rows, cols, _ptr(x_a), _ptr(x_b), _ptr(y_a), _ptr(y_b),
                                      _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                                      _stream(stream), flags), "pti_ssq_twin_gemv")
    return y_a, y_b


def ssq_twin_gemv_nstream(w, rows: int, cols: int, x_a, x_b, y_a=None, y_b=None, ws=None, stream=None,
                          flags: int = 0):
    """(y_A[s], y_B[s]) = (W_A x_A[s], W_B x_B[s]) for the n = x_a.shape[0]
    (1 or 2) streams per model, from one pass over the packed twin matrix."""
    import torch
    n = x_a.shape[0]
    if y_a is None:
        y_a = torch.empty((n, rows), dtype=torch.float32, device=x_a.device)
    if y_b is None:
        y_b = torch.empty((n, rows), dtype=torch.float32, device=x_a.device)
    need = lib().pti_ssq_twin_gemv_nstream_workspace_bytes(rows, cols, n)
    if ws is None:
        ws = workspace(need, x_a.device)
    _check(lib().pti_ssq_twin_gemv_nstream(_ptr(w), rows, cols, n, _ptr(x_a), _ptr(x_b), _ptr(y_a), _ptr(y_b),
                                           _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                                           _stream(stream), flags), "pti_ssq_twin_gemv_nstream")
    return y_a, y_b


def verify_greedy(logits, guess, argmax=None, match=None, accept=None, stream=None):
    """Greedy verify of ``logits`` [steps][n][vocab] f32 against ``guess`` [steps][n] i32."""
    import torch
    steps, n, vocab = logits.shape
    dev = logits.device
    if argmax is None:
        argmax = torch.empty((steps, n), dtype=torch.int32, device=dev)
    if match is None:
        match = torch.empty((steps, max(n - 1, 0)), dtype=torch.uint8, device=dev)
    if accept is None:
        accept = torch.empty(steps, dtype=torch.int32, device=dev)
    match_ptr = _ptr(match) if n > 1 else 0
    _check(lib().pti_verify_greedy(_ptr(logits), _ptr(guess), steps, n, vocab, _ptr(argmax), match_ptr,
                                   _ptr(accept), _stream(stream)), "pti_verify_greedy")
    return argmax, match, accept


def verify_sample(logits, guess, uniform, temperature: float, token=None, match=None, accept=None,
                  collision=None, stream=None):
    """Sampling-mode verify of ``logits`` [steps][n][vocab] f32: inverse-CDF
    draws from softmax(logits / temperature) with the supplied ``uniform``
    [steps][n] f32 in [0, 1), matched against ``guess`` [steps][n] i32.

    Returns ``(token [steps][n] i32, match [steps][n-1] u8, accept [steps] i32,
    collision [steps][n] f32)``; pass ``collision=False`` to skip the collision
    output."""
    import torch
    steps, n, vocab = logits.shape
    dev = logits.device
    if token is None:
        token = torch.empty((steps, n), dtype=torch.int32, device=dev)
    if match is None:
        match = torch.empty((steps, max(n - 1, 0)), dtype=torch.uint8, device=dev)
    if accept is None:
        accept = torch.empty(steps, dtype=torch.int32, device=dev)
    if collision is None:
        collision = torch.empty((steps, n), dtype=torch.float32, device=dev)
    col_ptr = _ptr(collision) if collision is not False else 0
    match_ptr = _ptr(match) if n > 1 else 0
    _check(lib().pti_verify_sample(_ptr(logits), _ptr(guess), _ptr(uniform), steps, n, vocab,
                                   float(temperature), _ptr(token), match_ptr, _ptr(accept), col_ptr,
                                   _stream(stream)), "pti_verify_sample")
    return token, match, accept, (collision if collision is not False else None)


def q8_gemv_nstream_noalloc(w, rows: int, cols: int, x, y=None, stream=None):
    """As ``q8_gemv_nstream`` but with the library's built-in scratch instead of
    a workspace (for callers that cannot allocate device memory)."""
    import torch
    if x.dim() == 1:
        x = x.unsqueeze(0)
    n = x.shape[0]
    if y is None:
        y = torch.empty((n, rows), dtype=torch.float32, device=x.device)
    _check(lib().pti_q8_gemv_nstream_noalloc(_ptr(w), rows, cols, n, _ptr(x), _ptr(y), _stream(stream)),
           "pti_q8_gemv_nstream_noalloc")
    return y


def mlp_decode_pass_workspace_bytes(hidden: int, ffn: int, n_streams: int) -> int:
    return lib().pti_mlp_decode_pass_workspace_bytes(hidden, ffn, n_streams)


def _ptr_array(tensors):
    arr = (ctypes.c_void_p * len(tensors))(*[t.data_ptr() for t in tensors])
    return arr


class DecodeWeights:
    """The host pointer arrays of a decode pass's layers (built once, reused
    by every call; holds references to the weight tensors)."""

    def __init__(self, w_gate, w_up, w_down):
        if not (len(w_gate) == len(w_up) == len(w_down)) or len(w_gate) == 0:
            raise ValueError("DecodeWeights: need the same number (>= 1) of gate, up and down matrices")
        self.tensors = (list(w_gate), list(w_up), list(w_down))
        self.gate = _ptr_array(self.tensors[0])
        self.up = _ptr_array(self.tensors[1])
        self.down = _ptr_array(self.tensors[2])
        self.n_layers = len(w_gate)


def mlp_decode_pass(weights, hidden: int, ffn: int, x, eps: float = 1e-6, x_out=None, ws=None, stream=None):
    """Runs the gated-MLP layers of ``weights`` (a ``DecodeWeights``) over the
    streams x [n][hidden] and returns x_out [n][hidden]."""
    import torch
    if x.dim() == 1:
        x = x.unsqueeze(0)
    n = x.shape[0]
    if x_out is None:
        x_out = torch.empty((n, hidden), dtype=torch.float32, device=x.device)
    need = mlp_decode_pass_workspace_bytes(hidden, ffn, n)
    if ws is None:
        ws = workspace(need, x.device)
    _check(lib().pti_mlp_decode_pass(weights.gate, weights.up, weights.down, weights.n_layers, hidden, ffn, n,
                                     float(eps), _ptr(x), _ptr(x_out), _ptr(ws),
                                     0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)),
           "pti_mlp_decode_pass")
    return x_out


class ToyModel(ctypes.Structure):
    """The C struct pti_toy_model (device pointers and sizes)."""
    _fields_ = [("embedding", ctypes.c_void_p), ("w_gate", ctypes.c_void_p), ("w_up", ctypes.c_void_p),
                ("w_down", ctypes.c_void_p), ("w_head", ctypes.c_void_p), ("vocab", ctypes.c_int64),
                ("hidden", ctypes.c_int64), ("ffn", ctypes.c_int64), ("eps", ctypes.c_double)]


def selfspec_greedy_workspace_bytes(vocab: int, hidden: int, ffn: int, n_streams: int) -> int:
    return lib().pti_selfspec_greedy_workspace_bytes(vocab, hidden, ffn, n_streams)


def selfspec_greedy(embedding, w_gate, w_up, w_down, w_head, vocab: int, hidden: int, ffn: int, n_streams: int,
                    first_token: int, steps: int, eps: float = 1e-6, capacity=None, ws=None, stream=None,
                    out=None):
    """Greedy self-speculative decoding of the toy model on ``n_streams``
    streams for ``steps`` steps, resident on the device.  Returns
    ``(tokens, count, accept)``: the confirmed-token buffer [capacity] int32
    (default steps * n_streams), the device count [1] and the accepted
    length of every step [steps], all device tensors (``out`` may supply
    them: int32 tensors of at least those sizes)."""
    import torch
    dev = embedding.device
    cap = steps * n_streams if capacity is None else capacity
    if out is None:
        tokens = torch.zeros(max(cap, 1), dtype=torch.int32, device=dev)
        count = torch.zeros(1, dtype=torch.int32, device=dev)
        accept = torch.zeros(max(steps, 1), dtype=torch.int32, device=dev)
    else:
        tokens, count, accept = out
        if tokens.numel() < cap or count.numel() < 1 or accept.numel() < steps:
            raise ValueError("selfspec_greedy: output buffers too small")
    need = selfspec_greedy_workspace_bytes(vocab, hidden, ffn, n_streams)
    if ws is None:
        ws = workspace(need, dev)
    model = ToyModel(embedding.data_ptr(), w_gate.data_ptr(), w_up.data_ptr(), w_down.data_ptr(),
                     w_head.data_ptr(), vocab, hidden, ffn, float(eps))
    _check(lib().pti_selfspec_greedy(ctypes.byref(model), n_streams, int(first_token), steps, _ptr(tokens), cap,
                                     _ptr(count), _ptr(accept), _ptr(ws),
                                     0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)),
           "pti_selfspec_greedy")
    return tokens[:cap], count, accept[:steps]


def test_q8_gemv_stall(w, rows: int, cols: int, x, stall_unit: int, wait_ns: int, y=None, ws=None, stream=None,
                      flags: int = 0):
    """The testing hook ``pti_test_q8_gemv_stall``: a fast-path Q8 GEMV whose
    first CTA stops issuing copies at unit ``stall_unit``, with every pipeline
    wait bounded by ``wait_ns`` (``flags``: FLAG_CUDA_CORES or
    FLAG_TENSOR_CORES).  Returns y (undefined after the stall)."""
    import torch
    n = x.shape[0]
    if y is None:
        y = torch.empty((n, rows), dtype=torch.float32, device=x.device)
    need = q8_gemv_workspace_bytes(rows, cols, n)
    if ws is None:
        ws = workspace(need, x.device)
    _check(lib().pti_test_q8_gemv_stall(_ptr(w), rows, cols, n, _ptr(x), _ptr(y), _ptr(ws),
                                        0 if ws is None else ws.numel() * ws.element_size(), _stream(stream),
                                        int(stall_unit), int(wait_ns), int(flags)), "pti_test_q8_gemv_stall")
    return y


def device_error() -> int:
    """Reads and clears the device error word (synchronises the device)."""
    v = ctypes.c_uint32(0)
    _check(lib().pti_device_error(ctypes.byref(v)), "pti_device_error")
    return v.value

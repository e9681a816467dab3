"""Seeded synthetic inputs for the Packed Twin Inference hot path.

This module is the one piece shared by the oracle side and the CUDA side of
the tests and the benchmark.  It only draws random numbers and writes them into
the byte layouts the kernels read; it holds none of the method's arithmetic (no
dequantisation, no dot products, no argmax over logits it did not plant).

Two generators:

* CPU, bit-reproducible on any host: a counter-based SplitMix64 stream.  The
  i-th draw of a tensor is ``mix(base + (i + 1) * GAMMA)``, where ``mix`` is the
  SplitMix64 output function (Steele, Lea & Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014) and ``base`` is ``mix`` of the
  (seed, tensor id) pair.  Used for every parity input up to a few hundred MB.
* Device (``*_device``), for workloads too large to draw on the host in
  seconds (the 18 GB decode pass, the 10 GB verify batch): torch's seeded
  Philox generator on the GPU.  Parity tests that use it copy the sampled
  inputs back to the host for the oracle.

Distributions (the workloads of the pages' Qwen3.6-27B measurements: hidden
5120, FFN 17408, vocabulary 151936):

* int8 weights uniform on [-127, 127]: ``((r >> 32) * 255) >> 32`` - 127, a
  multiply-high mapping whose non-uniformity is below 255 / 2^32;
* block scales: ``u`` uniform on [0.5, 2), stored as binary16(u / 127) with
  round-to-nearest-even (numpy's float64 -> float16 conversion);
* activations: N(0, 1) by Box-Muller in float64, rounded to float32;
* logits: N(0, sigma) with one planted maximum per row (greedy verify), or
  plain N(0, sigma) with uniform numbers on [0, 1) for the draws (sampling).
"""
from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_TID = np.uint64(0xD1B54A32D192ED03)

Q8_BLOCK_BYTES = 34
TWIN_BLOCK_BYTES = 68
BLOCK_COLS = 32

_CHUNK = 1 << 22  # draws per numpy chunk (32 MB of uint64 temporaries)


def _mix(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _base(seed: int, tensor_id: int) -> np.uint64:
    with np.errstate(over="ignore"):
        z = (np.array([seed & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64) * GAMMA
             + np.array([tensor_id & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64) * _TID)
    return _mix(z)[0]


def draws(seed: int, tensor_id: int, start: int, count: int) -> np.ndarray:
    """Draws ``start .. start+count-1`` of the (seed, tensor_id) stream, uint64."""
    base = _base(seed, tensor_id)
    i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(base + i * GAMMA)


def _int8_from(r: np.ndarray) -> np.ndarray:
    return (((r >> np.uint64(32)) * np.uint64(255)) >> np.uint64(32)).astype(np.int16) - 127


def _unit_from(r: np.ndarray) -> np.ndarray:
    """uniform on [0, 1) with 53 random bits"""
    return (r >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def int8_uniform(seed: int, tensor_id: int, count: int, start: int = 0) -> np.ndarray:
    """int8 values uniform on [-127, 127]."""
    out = np.empty(count, dtype=np.int8)
    for c0 in range(0, count, _CHUNK):
        c1 = min(count, c0 + _CHUNK)
        out[c0:c1] = _int8_from(draws(seed, tensor_id, start + c0, c1 - c0)).astype(np.int8)
    return out


def f16_scales(seed: int, tensor_id: int, count: int, lo: float = 0.5, hi: float = 2.0) -> np.ndarray:
    """binary16 bit patterns of u / 127 with u uniform on [lo, hi)."""
    out = np.empty(count, dtype="<u2")
    for c0 in range(0, count, _CHUNK):
        c1 = min(count, c0 + _CHUNK)
        u = lo + (hi - lo) * _unit_from(draws(seed, tensor_id, c0, c1 - c0))
        out[c0:c1] = (u / 127.0).astype(np.float16).view("<u2")
    return out


def normal_f32(seed: int, tensor_id: int, count: int, sigma: float = 1.0) -> np.ndarray:
    """float32 N(0, sigma^2) by Box-Muller in float64 (two draws per value)."""
    out = np.empty(count, dtype=np.float32)
    for c0 in range(0, count, _CHUNK // 2):
        c1 = min(count, c0 + _CHUNK // 2)
        r = draws(seed, tensor_id, 2 * c0, 2 * (c1 - c0))
        u1 = 1.0 - _unit_from(r[0::2])          # (0, 1]
        u2 = _unit_from(r[1::2])
        z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
        out[c0:c1] = (sigma * z).astype(np.float32)
    return out


def index_uniform(seed: int, tensor_id: int, count: int, n: int) -> np.ndarray:
    """int64 values uniform on [0, n) (multiply-high mapping)."""
    r = draws(seed, tensor_id, 0, count)
    return ((r >> np.uint64(32)) * np.uint64(n) >> np.uint64(32)).astype(np.int64)


def uniform_f32(seed: int, tensor_id: int, count: int) -> np.ndarray:
    """float32 uniform on [0, 1): the top 24 bits of each draw times 2^-24
    (exact in float32, so 1.0 never occurs)."""
    r = draws(seed, tensor_id, 0, count)
    return ((r >> np.uint64(40)).astype(np.float64) * (1.0 / 16777216.0)).astype(np.float32)


# --------------------------------------------------------------------------
# Byte layouts
# --------------------------------------------------------------------------

def q8_matrix(rows: int, cols: int, seed: int, tensor_id: int = 0,
              scale_lo: float = 0.5, scale_hi: float = 2.0) -> np.ndarray:
    """A rows x cols Q8 matrix: per block a binary16 scale then 32 int8 values.

    Returns the raw bytes, uint8 of length rows * cols/32 * 34.
    """
    if cols % BLOCK_COLS:
        raise ValueError("cols must be a multiple of 32")
    n_blocks = rows * (cols // BLOCK_COLS)
    out = np.empty((n_blocks, Q8_BLOCK_BYTES), dtype=np.uint8)
    out[:, 0:2] = f16_scales(seed, 2 * tensor_id + 1, n_blocks, scale_lo, scale_hi).view(np.uint8).reshape(n_blocks, 2)
    out[:, 2:] = int8_uniform(seed, 2 * tensor_id, n_blocks * BLOCK_COLS).view(np.uint8).reshape(n_blocks, BLOCK_COLS)
    return out.reshape(-1)


def twin_matrix(rows: int, cols: int, seed: int, tensor_id: int = 0, identical: bool = False,
                scale_lo: float = 0.5, scale_hi: float = 2.0) -> np.ndarray:
    """A rows x cols SSQ mode-16 twin matrix, 68 bytes per block.

    Bytes 0-1 and 2-3 are two binary16 scales, bytes 4..67 are 64 int8 values
    uniform on [-127, 127].  With ``identical=True`` the two scales are equal
    and bytes 4+2i and 5+2i are equal (the two packed models are the same).
    """
    if cols % BLOCK_COLS:
        raise ValueError("cols must be a multiple of 32")
    n_blocks = rows * (cols // BLOCK_COLS)
    out = np.empty((n_blocks, TWIN_BLOCK_BYTES), dtype=np.uint8)
    s0 = f16_scales(seed, 3 * tensor_id + 1, n_blocks, scale_lo, scale_hi)
    out[:, 0:2] = s0.view(np.uint8).reshape(n_blocks, 2)
    if identical:
        out[:, 2:4] = out[:, 0:2]
        q = int8_uniform(seed, 3 * tensor_id, n_blocks * BLOCK_COLS).view(np.uint8).reshape(n_blocks, BLOCK_COLS)
        out[:, 4::2] = q
        out[:, 5::2] = q
    else:
        s1 = f16_scales(seed, 3 * tensor_id + 2, n_blocks, scale_lo, scale_hi)
        out[:, 2:4] = s1.view(np.uint8).reshape(n_blocks, 2)
        out[:, 4:] = int8_uniform(seed, 3 * tensor_id, n_blocks * 2 * BLOCK_COLS).view(np.uint8).reshape(n_blocks, 2 * BLOCK_COLS)
    return out.reshape(-1)


def toy_model(vocab: int, hidden: int, ffn: int, seed: int) -> dict:
    """Synthetic weights of the toy model of the self-speculative loop: an fp32
    embedding table [vocab][hidden] N(0, 1), one gated-MLP layer (gate and up
    [ffn][hidden], down [hidden][ffn], Q8) and an LM head [vocab][hidden] Q8,
    each from its own tensor id."""
    return {
        "embedding": normal_f32(seed, 40, vocab * hidden).reshape(vocab, hidden),
        "w_gate": q8_matrix(ffn, hidden, seed, tensor_id=41),
        "w_up": q8_matrix(ffn, hidden, seed, tensor_id=42),
        "w_down": q8_matrix(hidden, ffn, seed, tensor_id=43),
        "w_head": q8_matrix(vocab, hidden, seed, tensor_id=44),
        "vocab": vocab, "hidden": hidden, "ffn": ffn,
    }


def activations(n: int, cols: int, seed: int, tensor_id: int = 0) -> np.ndarray:
    """[n][cols] float32 N(0, 1), stream-major."""
    return normal_f32(seed, tensor_id, n * cols).reshape(n, cols)


def verify_batch(steps: int, n: int, vocab: int, p: float, seed: int, tensor_id: int = 0,
                 sigma: float = 3.0):
    """Greedy-verify inputs with a planted maximum per row and planted guesses.

    Each row (t, s) of logits is N(0, sigma^2); a random index ``a[t][s]`` is
    then set to the row's maximum + 1.0 so that it is the unique maximum.  For
    s >= 1 the guess fed to stream s equals ``a[t][s-1]`` with probability p,
    otherwise a different token ``(a + 1 + U[0, vocab-2]) mod vocab``.  The
    guess of stream 0 is a random token (the verifier does not read it).

    Returns ``(logits [steps][n][vocab] f32, guess [steps][n] i32, planted [steps][n] i32)``.
    """
    logits = normal_f32(seed, 4 * tensor_id, steps * n * vocab, sigma).reshape(steps, n, vocab)
    planted = index_uniform(seed, 4 * tensor_id + 1, steps * n, vocab).reshape(steps, n)
    rows = logits.reshape(steps * n, vocab)
    flat = planted.reshape(-1)
    rows[np.arange(steps * n), flat] = rows.max(axis=1) + np.float32(1.0)
    guess = np.empty((steps, n), dtype=np.int32)
    guess[:, 0] = index_uniform(seed, 4 * tensor_id + 2, steps, vocab).astype(np.int32)
    if n > 1:
        r = draws(seed, 4 * tensor_id + 3, 0, 2 * steps * (n - 1))
        keep = _unit_from(r[0::2]).reshape(steps, n - 1) < p
        off = 1 + ((r[1::2] >> np.uint64(32)) * np.uint64(max(vocab - 1, 1)) >> np.uint64(32)).astype(np.int64)
        off = off.reshape(steps, n - 1)
        prev = planted[:, :-1]
        wrong = (prev + off) % vocab if vocab > 1 else prev
        guess[:, 1:] = np.where(keep, prev, wrong).astype(np.int32)
    return logits, guess, planted.astype(np.int32)


def sample_batch(steps: int, n: int, vocab: int, seed: int, tensor_id: int = 0, sigma: float = 3.0,
                 masked: float = 0.0):
    """Sampling-verify inputs: logits [steps][n][vocab] float32 N(0, sigma^2)
    and the draws' uniform numbers [steps][n] float32 on [0, 1).  With
    ``masked`` > 0 about that fraction of the tokens is set to -inf (token 0
    never is, so every row keeps a finite logit).  Guesses are left to the
    caller: they are draws, which need the method's arithmetic.

    Returns ``(logits, uniform)``.
    """
    logits = normal_f32(seed, 4 * tensor_id, steps * n * vocab, sigma).reshape(steps, n, vocab)
    uniform = uniform_f32(seed, 4 * tensor_id + 1, steps * n).reshape(steps, n)
    if masked > 0.0:
        drop = _unit_from(draws(seed, 4 * tensor_id + 2, 0, steps * n * vocab)).reshape(steps, n, vocab) < masked
        drop[:, :, 0] = False
        logits[drop] = -np.inf
    return logits, uniform


# --------------------------------------------------------------------------
# Device generators (torch Philox on the GPU) for multi-GB workloads
# --------------------------------------------------------------------------

def _gen(device, seed: int, tensor_id: int):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1000003 + tensor_id) & 0x7FFFFFFFFFFFFFFF)
    return g


def q8_matrix_device(rows: int, cols: int, seed: int, tensor_id: int, device="cuda",
                     scale_lo: float = 0.5, scale_hi: float = 2.0, out=None):
    """Same layout and distributions as ``q8_matrix``, drawn on the device.

    ``out`` (optional) is a preallocated uint8 device tensor of the right size.
    """
    import torch
    if cols % BLOCK_COLS:
        raise ValueError("cols must be a multiple of 32")
    n_blocks = rows * (cols // BLOCK_COLS)
    g = _gen(device, seed, tensor_id)
    if out is None:
        out = torch.empty(n_blocks * Q8_BLOCK_BYTES, dtype=torch.uint8, device=device)
    view = out.view(n_blocks, Q8_BLOCK_BYTES)
    q = torch.randint(-127, 128, (n_blocks, BLOCK_COLS), generator=g, device=device, dtype=torch.int16)
    view[:, 2:] = q.to(torch.int8).view(torch.uint8)
    del q
    u = torch.rand((n_blocks,), generator=g, device=device, dtype=torch.float64) * (scale_hi - scale_lo) + scale_lo
    view[:, 0:2] = (u / 127.0).to(torch.float16).view(torch.uint8).view(n_blocks, 2)
    return out


def twin_matrix_device(rows: int, cols: int, seed: int, tensor_id: int, device="cuda",
                       identical: bool = False, scale_lo: float = 0.5, scale_hi: float = 2.0):
    """Same layout and distributions as ``twin_matrix``, drawn on the device."""
    import torch
    if cols % BLOCK_COLS:
        raise ValueError("cols must be a multiple of 32")
    n_blocks = rows * (cols // BLOCK_COLS)
    g = _gen(device, seed, tensor_id)
    out = torch.empty((n_blocks, TWIN_BLOCK_BYTES), dtype=torch.uint8, device=device)
    if identical:
        q = torch.randint(-127, 128, (n_blocks, BLOCK_COLS), generator=g, device=device,
                          dtype=torch.int16).to(torch.int8).view(torch.uint8)
        out[:, 4::2] = q
        out[:, 5::2] = q
    else:
        q = torch.randint(-127, 128, (n_blocks, 2 * BLOCK_COLS), generator=g, device=device,
                          dtype=torch.int16).to(torch.int8).view(torch.uint8)
        out[:, 4:] = q
    del q
    u = torch.rand((n_blocks, 2), generator=g, device=device, dtype=torch.float64) * (scale_hi - scale_lo) + scale_lo
    if identical:
        u[:, 1] = u[:, 0]
    out[:, 0:4] = (u / 127.0).to(torch.float16).view(torch.uint8).view(n_blocks, 4)
    return out.view(-1)


def activations_device(n: int, cols: int, seed: int, tensor_id: int, device="cuda"):
    import torch
    g = _gen(device, seed, tensor_id)
    return torch.randn((n, cols), generator=g, device=device, dtype=torch.float32)


def sample_batch_device(steps: int, n: int, vocab: int, seed: int, tensor_id: int = 0, sigma: float = 3.0,
                        device="cuda"):
    """``sample_batch`` drawn on the device (no masking): N(0, sigma^2) logits
    and uniform numbers on [0, 1)."""
    import torch
    g = _gen(device, seed, tensor_id)
    logits = torch.randn((steps, n, vocab), generator=g, device=device, dtype=torch.float32)
    logits.mul_(sigma)
    uniform = torch.rand((steps, n), generator=g, device=device, dtype=torch.float32)
    return logits, uniform


def verify_batch_device(steps: int, n: int, vocab: int, p: float, seed: int, tensor_id: int = 0,
                        sigma: float = 3.0, device="cuda"):
    """Same construction as ``verify_batch``, drawn on the device."""
    import torch
    g = _gen(device, seed, tensor_id)
    logits = torch.randn((steps, n, vocab), generator=g, device=device, dtype=torch.float32)
    logits.mul_(sigma)
    planted = torch.randint(0, vocab, (steps, n), generator=g, device=device, dtype=torch.int64)
    rowmax = logits.amax(dim=2, keepdim=True)
    logits.scatter_(2, planted.unsqueeze(2), rowmax + 1.0)
    guess = torch.empty((steps, n), dtype=torch.int32, device=device)
    guess[:, 0] = torch.randint(0, vocab, (steps,), generator=g, device=device, dtype=torch.int32)
    if n > 1:
        keep = torch.rand((steps, n - 1), generator=g, device=device) < p
        off = torch.randint(1, max(vocab, 2), (steps, n - 1), generator=g, device=device, dtype=torch.int64)
        prev = planted[:, :-1]
        wrong = (prev + off) % vocab if vocab > 1 else prev
        guess[:, 1:] = torch.where(keep, prev, wrong).to(torch.int32)
    return logits, guess, planted.to(torch.int32)

"""The allocation-free Q8 GEMV entry point, for callers that cannot allocate
device memory (a plug-in inside a runtime that owns every device allocation,
or a decode loop that must not call the CUDA allocator once it runs).

Called through the C ABI, it must give the same results as the entry point that
takes a caller-supplied workspace, on two calls in a row that share its
built-in scratch.  This file sorts last so a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import pti_synth
import stream_quantized_gemv_gb300 as pti

pytestmark = pytest.mark.gpu

TOL = 1e-5


def test_noalloc_entry_point_matches_the_workspace_entry_point_on_two_calls():
    pti.build()
    L = pti.lib()
    stream = torch.cuda.current_stream().cuda_stream
    # two calls in a row with different shapes and stream counts share the
    # built-in scratch
    for call, (rows, cols, n) in enumerate(((1000, 2048, 4), (520, 1024, 1))):
        w_np = pti_synth.q8_matrix(rows, cols, seed=300 + call)
        x_np = pti_synth.activations(n, cols, seed=310 + call)
        w = torch.from_numpy(w_np).cuda()
        x = torch.from_numpy(x_np).cuda()
        y_ws = pti.q8_gemv_nstream(w, rows, cols, x)            # caller-supplied workspace
        y_na = torch.empty((n, rows), dtype=torch.float32, device="cuda")
        rc = L.pti_q8_gemv_nstream_noalloc(w.data_ptr(), rows, cols, n, x.data_ptr(), y_na.data_ptr(), stream)
        assert rc == 0, L.pti_status_string(rc)
        torch.cuda.synchronize()
        y_ref, bound = oracle.q8_gemv(w_np, rows, cols, x_np)
        y_na_np = y_na.cpu().numpy().astype(np.float64)
        diff = np.abs(y_na_np - y_ws.cpu().numpy())
        assert np.all(diff <= TOL * bound), f"call {call}: max diff/bound {np.max(diff / bound):.3g}"
        # and on its own against the oracle's exact values, within the same bar
        err = np.abs(y_na_np - y_ref)
        assert np.all(err <= TOL * bound), f"call {call}: max err/bound vs oracle {np.max(err / bound):.3g}"
    assert pti.device_error() == 0


def test_noalloc_scratch_covers_every_shape():
    """The fast path's scratch depends only on the stream count, so the 2 MiB
    array serves every valid shape; the entry point still validates its
    arguments like the workspace entry point."""
    pti.build()
    L = pti.lib()
    limit = L.pti_q8_gemv_noalloc_max_scratch_bytes()
    assert limit == 2 << 20
    for rows, cols in ((1 << 31, 256), (1, 1 << 31), (17408, 5120)):
        for n in (1, 2, 3, 4):
            assert L.pti_q8_gemv_workspace_bytes(rows, cols, n) <= limit
    fake = 0x7F0000000000  # never dereferenced: validation fails first
    assert L.pti_q8_gemv_nstream_noalloc(None, 128, 512, 4, fake, fake + (1 << 36), None) == 1
    assert L.pti_q8_gemv_nstream_noalloc(fake, 128, 48, 4, fake + (1 << 36), fake + (2 << 36), None) == 2
    assert L.pti_q8_gemv_nstream_noalloc(fake, 128, 512, 5, fake + (1 << 36), fake + (2 << 36), None) == 3

"""A bounded pipeline wait that runs out, without faulting the GPU.

The testing hook pti_test_q8_gemv_stall runs the fast-path Q8 GEMV (with
either consumer: CUDA cores or tensor core) with the first CTA's copy
producer stopping before one unit (as if that copy never arrived) and every
pipeline wait limited to 1 ms.  The consumer warps waiting
for the missing tile must give up, record PTI_DEVERR_FULL_TIMEOUT and wind
down; every copy that was issued must have landed before the kernel exits (no
PTI_DEVERR_DRAIN_TIMEOUT); the CUDA context, the stream and the library must
stay usable: a following normal call on the same stream matches the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import pti_synth
import stream_quantized_gemv_gb300 as pti

pytestmark = pytest.mark.gpu

FULL_TIMEOUT, EMPTY_TIMEOUT, DRAIN_TIMEOUT = 0x1, 0x2, 0x4


@pytest.fixture(scope="module", autouse=True)
def _built():
    pti.build()
    pti.lib()
    pti.device_error()  # start from a clear error word
    yield
    assert pti.device_error() == 0


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def first_cta_units(rows, cols):
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    units = ((rows + 127) // 128) * (cols // 256)
    return units // min(sms, units, 320)


@pytest.mark.parametrize("flags", [pti.FLAG_CUDA_CORES, pti.FLAG_TENSOR_CORES])
@pytest.mark.parametrize("n", [1, 4])
def test_stalled_copy_times_out_and_the_library_stays_usable(n, flags):
    rows, cols = 17408, 2048
    per_cta = first_cta_units(rows, cols)
    assert per_cta >= 7, "the shape must give the first CTA more units than the ring holds"
    w = pti_synth.q8_matrix(rows, cols, seed=5, tensor_id=60)
    x = pti_synth.activations(n, cols, seed=5, tensor_id=61)
    wd, xd = dev(w), dev(x)
    stream = torch.cuda.current_stream()

    y_bad = pti.test_q8_gemv_stall(wd, rows, cols, xd, stall_unit=per_cta - 1, wait_ns=1_000_000, flags=flags)
    torch.cuda.synchronize()                       # no CUDA error: the kernel returned
    err = pti.device_error()
    assert err & FULL_TIMEOUT, f"device error word {err:#x}: the consumers' wait did not run out"
    assert not err & DRAIN_TIMEOUT, f"device error word {err:#x}: copies were still in flight at exit"
    assert pti.device_error() == 0                 # reading cleared it
    del y_bad

    # the same stream, the same workspace: a normal call is exact again
    y = pti.q8_gemv_nstream(wd, rows, cols, xd, stream=stream, flags=flags).cpu().numpy()
    idx = np.unique(np.concatenate([np.arange(0, rows, 97), [rows - 1]])).astype(np.int64)
    y_ref, bound = oracle.q8_gemv(w, rows, cols, x, rows_idx=idx)
    assert np.all(np.abs(y[:, idx] - y_ref) <= 1e-5 * bound)
    assert pti.device_error() == 0


def test_stall_hook_rejects_a_unit_inside_the_first_fill():
    rows, cols = 17408, 2048
    w = dev(pti_synth.q8_matrix(256, cols, seed=1, tensor_id=62))
    x = dev(pti_synth.activations(1, cols, seed=1, tensor_id=63))
    with pytest.raises(pti.PTIError):
        pti.test_q8_gemv_stall(w, 256, cols, x, stall_unit=5, wait_ns=1_000_000)
    with pytest.raises(pti.PTIError):
        pti.test_q8_gemv_stall(w, 256, cols, x, stall_unit=first_cta_units(rows, cols) + 100, wait_ns=1_000_000)

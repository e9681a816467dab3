"""Why the 64-layer decode chain is compared layer by layer, not end to end.

The GPU test of 64 chained layers (hidden 256, ffn 512, N = 4, seed 21) prints
the drift of the whole chain against the oracle's own chain (max |err| about
4-5 with outputs of rms 1) instead of gating it, on the reading that random
gated-MLP layers amplify any rounding-sized difference of their input.  This
test pins that reading on the oracle alone: the same 64 layers, run from x and
from x moved by one fp32 ulp in every element, diverge by the same order.
Nothing here runs on a GPU.
"""
import numpy as np

import oracle
import pti_synth

HIDDEN, FFN, N, SEED, EPS = 256, 512, 4, 21, 1e-6


def layers(n_layers):
    """The layers of the GPU test: gate, up [ffn][hidden/32], down [hidden][ffn/32] Q8 blocks."""
    return [(pti_synth.q8_matrix(FFN, HIDDEN, SEED, 3 * l), pti_synth.q8_matrix(FFN, HIDDEN, SEED, 3 * l + 1),
             pti_synth.q8_matrix(HIDDEN, FFN, SEED, 3 * l + 2)) for l in range(n_layers)]


def test_one_ulp_at_the_input_grows_to_order_one_over_64_layers():
    x = pti_synth.activations(N, HIDDEN, SEED, 1000)
    x_ulp = np.nextafter(x, np.float32(np.inf))          # every element one fp32 ulp up
    a, b = x.astype(np.float64), x_ulp.astype(np.float64)
    diff = []
    for g, u, d in layers(64):
        a, _ = oracle.mlp_layer(g, u, d, HIDDEN, FFN, a, EPS)
        b, _ = oracle.mlp_layer(g, u, d, HIDDEN, FFN, b, EPS)
        diff.append(float(np.max(np.abs(a - b))))
    rms = float(np.sqrt(np.mean(a * a)))
    assert abs(rms - 1.0) < 1e-6                         # each layer ends with an RMS rescale
    # after one layer the difference is still of the size of the perturbation ...
    assert diff[0] < 1e-5
    # ... it grows layer by layer (by a factor above 1e5 over the first 40 layers) ...
    assert diff[40] > 1e5 * diff[0]
    assert all(diff[k + 8] > diff[k] for k in range(0, 32, 8))
    # ... and after 64 layers it is of order one: the size of the drift the GPU
    # chain shows against the oracle's chain, whose roundings differ from the
    # kernels' from the first layer on.
    assert 0.3 < diff[-1] < 20.0


def test_identical_inputs_give_identical_chains():
    # the amplification needs a difference to amplify: the oracle chain is
    # deterministic (a plain check that the growth above is not noise)
    x = pti_synth.activations(N, HIDDEN, SEED, 1000).astype(np.float64)
    a, b = x.copy(), x.copy()
    for g, u, d in layers(8):
        a, _ = oracle.mlp_layer(g, u, d, HIDDEN, FFN, a, EPS)
        b, _ = oracle.mlp_layer(g, u, d, HIDDEN, FFN, b, EPS)
    assert np.array_equal(a, b)

"""GPU parity of the chained decode pass (gated-MLP layers: gate, up, SiLU,
RMS, down, RMS) against the fp64 oracle.

Each layer is checked in isolation: the pass run over the first k layers must
equal the oracle's layer k applied to the pass's own output after k - 1
layers.  The bar per output element is the GEMV contract (|err| <= 1e-5 *
sum |w x| for each of the three GEMVs) carried through the layer to first
order:

  * g and u carry at most 1e-5 * bound_g and 1e-5 * bound_u, so h = SiLU(g) u
    carries at most dh = 1e-5 (|SiLU'(g) u| bound_g + |SiLU(g)| bound_u);
  * the down GEMV of the normalised h (hn = h / rms(h)) adds at most
    1e-5 * sum_j |W_down hn_j|, and carries sum_j |W_down| dh_j / rms(h);
  * the final RMS scale b multiplies both; the scales themselves are exact to
    a few fp32 roundings (1e-5 |x_out| covers them).

A factor of 2 is kept on top for the second-order terms.  Inputs come from the
seeded generator (pti_synth) only.
"""
import numpy as np
import pytest
import torch

import oracle
import pti_synth
import stream_quantized_gemv_gb300 as pti

pytestmark = pytest.mark.gpu

EPS = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _built():
    pti.build()
    pti.lib()
    yield
    assert pti.device_error() == 0


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_layers(n_layers, hidden, ffn, seed):
    """Layer l: gate, up [ffn][hidden/32] and down [hidden][ffn/32] Q8 blocks."""
    out = []
    for l in range(n_layers):
        out.append((pti_synth.q8_matrix(ffn, hidden, seed, 3 * l),
                    pti_synth.q8_matrix(ffn, hidden, seed, 3 * l + 1),
                    pti_synth.q8_matrix(hidden, ffn, seed, 3 * l + 2)))
    return out


def device_weights(layers):
    return pti.DecodeWeights([dev(g) for g, _, _ in layers], [dev(u) for _, u, _ in layers],
                             [dev(d) for _, _, d in layers])


def silu(v):
    return v / (1.0 + np.exp(-v))


def layer_tolerance(wg, wu, wd, hidden, ffn, x, eps=EPS):
    """Oracle output of one layer on x [n][hidden] and the per-element bar."""
    x32 = np.ascontiguousarray(x, dtype=np.float32)
    xo, hn = oracle.mlp_layer(wg, wu, wd, hidden, ffn, x32, eps)
    g, bg = oracle.q8_gemv(wg, ffn, hidden, x32)
    u, bu = oracle.q8_gemv(wu, ffn, hidden, x32)
    sig = 1.0 / (1.0 + np.exp(-g))
    dsilu = sig * (1.0 + g * (1.0 - sig))
    dh = 1e-5 * (np.abs(dsilu * u) * bg + np.abs(silu(g)) * bu)
    h = silu(g) * u
    rms_h = np.sqrt(np.mean(h * h, axis=1) + eps)
    z = np.empty((x.shape[0], hidden))
    carried = np.empty_like(z)
    own = np.empty_like(z)
    for s in range(x.shape[0]):
        z_s, own_s = oracle.q8_gemv(wd, hidden, ffn, hn[s].astype(np.float32))
        _, carried_s = oracle.q8_gemv(wd, hidden, ffn, (dh[s] / rms_h[s]).astype(np.float32))
        z[s], own[s], carried[s] = z_s[0], own_s[0], carried_s[0]
    b = 1.0 / np.sqrt(np.mean(z * z, axis=1) + eps)
    tol = 2.0 * (b[:, None] * (carried + 1e-5 * own) + 1e-5 * np.abs(xo))
    return xo, tol


def check_layer(got, xo, tol, what):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - xo)
    if np.any(err > tol):
        i = np.unravel_index(np.argmax(err / tol), err.shape)
        raise AssertionError(f"{what}: {(err > tol).sum()} outputs off; worst {i}: err {err[i]:.3g}, bar {tol[i]:.3g}")


def run_pass(weights, n_layers, hidden, ffn, x, eps=EPS):
    w = pti.DecodeWeights(weights.tensors[0][:n_layers], weights.tensors[1][:n_layers],
                          weights.tensors[2][:n_layers])
    y = pti.mlp_decode_pass(w, hidden, ffn, x, eps=eps)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def check_chain(layers, hidden, ffn, n, seed, eps=EPS, x=None):
    w = device_weights(layers)
    if x is None:
        x = pti_synth.activations(n, hidden, seed, 1000)
    xd = dev(x)
    prev = x.astype(np.float64)
    for k in range(1, len(layers) + 1):
        got = run_pass(w, k, hidden, ffn, xd, eps)
        xo, tol = layer_tolerance(*layers[k - 1], hidden, ffn, prev.astype(np.float32), eps)
        check_layer(got, xo, tol, f"hidden {hidden} ffn {ffn} n {n} layer {k}")
        prev = got.astype(np.float64)
    return prev


# shapes: stream-K tiles shared by several CTAs (256x512, 768x1280), whole
# tiles per CTA in the down kernel (4096x256), CTAs spanning more than two
# gate/up tiles (256x40960)
@pytest.mark.parametrize("hidden,ffn", [(256, 512), (768, 1280), (4096, 256), (256, 40960)])
@pytest.mark.parametrize("n", [1, 2, 3, 4])
def test_decode_pass_one_layer(hidden, ffn, n):
    layers = host_layers(1, hidden, ffn, seed=hidden + ffn)
    check_chain(layers, hidden, ffn, n, seed=n)


@pytest.mark.parametrize("n", [1, 4])
def test_decode_pass_three_layers(n):
    hidden, ffn = 512, 1536
    layers = host_layers(3, hidden, ffn, seed=5)
    check_chain(layers, hidden, ffn, n, seed=7)


def test_decode_pass_seventy_layers():
    """70 chained layers: layers 64, 65 and 70 each stay within their bars
    (the pass over k layers against the oracle's layer k applied to the pass's
    own output after k - 1)."""
    hidden, ffn, n = 256, 512, 2
    layers = host_layers(70, hidden, ffn, seed=31)
    x = pti_synth.activations(n, hidden, 31, 1000)
    w = device_weights(layers)
    for k in (64, 65, 70):
        g_k = run_pass(w, k, hidden, ffn, dev(x))
        g_prev = run_pass(w, k - 1, hidden, ffn, dev(x))
        xo, tol = layer_tolerance(*layers[k - 1], hidden, ffn, g_prev.astype(np.float32))
        check_layer(g_k, xo, tol, f"layer {k}")


def test_decode_pass_eps_matters():
    """A large eps next to small activations: the RMS scales differ visibly
    from eps = 0, and both still match the oracle."""
    hidden, ffn = 256, 512
    layers = host_layers(2, hidden, ffn, seed=9)
    x = (pti_synth.activations(4, hidden, 3, 0) * np.float32(1e-3)).astype(np.float32)
    out_big = check_chain(layers, hidden, ffn, 4, seed=3, eps=1e-2, x=x)
    out_zero = check_chain(layers, hidden, ffn, 4, seed=3, eps=0.0, x=x)
    assert np.max(np.abs(out_big - out_zero)) > 1e-3


def test_decode_pass_64_layers(capsys):
    """64 chained layers at a small size, every layer within its bar.  The
    drift of the whole chain against the oracle's own 64-layer chain is
    printed, not gated: rounding differences are amplified from layer to layer
    by the random layers themselves, whatever the kernels do
    (tests/test_drift_pins.py: the oracle's chain moved by one fp32 ulp at its
    input diverges to max |diff| of order one over the same 64 layers)."""
    hidden, ffn, n = 256, 512, 4
    layers = host_layers(64, hidden, ffn, seed=21)
    x = pti_synth.activations(n, hidden, 21, 1000)
    got = check_chain(layers, hidden, ffn, n, seed=21, x=x)
    ref = x.astype(np.float64)
    for wg, wu, wd in layers:
        ref, _ = oracle.mlp_layer(wg, wu, wd, hidden, ffn, ref, EPS)
    assert np.all(np.isfinite(got))
    with capsys.disabled():
        print(f"\n64-layer drift vs the oracle chain: max |err| {np.max(np.abs(got - ref)):.3g}, "
              f"rms of the output {np.sqrt(np.mean(ref * ref)):.3g}")


def test_decode_pass_is_deterministic_in_place_and_needs_no_workspace_init():
    hidden, ffn, n = 768, 1280, 4
    layers = host_layers(2, hidden, ffn, seed=4)
    w = device_weights(layers)
    x = dev(pti_synth.activations(n, hidden, 4, 1000))
    need = pti.mlp_decode_pass_workspace_bytes(hidden, ffn, n)
    ws = torch.full((need + 4096,), 255, dtype=torch.uint8, device="cuda")  # NaN patterns everywhere
    a = pti.mlp_decode_pass(w, hidden, ffn, x, ws=ws)
    b = pti.mlp_decode_pass(w, hidden, ffn, x, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    xi = x.clone()
    pti.mlp_decode_pass(w, hidden, ffn, xi, x_out=xi, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(xi, a)
    xo, tol = layer_tolerance(*layers[1], hidden, ffn,
                              run_pass(w, 1, hidden, ffn, x).astype(np.float32))
    check_layer(a.cpu().numpy(), xo, tol, "layer 2 on a garbage-filled workspace")
    # the same workspace then serves a plain GEMV of another shape
    wq = dev(pti_synth.q8_matrix(1000, 2048, 4, 77))
    xq = dev(pti_synth.activations(3, 2048, 4, 78))
    y = pti.q8_gemv_nstream(wq, 1000, 2048, xq, ws=ws).cpu().numpy()
    y_ref, bound = oracle.q8_gemv(wq.cpu().numpy(), 1000, 2048, xq.cpu().numpy())
    assert np.all(np.abs(y - y_ref) <= 1e-5 * bound)


def test_decode_pass_layers_may_share_matrices():
    hidden, ffn, n = 256, 512, 2
    (g, u, d), = host_layers(1, hidden, ffn, seed=12)
    gd, ud, dd = dev(g), dev(u), dev(d)
    w = pti.DecodeWeights([gd, gd], [ud, ud], [dd, dd])
    x = pti_synth.activations(n, hidden, 12, 1000)
    got1 = pti.mlp_decode_pass(pti.DecodeWeights([gd], [ud], [dd]), hidden, ffn, dev(x)).cpu().numpy()
    got2 = pti.mlp_decode_pass(w, hidden, ffn, dev(x)).cpu().numpy()
    xo, tol = layer_tolerance(g, u, d, hidden, ffn, got1)
    check_layer(got2, xo, tol, "shared matrices, layer 2")


def test_decode_pass_full_size_two_layers():
    """hidden 5120, ffn 17408, N = 4: the shapes of the 64-layer pass, two
    layers, every output checked."""
    hidden, ffn, n = 5120, 17408, 4
    layers_dev = []
    for l in range(2):
        layers_dev.append((pti_synth.q8_matrix_device(ffn, hidden, 0, 3 * l),
                           pti_synth.q8_matrix_device(ffn, hidden, 0, 3 * l + 1),
                           pti_synth.q8_matrix_device(hidden, ffn, 0, 3 * l + 2)))
    w = pti.DecodeWeights([g for g, _, _ in layers_dev], [u for _, u, _ in layers_dev],
                          [d for _, _, d in layers_dev])
    x = pti_synth.activations(n, hidden, 0, 1000)
    xd = dev(x)
    g, u, d = (t.cpu().numpy() for t in layers_dev[0])
    got1 = run_pass(w, 1, hidden, ffn, xd)
    xo, tol = layer_tolerance(g, u, d, hidden, ffn, x)
    check_layer(got1, xo, tol, "full size layer 1")
    g, u, d = (t.cpu().numpy() for t in layers_dev[1])
    xo, tol = layer_tolerance(g, u, d, hidden, ffn, got1.astype(np.float32))
    got2 = run_pass(w, 2, hidden, ffn, xd)
    check_layer(got2, xo, tol, "full size layer 2")
    del layers_dev, w
    torch.cuda.empty_cache()


@pytest.mark.parametrize("n", [1, 2, 3])
def test_decode_pass_full_size_fewer_streams(n):
    """hidden 5120, ffn 17408 with one to three streams: one layer, every
    output checked (the four-stream case is the two-layer test above)."""
    hidden, ffn = 5120, 17408
    gd = pti_synth.q8_matrix_device(ffn, hidden, 7, 0)
    ud = pti_synth.q8_matrix_device(ffn, hidden, 7, 1)
    dd = pti_synth.q8_matrix_device(hidden, ffn, 7, 2)
    x = pti_synth.activations(n, hidden, 7, 1000 + n)
    got = run_pass(pti.DecodeWeights([gd], [ud], [dd]), 1, hidden, ffn, dev(x))
    g, u, d = gd.cpu().numpy(), ud.cpu().numpy(), dd.cpu().numpy()
    xo, tol = layer_tolerance(g, u, d, hidden, ffn, x)
    check_layer(got, xo, tol, f"full size, {n} streams")
    del gd, ud, dd
    torch.cuda.empty_cache()

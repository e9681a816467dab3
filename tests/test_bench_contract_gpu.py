"""bench.py's JSON line on a short decode pass (2 layers of the 5120 / 17408
shapes, N = 4): every key of the measurement contract is present and the
numbers agree with one another (GPU)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LAYERS, STEPS, WARMUP, N = 2, 3, 3, 4


@pytest.mark.gpu
def test_decode_line_carries_the_contract():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "decode", "--layers", str(LAYERS),
           "--steps", str(STEPS), "--warmup", str(WARMUP), "--n", str(N)]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-4000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout[-4000:]
    d = json.loads(lines[0])

    assert d["n_gpus"] == 1 and d["steps"] == STEPS and d["warmup"] == WARMUP
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["vs_baseline"] is None and isinstance(d["metric"], str) and isinstance(d["dtype"], str)
    assert "synthetic" in d["data"] and isinstance(d["config"]["workload"], str)
    assert d["config"]["layers"] == LAYERS and d["config"]["n_streams"] == N

    # value = the step's algorithmic bytes over the step time; the weights are
    # almost all of them (activations add well under 1%)
    wbytes = d["config"]["weight_bytes_per_step"]
    assert wbytes == LAYERS * 3 * 17408 * (5120 // 32) * 34
    step_bytes = d["value"] * 1e9 * d["ms_per_step"] * 1e-3
    assert wbytes <= step_bytes * (1 + 1e-3) and step_bytes <= wbytes * 1.01
    assert d["stream_tokens_per_s"] == pytest.approx(N / (d["ms_per_step"] * 1e-3), rel=1e-3)

    r = d["roofline"]
    assert r["bound"] in ("hbm", "tensor", "alu") and r["unit"] == "GB/s"
    assert r["achieved"] > 0 and r["peak"] > 0 and "traffic" in r
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=2e-3)
    a = d["alu_roofline"]
    assert a["bound"] == "alu" and 0 < a["frac"] < 1.5

    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["value"] > 0 and c["cores"] >= 1 and c["sample"]
    assert c["single_core_value"] > 0 and (c["cores"] == 1 or c["value"] > c["single_core_value"])

    # the 17408 x 5120 Q8 GEMV at one and four streams, same harness
    q = d["q8_target"]
    for n in ("n1", "n2", "n3", "n4", "n4_tensor_cores"):
        assert q[n]["us_per_gemv"] > 0 and q[n]["gbs"] > 0
        assert q[n]["of_measured"] == pytest.approx(q[n]["gbs"] / r["peak"], rel=2e-3)
        assert isinstance(q[n]["clocks"]["reasons"], list)
    assert q["ratio_n4_over_n1"] == pytest.approx(q["n4"]["us_per_gemv"] / q["n1"]["us_per_gemv"], rel=1e-3)
    assert q["ratio_n2_over_n1"] == pytest.approx(q["n2"]["us_per_gemv"] / q["n1"]["us_per_gemv"], rel=1e-3)

    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == "GB/s"
    assert e["h2d_bytes_per_step"] == N * 5120 * 4 and e["d2h_bytes_per_step"] == N * 5120 * 4

    k = d["clocks"]
    assert k["sm_max_mhz"] > 0 and isinstance(k["reasons"], list) and "sm_mhz" in k

    # per layer two GEMVs and their two tile combines, then the final RMS kernel
    assert d["gpu_launches"] == STEPS * (4 * LAYERS + 1)

"""Benchmark of the Packed Twin Inference hot path on GB300.

Default line (N=1 GPU): the 4-stream decode weight pass, 64 layers of Q8 gate
and up (17408 x 5120) and down (5120 x 17408) GEMVs with the SiLU and RMS
glue, N = 4 fp32 activation streams chained layer to layer; one step = one
pass over all 18.2 GB of distinct weights (each byte read once per step).
Other lines: ``--workload q8`` (the N-stream Q8 GEMV over distinct
17408 x 5120 matrices), ``twin``, ``twin2``, ``verify``, ``verify_sample``, ``all``.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Metric: effective weight GB/s (algorithmic bytes / device time) with the
fraction of the measured HBM copy bandwidth, plus stream-tokens/s per weight
pass.  ``--impl reference`` times the fp64 CPU oracle on a bounded sample of
the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import contextlib
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "effective weight GB/s (% of GB300 HBM peak) and stream-tokens/s per weight pass"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


GEMV_SOURCES = ("pti_gemv_kernel.cuh", "pti_gemv_tc.cuh", "pti_gemv.cu", "pti_device.cuh", "pti_host.h")
DECODE_SOURCES = GEMV_SOURCES + ("pti_decode.cu",)
VERIFY_SOURCES = ("pti_verify.cu", "pti_device.cuh", "pti_host.h")


def kernel_source_hash(files) -> str:
    """Hash of the CUDA sources a workload's kernels are built from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "stream_quantized_gemv_gb300", "csrc")
    for name in sorted(files):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(wl):
    """DRAM bytes per launch of the workload's dominant kernel from the
    committed ncu summary, if it was taken on the current kernel sources;
    else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d.get(wl.name)
        if e and e.get("kernel_source_hash") == kernel_source_hash(wl.sources):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        # address the GPU by UUID: CUDA_VISIBLE_DEVICES may renumber devices
        self.gpu_id = str(device_index)
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            self.gpu_id = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            pass
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.text = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.text, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        rows = [r for r in csv.reader(io.StringIO(getattr(self, "text", ""))) if len(r) >= 9]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        loaded = sorted(sm)[len(sm) // 2:] if sm else []
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def dist_setup(n_gpus: int):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
Q8_BLOCK = 34
TWIN_BLOCK = 68


class Q8Pass:
    """N-stream Q8 GEMV over L distinct rows x cols matrices (one step = one pass)."""
    sources = GEMV_SOURCES

    def __init__(self, rows=17408, cols=5120, n=4, layers=16, seed=0, w=None, flags=0):
        import torch
        import pti_synth
        import stream_quantized_gemv_gb300 as pti
        self.pti, self.torch = pti, torch
        self.rows, self.cols, self.n, self.layers = rows, cols, n, layers
        self.flags = flags  # FLAG_TENSOR_CORES: the tensor-core consumer
        tc = bool(flags & pti.FLAG_TENSOR_CORES)
        self.name = f"q8_gemv_n{n}_{rows}x{cols}_x{layers}" + ("_tensor_cores" if tc else "")
        self.w = w if w is not None else [pti_synth.q8_matrix_device(rows, cols, seed, 1000 + i)
                                          for i in range(layers)]
        self.x = pti_synth.activations_device(n, cols, seed, 1)
        self.y = torch.empty((n, rows), dtype=torch.float32, device="cuda")
        need = pti.q8_gemv_workspace_bytes(rows, cols, n)
        self.ws = torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda")
        self.weight_bytes = rows * (cols // 32) * Q8_BLOCK
        self.launch_bytes = self.weight_bytes + 4 * n * (rows + cols)
        self.step_bytes = layers * self.launch_bytes
        # each GEMV launch is followed by the launch that combines its shared tiles
        self.launches_per_step = 2 * layers
        self.gemv_launches_per_step = layers
        self.tokens_per_step = n
        self.dominant = ("gemv_tc_kernel<%d>" if tc else "gemv_tma_kernel<Q8,%d>") % n
        self.dtype = "f32"
        # FP32 FMA lane-operations: per weight N products and one dequantising FMA
        self.fma_ops_per_step = layers * rows * cols * (n + 1)

    def step(self, x=None, y=None):
        # a chain of GEMVs as in a decode step: every launch after the first
        # may start while the previous one finishes (programmatic dependent
        # launch; the weights are never written)
        x = self.x if x is None else x
        y = self.y if y is None else y
        for k, w in enumerate(self.w):
            self.pti.q8_gemv_nstream(w, self.rows, self.cols, x, y=y, ws=self.ws,
                                     flags=(self.pti.FLAG_PDL if k > 0 else 0) | self.flags)

    def e2e_buffers(self):
        t = self.torch
        hx = t.empty_like(self.x, device="cpu").pin_memory()
        hx.copy_(self.x.cpu())
        hy = t.empty_like(self.y, device="cpu").pin_memory()
        return hx, hy, self.x, self.y

    def config(self):
        return {"workload": f"N-stream Q8 GEMV weight pass: {self.layers} distinct {self.rows}x{self.cols} "
                            f"Q8 matrices (f16 scale + 32 int8 per 34-byte block), N={self.n} fp32 streams, "
                            "launches after the first with programmatic dependent launch",
                "rows": self.rows, "cols": self.cols, "n_streams": self.n, "matrices_per_step": self.layers,
                "weight_bytes_per_step": self.layers * self.weight_bytes,
                "l2": f"inputs larger than L2: {self.layers * self.weight_bytes / 1e9:.2f} GB of distinct "
                      "weights per step, streamed with an L2 evict-first policy"}

    def cpu_sample(self):
        import oracle
        import pti_synth
        rows = 48
        w = pti_synth.q8_matrix(rows, self.cols, seed=0, tensor_id=1)
        x = pti_synth.activations(self.n, self.cols, seed=0, tensor_id=1)
        sample_bytes = rows * (self.cols // 32) * Q8_BLOCK + 4 * self.n * (rows + self.cols)

        def run():
            oracle.q8_gemv(w, rows, self.cols, x)
        return run, sample_bytes, f"oracle q8_gemv on {rows} of the {self.rows} rows, N={self.n}"


class TwinPass(Q8Pass):
    """SSQ twin GEMV over L distinct twin matrices, `per_model` streams of each
    model (per_model = 2: four tokens per weight load)."""

    def __init__(self, rows=17408, cols=5120, layers=8, seed=0, per_model=1):
        import torch
        import pti_synth
        import stream_quantized_gemv_gb300 as pti
        self.pti, self.torch = pti, torch
        self.rows, self.cols, self.layers, self.per_model = rows, cols, layers, per_model
        self.n = 2 * per_model
        self.name = (f"ssq_twin_gemv_{rows}x{cols}_x{layers}" if per_model == 1
                     else f"ssq_twin_gemv_n{per_model}_{rows}x{cols}_x{layers}")
        self.w = [pti_synth.twin_matrix_device(rows, cols, seed, 2000 + i) for i in range(layers)]
        self.x = pti_synth.activations_device(self.n, cols, seed, 2)
        self.y = torch.empty((self.n, rows), dtype=torch.float32, device="cuda")
        need = pti.lib().pti_ssq_twin_gemv_nstream_workspace_bytes(rows, cols, per_model)
        self.ws = torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda")
        self.weight_bytes = rows * (cols // 32) * TWIN_BLOCK
        self.launch_bytes = self.weight_bytes + 4 * self.n * (rows + cols)
        self.step_bytes = layers * self.launch_bytes
        self.launches_per_step = 2 * layers  # GEMV + tile combine
        self.gemv_launches_per_step = layers
        self.tokens_per_step = self.n
        self.dominant = f"gemv_tma_kernel<Twin,{per_model}>"
        self.dtype = "f32"
        # per element two weights (models A and B), each with per_model products and one dequantising FMA
        self.fma_ops_per_step = layers * rows * cols * 2 * (per_model + 1)

    def step(self, x=None, y=None):
        x = self.x if x is None else x
        y = self.y if y is None else y
        m = self.per_model
        for k, w in enumerate(self.w):
            self.pti.ssq_twin_gemv_nstream(w, self.rows, self.cols, x[:m], x[m:], y_a=y[:m], y_b=y[m:], ws=self.ws,
                                           flags=self.pti.FLAG_PDL if k > 0 else 0)

    def config(self):
        return {"workload": f"SSQ mode-16 twin GEMV: {self.layers} distinct {self.rows}x{self.cols} twin "
                            f"matrices (68-byte blocks), {self.per_model} stream(s) of model A and of model B, "
                            "launches after the first with programmatic dependent launch",
                "rows": self.rows, "cols": self.cols, "matrices_per_step": self.layers,
                "streams_per_model": self.per_model,
                "weight_bytes_per_step": self.layers * self.weight_bytes,
                "l2": f"inputs larger than L2: {self.layers * self.weight_bytes / 1e9:.2f} GB per step"}

    def cpu_sample(self):
        import oracle
        import pti_synth
        rows = 48
        w = pti_synth.twin_matrix(rows, self.cols, seed=0, tensor_id=1)
        x = pti_synth.activations(self.n, self.cols, seed=0, tensor_id=2)
        m = self.per_model
        sample_bytes = rows * (self.cols // 32) * TWIN_BLOCK + 4 * self.n * (rows + self.cols)

        def run():
            for s in range(m):
                oracle.twin_gemv(w, rows, self.cols, x[s], x[m + s])
        return run, sample_bytes, f"oracle twin_gemv on {rows} of the {self.rows} rows, {m} stream(s) per model"


class VerifyBatch(Q8Pass):
    sources = VERIFY_SOURCES

    def __init__(self, steps=4096, n=4, vocab=151936, p=0.6, seed=0):
        import torch
        import pti_synth
        import stream_quantized_gemv_gb300 as pti
        self.pti, self.torch = pti, torch
        self.steps, self.n, self.vocab, self.p = steps, n, vocab, p
        self.name = f"verify_greedy_{steps}x{n}x{vocab}"
        self.logits, self.guess, _ = pti_synth.verify_batch_device(steps, n, vocab, p, seed)
        self.out = (torch.empty((steps, n), dtype=torch.int32, device="cuda"),
                    torch.empty((steps, n - 1), dtype=torch.uint8, device="cuda"),
                    torch.empty(steps, dtype=torch.int32, device="cuda"))
        self.launch_bytes = steps * n * vocab * 4 + steps * n * 4 * 2 + steps * (n - 1) + steps * 4
        self.step_bytes = self.launch_bytes
        self.launches_per_step = 1
        self.tokens_per_step = steps * n
        self.dominant = "verify_greedy_kernel"
        self.dtype = "f32"
        self.x = self.logits
        self.y = self.out[2]

    def step(self, x=None, y=None):
        self.pti.verify_greedy(self.logits, self.guess, *self.out)

    def config(self):
        return {"workload": f"greedy verify batch {self.steps} steps x {self.n} streams x vocab {self.vocab}, "
                            f"N(0,3) logits, planted guesses p={self.p}",
                "l2": f"inputs larger than L2: {self.launch_bytes / 1e9:.2f} GB of logits per step"}

    def cpu_sample(self):
        import oracle
        import pti_synth
        steps = 24
        lg, gs, _ = pti_synth.verify_batch(steps, self.n, self.vocab, self.p, seed=0)
        b = steps * self.n * self.vocab * 4

        def run():
            oracle.verify_greedy(lg, gs)
        return run, b, f"oracle verify_greedy on {steps} of the {self.steps} steps"


class VerifySampleBatch(Q8Pass):
    """Sampling-mode verify of a batch: inverse-CDF draws from softmax(l / T)
    per stream, acceptance against guesses and sum p^2 (one step = one batch)."""
    sources = VERIFY_SOURCES

    def __init__(self, steps=4096, n=4, vocab=151936, temperature=1.0, seed=0):
        import torch
        import pti_synth
        import stream_quantized_gemv_gb300 as pti
        self.pti, self.torch = pti, torch
        self.steps, self.n, self.vocab, self.temperature = steps, n, vocab, temperature
        self.name = f"verify_sample_{steps}x{n}x{vocab}"
        self.logits, self.uniform = pti_synth.sample_batch_device(steps, n, vocab, seed)
        _, u2 = pti_synth.sample_batch_device(steps, n, 1, seed + 1)
        # guesses: independent draws from the same rows (the draft the pages'
        # acceptance rule assumes), so about sum p^2 of them are accepted
        zeros = torch.zeros((steps, n), dtype=torch.int32, device="cuda")
        t2, _, _, _ = pti.verify_sample(self.logits, zeros, u2, temperature, collision=False)
        self.guess = torch.zeros_like(zeros)
        self.guess[:, 1:] = t2[:, :-1]
        del t2, u2
        self.out = (torch.empty((steps, n), dtype=torch.int32, device="cuda"),
                    torch.empty((steps, n - 1), dtype=torch.uint8, device="cuda"),
                    torch.empty(steps, dtype=torch.int32, device="cuda"),
                    torch.empty((steps, n), dtype=torch.float32, device="cuda"))
        self.launch_bytes = steps * n * vocab * 4 + steps * n * 4 * 2 + steps * n * 4 * 2 + steps * (n - 1) + steps * 4
        self.step_bytes = self.launch_bytes
        self.launches_per_step = 1
        self.tokens_per_step = steps * n
        self.dominant = "verify_sample_kernel"
        self.dtype = "f32"
        self.x = self.logits
        self.y = self.out[2]

    def step(self, x=None, y=None):
        t, m, a, c = self.out
        self.pti.verify_sample(self.logits, self.guess, self.uniform, self.temperature, token=t, match=m,
                               accept=a, collision=c)

    def config(self):
        return {"workload": f"sampling verify batch {self.steps} steps x {self.n} streams x vocab {self.vocab}, "
                            f"N(0,3) logits, T={self.temperature}, uniform draws, guesses drawn independently "
                            "from the same rows",
                "l2": f"inputs larger than L2: {self.launch_bytes / 1e9:.2f} GB of logits per step"}

    def cpu_sample(self):
        import numpy as np
        import oracle
        import pti_synth
        steps = 16
        lg, u = pti_synth.sample_batch(steps, self.n, self.vocab, seed=0)
        gs = np.zeros((steps, self.n), np.int32)
        b = steps * self.n * self.vocab * 4

        def run():
            oracle.verify_sample(lg, gs, u, self.temperature)
        return run, b, f"oracle verify_sample on {steps} of the {self.steps} steps"


class DecodePass(Q8Pass):
    """The chained decode weight pass: L layers of gate/up/down Q8 GEMVs with
    the fused SiLU and RMS glue, N streams (one step = one pass)."""
    sources = DECODE_SOURCES

    def __init__(self, hidden=5120, ffn=17408, n=4, layers=64, seed=0):
        import torch
        import pti_synth
        import stream_quantized_gemv_gb300 as pti
        self.pti, self.torch = pti, torch
        self.hidden, self.ffn, self.n, self.layers = hidden, ffn, n, layers
        self.name = f"mlp_decode_pass_n{n}_{hidden}x{ffn}_x{layers}"
        gate = [pti_synth.q8_matrix_device(ffn, hidden, seed, 3 * l) for l in range(layers)]
        up = [pti_synth.q8_matrix_device(ffn, hidden, seed, 3 * l + 1) for l in range(layers)]
        down = [pti_synth.q8_matrix_device(hidden, ffn, seed, 3 * l + 2) for l in range(layers)]
        self.weights = pti.DecodeWeights(gate, up, down)
        self.x = pti_synth.activations_device(n, hidden, seed, 1000)
        self.y = torch.empty((n, hidden), dtype=torch.float32, device="cuda")
        need = pti.mlp_decode_pass_workspace_bytes(hidden, ffn, n)
        self.ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
        self.weight_bytes = 3 * ffn * (hidden // 32) * Q8_BLOCK   # per layer
        # algorithmic bytes: every weight once, each kernel's input and output vectors once
        act = 4 * n * ((hidden + ffn) + (ffn + hidden))
        self.step_bytes = layers * (self.weight_bytes + act) + 4 * n * 2 * hidden
        self.launch_bytes = self.step_bytes / (2 * layers)       # mean over the pass's GEMV launches
        # per layer: gate/up GEMV, its tile combine, down GEMV, its tile combine;
        # then the final RMS kernel
        self.launches_per_step = 4 * layers + 1
        self.gemv_launches_per_step = 2 * layers
        self.fma_ops_per_step = layers * 3 * ffn * hidden * (n + 1)
        self.tokens_per_step = n
        self.dominant = f"gemv_tma_kernel<Q8,{n},GateUp|Down> (the pass's {2 * layers} GEMV launches)"
        self.dtype = "f32"

    def step(self, x=None, y=None):
        x = self.x if x is None else x
        y = self.y if y is None else y
        self.pti.mlp_decode_pass(self.weights, self.hidden, self.ffn, x, x_out=y, ws=self.ws)

    def config(self):
        return {"workload": f"{self.layers}-layer decode weight pass, N={self.n} fp32 streams: per layer Q8 gate "
                            f"and up {self.ffn}x{self.hidden}, SiLU(g)*u, RMS, Q8 down {self.hidden}x{self.ffn}, "
                            "RMS; distinct random weights per layer",
                "hidden": self.hidden, "ffn": self.ffn, "n_streams": self.n, "layers": self.layers,
                "weight_bytes_per_step": self.layers * self.weight_bytes,
                "l2": f"inputs larger than L2: {self.layers * self.weight_bytes / 1e9:.2f} GB of distinct "
                      "weights per step, streamed with an L2 evict-first policy"}

    def cpu_sample(self):
        import oracle
        import pti_synth
        hidden, ffn = 1024, 3584     # one layer of the same structure at a fifth of the width
        wg = pti_synth.q8_matrix(ffn, hidden, seed=0, tensor_id=0)
        wu = pti_synth.q8_matrix(ffn, hidden, seed=0, tensor_id=1)
        wd = pti_synth.q8_matrix(hidden, ffn, seed=0, tensor_id=2)
        x = pti_synth.activations(self.n, hidden, seed=0, tensor_id=1000)
        b = 3 * ffn * (hidden // 32) * Q8_BLOCK + 4 * self.n * 2 * (hidden + ffn)

        def run():
            oracle.mlp_layer(wg, wu, wd, hidden, ffn, x)
        return run, b, f"oracle mlp_layer: one {hidden}x{ffn} layer (gate, up, down), N={self.n}"


class SelfSpecLoop(Q8Pass):
    """The device-resident greedy self-speculative loop on a toy model at the
    pages' Qwen3.6-27B shapes (vocab 151936, hidden 5120, ffn 17408): per loop
    step the embedding gather, one decode layer, the LM head and greedy verify
    for N streams.  One bench step = one call running `loop_steps` steps."""
    sources = DECODE_SOURCES + ("pti_verify.cu", "pti_selfspec.cu")

    def __init__(self, vocab=151936, hidden=5120, ffn=17408, n=4, loop_steps=16, seed=0):
        import torch
        import pti_synth
        import stream_quantized_gemv_gb300 as pti
        self.pti, self.torch = pti, torch
        self.vocab, self.hidden, self.ffn, self.n, self.loop_steps = vocab, hidden, ffn, n, loop_steps
        self.name = f"selfspec_greedy_n{n}_{vocab}x{hidden}x{ffn}_x{loop_steps}"
        self.emb = pti_synth.activations_device(vocab, hidden, seed, 40)
        self.wg = pti_synth.q8_matrix_device(ffn, hidden, seed, 41)
        self.wu = pti_synth.q8_matrix_device(ffn, hidden, seed, 42)
        self.wd = pti_synth.q8_matrix_device(hidden, ffn, seed, 43)
        self.wh = pti_synth.q8_matrix_device(vocab, hidden, seed, 44)
        need = pti.selfspec_greedy_workspace_bytes(vocab, hidden, ffn, n)
        self.ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
        self.out = (torch.zeros(loop_steps * n, dtype=torch.int32, device="cuda"),
                    torch.zeros(1, dtype=torch.int32, device="cuda"),
                    torch.zeros(loop_steps, dtype=torch.int32, device="cuda"))
        layer = 3 * ffn * (hidden // 32) * Q8_BLOCK
        head = vocab * (hidden // 32) * Q8_BLOCK
        # algorithmic bytes of a loop step: every weight once, the N embedding
        # rows, the layer's and the head's activations, the logits written by
        # the head and read by verify
        act = 4 * n * (hidden + 2 * (hidden + ffn) + hidden) + 4 * n * 2 * hidden
        self.weight_bytes = layer + head
        self.step_bytes = loop_steps * (layer + head + act + 2 * 4 * n * vocab)
        # per loop step: gather, gate/up + combine, down + combine, RMS,
        # head + combine, argmax, verify rule + window update; one window init per call
        self.launches_per_step = 10 * loop_steps + 1
        self.gemv_launches_per_step = 3 * loop_steps
        self.launch_bytes = self.step_bytes / self.gemv_launches_per_step
        self.fma_ops_per_step = loop_steps * (3 * ffn * hidden + vocab * hidden) * (n + 1)
        self.step()
        torch.cuda.synchronize()
        self.tokens_per_step = int(self.out[1].item())   # confirmed tokens per call
        self.dominant = f"gemv_tma_kernel<Q8,{n}> (LM head {vocab}x{hidden} and the layer's GEMVs)"
        self.dtype = "f32"

    def step(self, x=None, y=None):
        self.pti.selfspec_greedy(self.emb, self.wg, self.wu, self.wd, self.wh, self.vocab, self.hidden, self.ffn,
                                 self.n, 7, self.loop_steps, ws=self.ws, out=self.out)

    def e2e_buffers(self):
        # the first token is a scalar argument: nothing to copy in; the
        # confirmed tokens and their count come back
        t = self.torch
        hy = t.empty_like(self.out[0], device="cpu").pin_memory()
        return None, hy, None, self.out[0]

    def config(self):
        return {"workload": f"greedy self-speculative loop, N={self.n} streams, {self.loop_steps} loop steps per "
                            f"call, toy model at vocab {self.vocab}, hidden {self.hidden}, ffn {self.ffn}: fp32 "
                            "embedding, one Q8 gated-MLP layer, Q8 LM head, random weights (about one confirmed "
                            "token per loop step: the window rarely holds the model's continuation)",
                "confirmed_tokens_per_call": self.tokens_per_step,
                "weight_bytes_per_loop_step": self.weight_bytes,
                "l2": f"inputs larger than L2: {self.weight_bytes / 1e9:.2f} GB of weights per loop step"}

    def cpu_sample(self):
        import numpy as np
        import oracle
        import pti_synth
        vocab, hidden, ffn = 4096, 1024, 3584   # the same structure at a fifth of the width
        m = pti_synth.toy_model(vocab, hidden, ffn, seed=0)
        toks = np.arange(self.n) * 5
        b = 3 * ffn * (hidden // 32) * Q8_BLOCK + vocab * (hidden // 32) * Q8_BLOCK

        def run():
            oracle.toy_logits(m["embedding"], m["w_gate"], m["w_up"], m["w_down"], m["w_head"], vocab, hidden,
                              ffn, toks)
        return run, b, f"oracle toy_logits of {self.n} window tokens, vocab {vocab}, hidden {hidden}, ffn {ffn}"


WORKLOADS = {
    "decode": lambda a: DecodePass(a.cols or 5120, a.rows or 17408, a.n, a.layers or 64),
    "q8": lambda a: Q8Pass(a.rows or 17408, a.cols or 5120, a.n, a.layers or 16,
                           flags=0x4 if a.cores == "tensor" else 0),
    "twin": lambda a: TwinPass(a.rows or 17408, a.cols or 5120, a.layers or 8),
    "twin2": lambda a: TwinPass(a.rows or 17408, a.cols or 5120, a.layers or 8, per_model=2),
    "verify": lambda a: VerifyBatch(steps=a.vsteps),
    "verify_sample": lambda a: VerifySampleBatch(steps=a.vsteps),
    "selfspec": lambda a: SelfSpecLoop(n=a.n, loop_steps=a.layers or 16),
}


# ---------------------------------------------------------------------------
# timing
# ---------------------------------------------------------------------------
def time_gpu(wl, steps, warmup, world, local):
    import torch
    torch.cuda.synchronize()
    for _ in range(warmup):
        wl.step()
    torch.cuda.synchronize()
    # CUDA graph of one step (all launches of the pass), replayed K times
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        wl.step()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            wl.step()
    torch.cuda.synchronize()
    for _ in range(max(1, warmup)):
        g.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(steps):
            g.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    ms = ev0.elapsed_time(ev1)
    ms = max_over_ranks(ms, world)
    return ms / steps, clk.summary()


def time_e2e(wl, steps, warmup):
    """Same pass through the public API with inputs in pinned host memory:
    per step H2D of the step's inputs, the pass, D2H of the result.  For the
    verify batches the logits are the model's output, already on the device;
    the host supplies the guesses (and, for sampling, the uniform numbers)."""
    import torch

    def pinned(d):
        h = torch.empty_like(d, device="cpu").pin_memory()
        h.copy_(d.cpu())
        return h

    if isinstance(wl, (VerifyBatch, VerifySampleBatch)):
        ins = [(pinned(wl.guess), wl.guess)]
        if isinstance(wl, VerifySampleBatch):
            ins.append((pinned(wl.uniform), wl.uniform))
        hy, dy = pinned(wl.out[2]), wl.out[2]
    else:
        hx, hy, dx, dy = wl.e2e_buffers()
        ins = [] if hx is None else [(hx, dx)]
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        for h, d in ins:
            d.copy_(h, non_blocking=True)
        wl.step()
        hy.copy_(dy, non_blocking=True)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        for h, d in ins:
            d.copy_(h, non_blocking=True)
        wl.step()
        hy.copy_(dy, non_blocking=True)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / steps
    return ms, sum(h.numel() * h.element_size() for h, _ in ins), hy.numel() * hy.element_size()


def host_cores() -> int:
    """Host cores online (sysconf), the thread count of the all-core oracle."""
    try:
        return int(os.sysconf("SC_NPROCESSORS_ONLN"))
    except (ValueError, OSError, AttributeError):
        return os.cpu_count() or 1


def time_cpu(wl, budget_s=8.0):
    """The oracle on a bounded sample of the workload: single-threaded, and with
    its row loops split over all host cores (OpenMP build of the same source).
    Returns (all-core GB/s, cores, single-core GB/s, sample description,
    seconds per sample on all cores)."""
    import oracle
    run, sample_bytes, what = wl.cpu_sample()

    def rate():
        t0 = time.perf_counter()
        run()
        one = time.perf_counter() - t0
        reps = max(1, min(100000, int(budget_s / max(one, 1e-6))))
        t0 = time.perf_counter()
        for _ in range(reps):
            run()
        return (time.perf_counter() - t0) / reps

    oracle.use_all_cores(False)
    dt1 = rate()
    cores = 1
    dtn = dt1
    if oracle.has_all_cores():
        oracle.use_all_cores(True)
        try:
            dtn = rate()
            cores = host_cores()
        finally:
            oracle.use_all_cores(False)
    return sample_bytes / dtn / 1e9, cores, sample_bytes / dt1 / 1e9, what, dtn


def q8_target(a, world, local, peak, peak_kind):
    """The 4-stream Q8 GEMV on 17408 x 5120 against the 1-stream one, in the
    same harness (16 distinct matrices per step, launches after the first
    chained by programmatic dependent launch, CUDA-graph replay): time per
    GEMV, effective GB/s, fractions of the measured and the nominal HBM rate,
    and the step-time ratios N / N=1 (N = 2, 3, 4); also N=4 with the products
    on the tensor core (the opt-in consumer) for comparison."""
    import torch
    import stream_quantized_gemv_gb300 as pti
    out = {"shape": "17408x5120", "matrices_per_step": 16, "steps": a.steps}
    shared = None
    for n, key, flags in ((1, "n1", 0), (2, "n2", 0), (3, "n3", 0), (4, "n4", 0),
                          (4, "n4_tensor_cores", pti.FLAG_TENSOR_CORES)):
        wl = Q8Pass(17408, 5120, n, 16, w=shared, flags=flags)
        shared = wl.w
        ms, clocks = time_gpu(wl, a.steps, a.warmup, world, local)
        us = ms * 1e3 / wl.layers
        gbs = wl.launch_bytes / (us * 1e-6) / 1e9
        out[key] = {"us_per_gemv": round(us, 3), "gbs": round(gbs, 1),
                        "of_measured": round(gbs / peak, 4), "of_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
                        "stream_tokens_per_s": round(n / (us * 1e-6), 1), "clocks": clocks}
        del wl
    out["ratio_n4_over_n1"] = round(out["n4"]["us_per_gemv"] / out["n1"]["us_per_gemv"], 4)
    out["ratio_n2_over_n1"] = round(out["n2"]["us_per_gemv"] / out["n1"]["us_per_gemv"], 4)
    out["ratio_n3_over_n1"] = round(out["n3"]["us_per_gemv"] / out["n1"]["us_per_gemv"], 4)
    out["peak_kind"] = peak_kind
    del shared
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="decode", choices=sorted(WORKLOADS) + ["all"])
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--n", type=int, default=4)
    ap.add_argument("--rows", type=int, default=0)
    ap.add_argument("--cols", type=int, default=0)
    ap.add_argument("--layers", type=int, default=0)
    ap.add_argument("--vsteps", type=int, default=4096, help="steps of the verify batches")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cores", default="cuda", choices=["cuda", "tensor"],
                    help="q8 workload: the GEMV's products on the CUDA cores (default) or the tensor core")
    ap.add_argument("--no-q8-target", action="store_true",
                    help="decode line: skip the 17408x5120 Q8 GEMV timing at N = 1 and N = 4")
    a = ap.parse_args()
    a.warmup = max(a.warmup, 3)

    rank, world, local = dist_setup(a.gpus)
    names = sorted(WORKLOADS) if a.workload == "all" else [a.workload]

    if a.impl == "reference":
        if rank != 0:
            return
        import oracle
        oracle.build()
        for name in names:
            wl = _cpu_only_workload(name, a)
            run, sample_bytes, what = wl.cpu_sample()
            cores = 1
            if oracle.has_all_cores():
                oracle.use_all_cores(True)
                cores = host_cores()
            for _ in range(a.warmup):
                run()
            t0 = time.perf_counter()
            for _ in range(a.steps):
                run()
            dt = (time.perf_counter() - t0) / a.steps
            v = sample_bytes / dt / 1e9
            line = {"metric": METRIC, "value": round(v, 6), "unit": "GB/s", "n_gpus": a.gpus,
                    "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(dt * 1e3, 4),
                    "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                    "dtype": "f64", "data": "synthetic", "impl": "reference",
                    "config": wl.config(),
                    "cpu_baseline": {"value": round(v, 6), "unit": "GB/s", "cores": cores, "kind": "oracle",
                                     "sample": what},
                    "e2e": {"value": round(v, 6), "unit": "GB/s", "h2d_bytes_per_step": 0,
                            "d2h_bytes_per_step": 0}}
            print(json.dumps(line), flush=True)
        return

    import torch
    import stream_quantized_gemv_gb300 as pti
    pti.build()
    pti.lib()
    peak, peak_kind = measured_peaks()
    for name in names:
        wl = WORKLOADS[name](a)
        ms, clocks = time_gpu(wl, a.steps, a.warmup, world, local)
        e2e_ms, h2d, d2h = time_e2e(wl, max(3, a.steps // 2), 2)
        err = pti.device_error()
        value = wl.step_bytes * world / (ms * 1e-3) / 1e9
        per_launch_ms = ms / getattr(wl, "gemv_launches_per_step", wl.launches_per_step)
        achieved = wl.launch_bytes / (per_launch_ms * 1e-3) / 1e9
        traffic = recorded_traffic(wl)
        line = {"metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
                "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(ms, 5),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": wl.dtype, "data": "synthetic (seeded; no model weights)",
                "config": wl.config(),
                "stream_tokens_per_s": round(wl.tokens_per_step * world / (ms * 1e-3), 2),
                "hbm_frac": {"of_measured": round(value / world / peak, 4), "measured_gbs": peak,
                             "peak_kind": peak_kind, "of_nominal_8tbs": round(value / world / NOMINAL_HBM_GBS, 4)},
                "roofline": {"bound": "hbm", "kernel": wl.dominant, "achieved": round(achieved, 2),
                             "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                             "peak_kind": peak_kind, "traffic": traffic,
                             "algorithmic_bytes_per_launch": wl.launch_bytes,
                             "avg_launch_us": round(per_launch_ms * 1e3, 3)},
                "e2e": {"value": round(wl.step_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                        "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
                "gpu_launches": wl.launches_per_step * a.steps,
                "clocks": clocks, "device_error": err}
        fma_ops = getattr(wl, "fma_ops_per_step", None)
        if fma_ops:
            # the 4-stream GEMVs are limited by FP32 arithmetic on the CUDA
            # cores as much as by HBM: FMA lane-operations per second against
            # 128 FP32 lanes per SM x SMs x the SM clock sampled under load
            sms = torch.cuda.get_device_properties(local).multi_processor_count
            mhz = clocks.get("sm_mhz") or clocks.get("sm_max_mhz") or 2070.0
            fma_peak = 128.0 * sms * mhz * 1e6
            fma_rate = fma_ops / (ms * 1e-3)
            line["alu_roofline"] = {"bound": "alu", "kernel": wl.dominant, "unit": "FMA lane-ops/s",
                                    "achieved": round(fma_rate, 1), "peak": round(fma_peak, 1),
                                    "frac": round(fma_rate / fma_peak, 4),
                                    "peak_derivation": f"128 FP32 lanes x {sms} SMs x {mhz:.0f} MHz",
                                    "ops": "per weight: N product FMAs + 1 dequantising FMA"}
        if name == "decode" and not a.no_q8_target:
            line["q8_target"] = q8_target(a, world, local, peak, peak_kind)
        if rank == 0 and world == 1 and not a.no_cpu_baseline:
            import oracle
            oracle.build()
            v, cores, v1, what, dt = time_cpu(wl)
            line["cpu_baseline"] = {"value": round(v, 6), "unit": "GB/s", "cores": cores, "kind": "oracle",
                                    "sample": what, "seconds_per_sample": round(dt, 4),
                                    "single_core_value": round(v1, 6),
                                    "threads": "row loops split over all host cores (OpenMP build of the oracle)"}
        if rank == 0:
            print(json.dumps(line), flush=True)
        del wl
        torch.cuda.empty_cache()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


class _CpuOnly:
    pass


def _cpu_only_workload(name, a):
    """The workload's config and CPU sample without allocating device memory."""
    cls = {"decode": DecodePass, "q8": Q8Pass, "twin": TwinPass, "twin2": TwinPass, "verify": VerifyBatch,
           "verify_sample": VerifySampleBatch, "selfspec": SelfSpecLoop}[name]
    wl = cls.__new__(cls)
    if name == "selfspec":
        wl.vocab, wl.hidden, wl.ffn, wl.n, wl.loop_steps = 151936, 5120, 17408, a.n, a.layers or 16
        wl.weight_bytes = 3 * wl.ffn * (wl.hidden // 32) * Q8_BLOCK + wl.vocab * (wl.hidden // 32) * Q8_BLOCK
        wl.tokens_per_step = None
    elif name == "decode":
        wl.hidden, wl.ffn, wl.n, wl.layers = a.cols or 5120, a.rows or 17408, a.n, a.layers or 64
        wl.weight_bytes = 3 * wl.ffn * (wl.hidden // 32) * Q8_BLOCK
    elif name == "q8":
        wl.rows, wl.cols, wl.n, wl.layers = a.rows or 17408, a.cols or 5120, a.n, a.layers or 16
        wl.weight_bytes = wl.rows * (wl.cols // 32) * Q8_BLOCK
    elif name in ("twin", "twin2"):
        wl.per_model = 2 if name == "twin2" else 1
        wl.rows, wl.cols, wl.n, wl.layers = a.rows or 17408, a.cols or 5120, 2 * wl.per_model, a.layers or 8
        wl.weight_bytes = wl.rows * (wl.cols // 32) * TWIN_BLOCK
    elif name == "verify_sample":
        wl.steps, wl.n, wl.vocab, wl.temperature = a.vsteps, 4, 151936, 1.0
        wl.launch_bytes = wl.steps * wl.n * wl.vocab * 4
    else:
        wl.steps, wl.n, wl.vocab, wl.p = a.vsteps, 4, 151936, 0.6
        wl.launch_bytes = wl.steps * wl.n * wl.vocab * 4
    return wl


if __name__ == "__main__":
    main()

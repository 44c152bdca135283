"""Benchmark of the MXFP4 training hot path on GB300.

A step is one pass of the whole hot path for one linear layer of a training
step: the fused quantization of the activation X, the weight W and the output
gradient dY (each in both orientations in one pass), then the three
block-scaled MXFP4 GEMMs Fprop Y = X W^T, Dgrad dX = dY W, Wgrad dW = dY^T X.

Default workload (N = 1): the 70B-dense-shaped layer (tokens 16384, d 8192,
ffn 28672): X ~ Student-t(4), W ~ N(0, 0.02), dY ~ Laplace(0, 1e-3) with 0.1% of
entries x100, all bf16; W and dY in 32x32 blocks, X in 1x32 blocks; round-up
scales; Fprop operands nearest-even without rotation; Dgrad's dY by stochastic
rounding; the Wgrad operands (dY and X column-wise) with the random-sign
32-point rotation and stochastic rounding.

Prints one JSON line. `value` = GEMM FLOPs of the step / step time (the
quantization time included), TFLOP/s summed over ranks; the parts (GEMM
TFLOP/s against the dense FP4 peak, quantizer GB/s against the HBM peak) are
reported alongside, with the roofline of the dominant kernel.

At N = 1 the default run then measures the pages' other configurations
briefly (`other_configs`: the tiny layer, the 2D-block consistency check,
the Llama-3.1-8B-shaped MLP step and the square sweep), outside the headline's
timed region.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
       [--workload NAME] [--no-cpu-baseline] [--no-e2e] [--no-configs]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time
from dataclasses import dataclass, field, replace

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MXFP4 GEMM TFLOPS (% FP4 peak); fused RHT+quantize GB/s (% HBM peak)"
FP4_OVER_BF16 = 13.5 / 2.25        # nominal dense FP4 : BF16 tensor rate
NOMINAL_FP4_TFLOPS = 13500.0       # NVIDIA's dense FP4 figure for one GB300 (context)
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# Training-step workloads: name -> (tokens T, d D, ffn F, data seed, description).
LAYERS = {
    "70b-layer": (16384, 8192, 28672, 1003,
                  "70B-dense-shaped layer training step: tokens 16384, d 8192, ffn 28672"),
    "8b-mlp-up": (8192, 4096, 14336, 1002,
                  "Llama-3.1-8B-shaped MLP up-proj training step: tokens 8192, d 4096, ffn 14336"),
    "70b-layer-det": (16384, 8192, 28672, 1003,
                      "70B-dense-shaped layer training step, deterministic rotation: tokens 16384, "
                      "d 8192, ffn 28672"),
    "70b-layer-nvfp4": (16384, 8192, 28672, 1003,
                        "70B-dense-shaped layer training step in NVFP4 (1x16 blocks, E4M3 scales "
                        "under per-tensor power-of-two factors): tokens 16384, d 8192, ffn 28672"),
}
# Square sweep points: quantize A and B (1x32 floor nearest-even) + one n^3 GEMM.
SQUARES = {f"sq{n}": n for n in (1024, 2048, 4096, 8192, 16384)}
# Quantize-only workload: the 2D-block consistency check (W [4096, 4096]).
TWO_D = "2d-blocks"
WORKLOADS = sorted(LAYERS) + ["tiny", TWO_D] + sorted(SQUARES, key=lambda k: SQUARES[k])


# ------------------------------------------------------------ workloads ---

@dataclass
class QuantOp:
    name: str
    rows: int
    cols: int
    dist: tuple           # ("t", df) | ("normal", std) | ("laplace", b, outlier_frac) | ("outcols", n, mult)
    seed: int
    prow: object          # gemm_pt_block_gb300.QuantParams or None
    pcol: object


@dataclass
class GemmOp:
    label: str
    a: tuple              # (input name, "row" | "col")
    b: tuple
    M: int
    N: int
    K: int


@dataclass
class Spec:
    name: str
    desc: str
    quants: list = field(default_factory=list)
    gemms: list = field(default_factory=list)
    nvfp4: bool = False   # 1x16 blocks with E4M3 scales; GEMMs through nvfp4_gemm

    def scale_bytes_per_elem(self) -> float:
        return 1 / 16 if self.nvfp4 else 1 / 32

    def quant_bytes(self):
        """Algorithmic bytes per quantize launch: read the bf16 input once, write
        each requested orientation's codes (0.5 B/elem) and scales (1/32 B/elem;
        1/16 for NVFP4)."""
        sb = self.scale_bytes_per_elem()
        return [q.rows * q.cols * (2 + ((q.prow is not None) + (q.pcol is not None)) * (0.5 + sb))
                for q in self.quants]

    def gemm_flops(self):
        return [2.0 * g.M * g.N * g.K for g in self.gemms]

    def labels(self):
        return [f"quantize {q.name}" for q in self.quants] + [f"gemm {g.label}" for g in self.gemms]


def make_spec(name: str) -> Spec:
    import gemm_pt_block_gb300 as mx
    import synth

    P, mma = mx.QuantParams, mx.LAYOUT_MMA
    if name in LAYERS:
        T, D, F, seed, desc = LAYERS[name]
        big = name.startswith("70b-layer")
        mask = 0 if name.endswith("-det") else synth.sign_mask(seed)
        # 70B step: W, dY in 32x32 blocks, round-up scales, random-sign rotation
        # for Wgrad, SR on Dgrad's dY. 8B step: 1x32 floor, deterministic
        # rotation + SR for the Wgrad operands only. Each tensor has its own
        # Philox stream (X: 0, dY: 1); both orientations of dY share it, so a
        # source element draws the same bits for Dgrad and Wgrad.
        wblk = mx.BLOCK_32X32 if big else mx.BLOCK_1X32
        smode = mx.SCALE_ROUNDUP if big else mx.SCALE_FLOOR
        wmask = mask if big else 0
        dgrad = mx.ROUND_SR if big else mx.ROUND_RTN
        s = Spec(name, desc)
        s.quants = [
            QuantOp("X", T, D, ("t", 4.0), seed,
                    P(mx.BLOCK_1X32, smode, mx.ROUND_RTN, mma),
                    P(mx.BLOCK_1X32, smode, mx.ROUND_SR, mma, True, wmask, 1, 0)),
            QuantOp("W", F, D, ("normal", 0.02), seed + 100,
                    P(wblk, smode, mx.ROUND_RTN, mma), P(wblk, smode, mx.ROUND_RTN, mma)),
            QuantOp("dY", T, F, ("laplace", 1e-3, 0.001 if big else 0.0), seed + 200,
                    P(wblk, smode, dgrad, mma, False, 0, 1, 1),
                    P(wblk, smode, mx.ROUND_SR, mma, True, wmask, 1, 1)),
        ]
        s.gemms = [GemmOp("Fprop", ("X", "row"), ("W", "row"), T, F, D),
                   GemmOp("Dgrad", ("dY", "row"), ("W", "col"), T, D, F),
                   GemmOp("Wgrad", ("dY", "col"), ("X", "col"), F, D, T)]
        if name.endswith("-nvfp4"):
            # The same recipe with every block 1x16 (E4M3 scales, round-up);
            # each tensor's factor 2^k comes from its max-abs (set in Step).
            s.nvfp4 = True
            for q in s.quants:
                q.prow = replace(q.prow, block=mx.BLOCK_1X16, scale_mode=mx.SCALE_ROUNDUP)
                q.pcol = replace(q.pcol, block=mx.BLOCK_1X16, scale_mode=mx.SCALE_ROUNDUP)
        return s
    if name == TWO_D:
        s = Spec(name, "2D-block consistency: W [4096,4096] N(0,0.02) bf16; 32x32 blocks, round-up "
                       "scales, nearest-even, no rotation; W and W^T quantized in one pass")
        p = P(mx.BLOCK_32X32, mx.SCALE_ROUNDUP, mx.ROUND_RTN, mx.LAYOUT_MMA)
        s.quants = [QuantOp("W", 4096, 4096, ("normal", 0.02), 1001, p, p)]
        return s
    if name == "tiny":
        mask = synth.sign_mask(1000)
        s = Spec(name, "tiny: X [512,1024] N(0,1) with 8 outlier columns x50, W [512,1024] N(0,0.02); "
                       "random-sign rotation, 1x32 floor; W nearest-even, X SR seed 0; Y = Xq Wq^T")
        s.quants = [
            QuantOp("X", 512, 1024, ("outcols", 8, 50.0), 1000,
                    P(mx.BLOCK_1X32, mx.SCALE_FLOOR, mx.ROUND_SR, mma, True, mask, 0, 0), None),
            QuantOp("W", 512, 1024, ("normal", 0.02), 1100,
                    P(mx.BLOCK_1X32, mx.SCALE_FLOOR, mx.ROUND_RTN, mma, True, mask), None)]
        s.gemms = [GemmOp("Fprop", ("X", "row"), ("W", "row"), 512, 512, 1024)]
        return s
    n = SQUARES[name]
    s = Spec(name, f"square sweep point n={n}: A, B [{n},{n}] ~ t(3) bf16, 1x32 floor nearest-even; C = A B^T")
    p = P(mx.BLOCK_1X32, mx.SCALE_FLOOR, mx.ROUND_RTN, mma)
    s.quants = [QuantOp("A", n, n, ("t", 3.0), 1004, p, None),
                QuantOp("B", n, n, ("t", 3.0), 1104, p, None)]
    s.gemms = [GemmOp("C", ("A", "row"), ("B", "row"), n, n, n)]
    return s


def gen_input(q: QuantOp, device, rows=None, cols=None, seed_offset=0):
    """Seeded bf16 input of the op's distribution (device tensor, or CPU for the oracle)."""
    import synth

    r = q.rows if rows is None else rows
    c = q.cols if cols is None else cols
    seed = q.seed + seed_offset
    kind = q.dist[0]
    if str(device) == "cpu":
        if kind == "t":
            return synth.student_t(r, c, q.dist[1], seed)
        if kind == "normal":
            return synth.normal(r, c, q.dist[1], seed)
        if kind == "laplace":
            return synth.laplace(r, c, q.dist[1], seed, outlier_frac=q.dist[2])
        return synth.normal_outlier_cols(r, c, 1.0, q.dist[1], q.dist[2], seed)
    if kind == "t":
        return synth.dev_student_t(r, c, q.dist[1], seed, device)
    if kind == "normal":
        return synth.dev_normal(r, c, q.dist[1], seed, device)
    if kind == "laplace":
        return synth.dev_laplace(r, c, q.dist[1], seed, device, outlier_frac=q.dist[2])
    return synth.normal_outlier_cols(r, c, 1.0, q.dist[1], q.dist[2], seed).to(device)


class Step:
    """Device inputs, preallocated outputs and the launch sequence of one step."""

    def __init__(self, spec: Spec, device):
        import torch

        import gemm_pt_block_gb300 as mx

        self.spec = spec
        u8 = torch.uint8
        self.inputs, self.bufs, self.outs, self.params = {}, {}, {}, {}
        for q in spec.quants:
            self.inputs[q.name] = gen_input(q, device)
            prow, pcol = q.prow, q.pcol
            if spec.nvfp4:   # per-tensor factor from the tensor's max-abs (on the device)
                k = mx.nvfp4_tensor_exp(self.inputs[q.name])
                prow = prow and replace(prow, tensor_exp=k)
                pcol = pcol and replace(pcol, tensor_exp=k)
            self.params[q.name] = (prow, pcol)
            r, c = q.rows, q.cols
            ns = int(r * c * spec.scale_bytes_per_elem())
            self.bufs[q.name] = (
                torch.empty(r, c // 2, dtype=u8, device=device) if q.prow else None,
                torch.empty(ns, dtype=u8, device=device) if q.prow else None,
                torch.empty(c, r // 2, dtype=u8, device=device) if q.pcol else None,
                torch.empty(ns, dtype=u8, device=device) if q.pcol else None)
        for g in spec.gemms:
            self.outs[g.label] = torch.empty(g.M, g.N, device=device)
        # NVFP4: each step also takes every tensor's max-abs on the device, the
        # per-tensor factors of the next step (delayed scaling)
        self.amax = {q.name: (torch.empty(1, device=device), torch.empty(1, dtype=torch.int32, device=device))
                     for q in spec.quants} if spec.nvfp4 else {}
        # one workspace for the GEMMs' scale images (the largest the step needs)
        blk = 16 if spec.nvfp4 else 32
        self.ws = torch.empty(max([mx.gemm_workspace_size(g.M, g.N, g.K, blk) for g in spec.gemms],
                                  default=0), dtype=u8, device=device)
        torch.cuda.empty_cache()

    @property
    def ops(self):
        return len(self.spec.quants) + len(self.spec.gemms)

    @property
    def launches(self):
        """Kernel launches per step: one per quantize, two per GEMM (the scale
        images for the tensor-memory copies, then the GEMM) when it uses the
        workspace, which every CTA-pair shape (M % 256 == 0) does; for NVFP4
        two per tensor for its max-abs and exponent."""
        return (len(self.spec.quants) + sum(2 if g.M % 256 == 0 else 1 for g in self.spec.gemms)
                + 2 * len(self.amax))

    def operand(self, ref):
        q, s, qc, sc = self.bufs[ref[0]]
        return (q, s) if ref[1] == "row" else (qc, sc)

    def tensor_exp(self, ref) -> int:
        prow, pcol = self.params[ref[0]]
        return (prow if ref[1] == "row" else pcol).tensor_exp

    def run(self, inputs=None, events=None, outs=None):
        """Enqueue the step on the current stream; events[i], events[i+1] bracket launch i.
        `inputs` / `outs` replace the step's own input and GEMM output tensors."""
        import gemm_pt_block_gb300 as mx

        inp = self.inputs if inputs is None else inputs
        out = self.outs if outs is None else outs
        k = 0
        if events is not None:
            events[0].record()
        for q in self.spec.quants:
            qr, sr, qc, sc = self.bufs[q.name]
            prow, pcol = self.params[q.name]
            mx.mxfp4_quantize(inp[q.name], prow, pcol, q_row=qr, s_row=sr, q_col=qc, s_col=sc)
            k += 1
            if events is not None:
                events[k].record()
        for g in self.spec.gemms:
            qa, sa = self.operand(g.a)
            qb, sb = self.operand(g.b)
            if self.spec.nvfp4:
                mx.nvfp4_gemm(qa, sa, self.tensor_exp(g.a), qb, sb, self.tensor_exp(g.b),
                              g.M, g.N, g.K, c=out[g.label], workspace=self.ws)
            else:
                mx.mxfp4_gemm(qa, sa, qb, sb, g.M, g.N, g.K, c=out[g.label], workspace=self.ws)
            k += 1
            if events is not None:
                events[k].record()
        for name, (a, e) in self.amax.items():
            mx.tensor_amax(inp[name], amax=a, tensor_exp=e)


# ------------------------------------------------------------ utilities ---

def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return FALLBACK, "fallback"


def _dist():
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value: float, ws: int, device="cpu") -> float:
    """The largest `value` over all ranks (the job is as slow as its slowest
    replica); a no-op for one rank. `device` must suit the process group's
    backend (a CUDA device for NCCL, the CPU for gloo)."""
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(work_per_rank: float, ws: int, ms: float) -> float:
    """Whole-job throughput: the work of all replicas over the (max) step time,
    per second (weak scaling: every rank does the same work)."""
    return ws * work_per_rank / (ms / 1e3)


class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons while the block runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index: int, interval_ms: int = 100):
        self.index, self.proc, self.lines = index, None, []
        self.interval_ms = interval_ms

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, power, reasons = [], None, [], set()
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
                power.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(self.NAMES, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        # samples taken under load: power at least half of the largest seen
        loaded = [c for c, w in zip(sm, power) if power and w >= 0.5 * max(power)]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None,
                "sm_mhz_loaded": statistics.median(loaded) if loaded else None,
                "samples_loaded": len(loaded)}


def source_digest(path: str) -> str:
    """Hash of a C++/CUDA source with comments and whitespace removed, so that
    a record taken on a kernel stays valid across comment edits only."""
    import re

    with open(path) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    text = re.sub(r"\s+", "", text)
    return hashlib.sha256(text.encode()).hexdigest()[:16]


def _traffic_record():
    """DRAM traffic per GEMM launch from the committed ncu summary, if it was
    taken on the current GEMM source (else None)."""
    path = os.path.join(ROOT, "profiles", "gemm_traffic.txt")
    src = os.path.join(ROOT, "gemm_pt_block_gb300", "csrc", "gemm.cu")
    try:
        rec = {}
        with open(path) as f:
            for ln in f:
                if ":" in ln and not ln.startswith("#"):
                    k, v = ln.split(":", 1)
                    rec[k.strip()] = v.strip()
        return rec if rec.get("gemm_cu_code_sha256_16") == source_digest(src) else None
    except OSError:
        return None


# ------------------------------------------------------------ CPU oracle ---

class OracleSample:
    """The oracle on a bounded sample of the same step: for every quantize op
    an r-row band (row-wise output) and an r-column band (column-wise output),
    and for every GEMM r output rows (dequantize + fp64 product). The inputs
    are generated once, in __init__; run() is the timed part and returns its
    seconds."""

    def __init__(self, spec: Spec, r: int):
        import numpy as np

        import oracle
        import synth

        def op(p, band):
            if p is None:
                return None
            k = 0
            if p.block == oracle.BLOCK_1X16:   # the band's own per-tensor factor
                amax = float(np.abs((band.astype(np.uint32) << 16).view(np.float32)).max())
                k = math.ceil(math.log2(amax / 2688.0)) if amax > 0 else 0
            return oracle.Params(p.block, p.scale_mode, p.rounding, p.wht, p.wht_sign_mask, p.seed,
                                 p.sr_stream, p.elem_format, k)

        self.spec, self.r = spec, r
        sb = spec.scale_bytes_per_elem()
        self.jobs, self.qbytes, self.flops = [], 0.0, 0.0
        for q in spec.quants:
            rr = min(r, q.rows)
            if q.prow is not None:
                band = synth.bf16_bits(gen_input(q, "cpu", rows=rr))
                self.jobs.append(("rows", band, op(q.prow, band)))
                self.qbytes += band.size * (2 + 0.5 + sb)
            if q.pcol is not None:
                cc = min(r, q.cols)
                band = synth.bf16_bits(gen_input(q, "cpu", cols=cc, seed_offset=1))
                self.jobs.append(("cols", band, op(q.pcol, band)))
                self.qbytes += band.size * (2 + 0.5 + sb)
        self.gem = []
        for g in spec.gemms:
            m = min(r, g.M)
            if spec.nvfp4:   # random E4M3 scale codes near 1
                sa = np.random.default_rng(2).integers(40, 70, m * g.K // 16, dtype=np.uint8)
                sbb = np.random.default_rng(4).integers(40, 70, g.N * g.K // 16, dtype=np.uint8)
            else:
                sa, sbb = synth.random_scales(m, g.K, 2), synth.random_scales(g.N, g.K, 4)
            self.gem.append((synth.random_codes(m, g.K, 1), sa, synth.random_codes(g.N, g.K, 3), sbb,
                             m, g.N, g.K))
            self.flops += 2.0 * m * g.N * g.K
        self.threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
        self.desc = (f"{r}-row / {r}-column bands of every quantized tensor (oracle quantize, both "
                     f"orientations as the step asks) and {r} output rows of every GEMM (oracle "
                     f"dequantize + fp64 product); value = sampled GEMM FLOPs / oracle seconds")

    def run(self) -> float:
        import oracle

        t0 = time.perf_counter()
        for kind, band, p in self.jobs:
            (oracle.quantize_rows if kind == "rows" else oracle.quantize_cols)(band, p)
        for qa, sa, qb, sbb, m, N, K in self.gem:
            if self.spec.nvfp4:
                A = oracle.dequantize_nv(qa, sa.reshape(m, K // 16), m, K)
                B = oracle.dequantize_nv(qb, sbb.reshape(N, K // 16), N, K)
            else:
                A = oracle.dequantize(qa, sa.reshape(m, K // 32), m, K, f64=True)
                B = oracle.dequantize(qb, sbb.reshape(N, K // 32), N, K, f64=True)
            _ = A @ B.T
        return time.perf_counter() - t0


def run_oracle_sample(args):
    """--oracle-sample R: time the oracle once on an R-row sample of the
    workload in this process (its thread count from the environment) and print
    the seconds and work as JSON."""
    sample = OracleSample(make_spec(args.workload), args.oracle_sample)
    dt = sample.run()
    print(json.dumps({"seconds": dt, "flops": sample.flops, "qbytes": sample.qbytes,
                      "threads": sample.threads, "sample": sample.desc}), flush=True)
    return 0


def run_single_thread_oracle(workload: str, r: int = 512):
    """The oracle sample on one core: a child process with every thread pool
    (OpenMP, BLAS) set to one thread, on 512-row bands (about 10-20 s)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        out = subprocess.run([sys.executable, os.path.abspath(__file__), "--workload", workload,
                              "--oracle-sample", str(r)], env=env, capture_output=True, text=True,
                             timeout=180)
        d = json.loads(out.stdout.strip().splitlines()[-1])
    except (subprocess.SubprocessError, ValueError, IndexError, OSError):
        return None
    return {"value": d["flops"] / d["seconds"] / 1e12, "unit": "TFLOP/s", "cores": d["threads"],
            "seconds": d["seconds"], "quantize_gbs": d["qbytes"] / d["seconds"] / 1e9,
            "sample": d["sample"]}


def bench_config(spec: Spec, ws: int) -> dict:
    """The `config` object of the JSON line (both arms print the same one)."""
    if spec.name == TWO_D:
        l2 = "flushed (512 MB rewrite and read-back) before each launch: W is 33.5 MB"
    elif spec.name in LAYERS:
        l2 = ("no flush: every input tensor and operand of the default workload is larger "
              "than the 129 MB L2 (X 268 MB, W 470 MB, dY 940 MB bf16; codes 67-235 MB)"
              if spec.name.startswith("70b") else
              "no flush: inputs of 67-235 MB bf16 are larger than the 129 MB L2; some operands are not")
    else:
        l2 = "no flush"
    return {"workload": spec.desc,
            "parallelism": f"{ws} independent replicas" if ws > 1 else "1 GPU", "l2": l2}


def run_reference(args):
    """The reference arm: the oracle as it stands, on the host cores, on a
    bounded sample of the same workload per step (2048-row / 2048-column bands,
    2048 GEMM output rows), inputs generated once before the first step."""
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    spec = make_spec(args.workload)
    sample = OracleSample(spec, 2048)
    times = []
    for i in range(args.warmup + args.steps):
        dt = sample.run()
        if i >= args.warmup:
            times.append(dt)
    ms = 1000.0 * statistics.mean(times)
    if spec.gemms:
        value, unit = sample.flops / (ms / 1000.0) / 1e12, "TFLOP/s"
    else:                                     # quantize-only workload
        value, unit = sample.qbytes / (ms / 1000.0) / 1e9, "GB/s"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(spec, ws),
        "cpu_baseline": {"value": value, "unit": unit, "cores": sample.threads, "kind": "oracle",
                         "sample": sample.desc},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ main ---

def measure_e2e(st: Step, steps: int, ws: int):
    """The same metric through the public API with host buffers: every step
    copies its bf16 inputs from pinned host memory to the device, runs the step
    and reads its fp32 GEMM results back to pinned host memory. Steps are
    pipelined over two buffer slots as a training loop with a prefetching data
    loader runs them: the copy-in of step i + 1 (its own stream) and the
    copy-out of step i - 1 (another stream) overlap the compute of step i;
    events order every reuse of a slot. The timed region runs from before the
    first copy-in to after the last copy-out. (One stream per tensor for the
    copies measured no faster: the copy bandwidth is the limit.)"""
    import torch

    dev0 = next(iter(st.outs.values())).device
    bw_before = copy_bandwidth(dev0)
    host_in = {k: v.cpu().pin_memory() for k, v in st.inputs.items()}
    dev_in = [{k: torch.empty_like(v) for k, v in st.inputs.items()} for _ in range(2)]
    dev_out = [{k: torch.empty_like(v) for k, v in st.outs.items()} for _ in range(2)]
    host_out = [{k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in st.outs.items()}
                for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out[0].values())
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    in_ready, in_free = [ev(), ev()], [ev(), ev()]
    out_ready, out_free = [ev(), ev()], [ev(), ev()]
    used = [False, False]

    marks = []

    def one(i, mark=False):
        b = i % 2
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(in_free[b])
            for k in host_in:
                dev_in[b][k].copy_(host_in[k], non_blocking=True)
            in_ready[b].record(s_in)
        comp.wait_event(in_ready[b])
        if used[b]:
            comp.wait_event(out_free[b])
        st.run(inputs=dev_in[b], outs=dev_out[b])
        in_free[b].record(comp)
        out_ready[b].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(out_ready[b])
            for k in host_out[b]:
                host_out[b][k].copy_(dev_out[b][k], non_blocking=True)
            out_free[b].record(s_out)
            if mark:                       # end of this step's copy-out
                e = torch.cuda.Event(enable_timing=True)
                e.record(s_out)
                marks.append(e)
        used[b] = True

    # A first copy from or into freshly pinned host memory runs several times
    # slower than later ones (measured: 57 ms instead of 8 for the 1.68 GB of
    # inputs), so every host buffer is copied once each way before warm-up.
    for b in range(2):
        for k in host_in:
            dev_in[b][k].copy_(host_in[k], non_blocking=True)
        for k in host_out[b]:
            host_out[b][k].copy_(dev_out[b][k], non_blocking=True)
    torch.cuda.synchronize()
    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    for i in range(steps):
        one(i, mark=True)
    stop.record(s_out)
    torch.cuda.synchronize()
    ms = start.elapsed_time(stop) / steps
    # Per-step intervals between the ends of consecutive copy-outs (the first
    # also holds the pipeline fill). Steps far above the median are pauses of
    # the host copies on the GPU machine (seen after many pinned allocations by
    # earlier processes); `value` keeps them.
    iv = [start.elapsed_time(marks[0])] + [marks[j].elapsed_time(marks[j + 1])
                                           for j in range(len(marks) - 1)]
    med = statistics.median(iv[1:]) if len(iv) > 1 else iv[0]
    dev = next(iter(st.outs.values())).device
    ms = max_over_ranks(ms, ws, dev)
    flops = sum(st.spec.gemm_flops())
    del dev_in, dev_out, host_out, host_in
    # The copy rates, measured before and after the timed steps (best of five
    # each time): the host copies pause at times on the GPU machine, and a probe
    # caught in a pause would understate the bound.
    bw_after = copy_bandwidth(dev)
    bw = {k: max(bw_before[k], bw_after[k]) if k.endswith("_gbs") else bw_after[k] for k in bw_after}
    # Copy bound of one step: each direction at its own rate, and both together
    # at the combined rate while they overlap.
    bound = 1e3 * max(h2d / (bw["h2d_gbs"] * 1e9), d2h / (bw["d2h_gbs"] * 1e9),
                      (h2d + d2h) / (bw["both_gbs"] * 1e9))
    bw["step_bound_ms"] = bound
    return {"value": job_rate(flops, ws, ms) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "pipelined": "copy-in, compute and copy-out on three streams, two buffer slots",
            "copy_roofline": bw, "frac_of_copy_bound": bound / ms,
            "step_ms_median": med, "step_ms_max": max(iv[1:] or iv),
            "stalled_steps": sum(1 for t in iv[1:] if t > 2 * med),
            "frac_of_copy_bound_median_step": bound / med}


def copy_bandwidth(device, nbytes: int = 1 << 30, reps: int = 5) -> dict:
    """Raw pinned-host <-> device copy rates on this machine, in the same run: one
    nbytes cudaMemcpyAsync host->device, one device->host, and both at once on
    two streams (best of `reps` each, CUDA events)."""
    import torch

    h_src = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    h_dst = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d_a = torch.empty(nbytes, dtype=torch.uint8, device=device)
    d_b = torch.empty(nbytes, dtype=torch.uint8, device=device)
    s1, s2 = torch.cuda.Stream(device), torch.cuda.Stream(device)

    def best(fn):
        ms = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(s1)
            fn(e0)
            e1.record(s1)
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1))
        return min(ms)

    def h2d(_):
        with torch.cuda.stream(s1):
            d_a.copy_(h_src, non_blocking=True)

    def d2h(_):
        with torch.cuda.stream(s1):
            h_dst.copy_(d_b, non_blocking=True)

    def both(e0):
        s2.wait_event(e0)
        with torch.cuda.stream(s2):
            h_dst.copy_(d_b, non_blocking=True)
        h2d(e0)
        done = torch.cuda.Event()
        done.record(s2)
        s1.wait_event(done)

    t_in, t_out, t_both = best(h2d), best(d2h), best(both)
    del h_src, h_dst, d_a, d_b
    return {"bytes": nbytes, "h2d_gbs": nbytes / (t_in / 1e3) / 1e9,
            "d2h_gbs": nbytes / (t_out / 1e3) / 1e9,
            "both_gbs": 2 * nbytes / (t_both / 1e3) / 1e9}


def measure_graph(st, steps: int):
    """The same step captured once into a CUDA graph and replayed: launch
    overhead paid once per step instead of once per call. The library's
    per-device caches (kernel attributes, occupancy) are filled by an eager
    step first; the captured calls then enqueue only kernel launches (and, for
    NVFP4, async memsets). Outputs of the replay equal the eager step's."""
    import torch

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        st.run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    want = {k: v.clone() for k, v in st.outs.items()}
    g = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(g):
            st.run()
    except Exception as e:        # report, do not fail the benchmark
        torch.cuda.synchronize()
        return {"unavailable": (str(e).splitlines() or [repr(e)])[0][:200]}
    for o in st.outs.values():
        o.zero_()
    g.replay()
    torch.cuda.synchronize()
    same = all(torch.equal(want[k], st.outs[k]) for k in want)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(steps):
        g.replay()
    t1.record()
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    return {"value": sum(st.spec.gemm_flops()) / (ms / 1e3) / 1e12, "unit": "TFLOP/s",
            "ms_per_step": ms, "steps": steps, "outputs_equal_eager": same,
            "what": "the step captured once in a CUDA graph (torch.cuda.graph) and replayed"}


def measure_linear(spec: Spec, st: "Step", steps: int):
    """The same layer step through the autograd op (mxfp4_linear forward +
    backward on the step's X, W and dY, recipe taken from the workload), timed
    with CUDA events; includes autograd's bookkeeping. Y, dY and the gradients
    are bf16 here (the GEMMs round their fp32 sums to bf16 in the epilogue)."""
    import torch
    import gemm_pt_block_gb300 as mx

    q = {o.name: o for o in spec.quants}
    recipe = mx.LinearRecipe(q["X"].prow, q["X"].pcol, q["W"].prow, q["W"].pcol,
                             q["dY"].prow, q["dY"].pcol)
    x = st.inputs["X"].detach().requires_grad_()
    w = st.inputs["W"].detach().requires_grad_()
    g = st.inputs["dY"]

    def one():
        y = mx.mxfp4_linear(x, w, recipe, out_dtype=torch.bfloat16)
        return torch.autograd.grad(y, (x, w), g)

    for _ in range(2):
        one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        one()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return {"value": sum(spec.gemm_flops()) / (ms / 1e3) / 1e12, "unit": "TFLOP/s",
            "ms_per_step": ms, "steps": steps,
            "what": "mxfp4_linear forward + backward (autograd) on the step's tensors, "
                    "bf16 Y / dY / dX / dW"}


def run_op(args):
    """Time one operation of the step alone (its own tensors only, so a profiler
    can capture a full-size launch with a small device footprint)."""
    import torch
    import gemm_pt_block_gb300 as mx

    spec = make_spec(args.workload)
    qs = {q.name: q for q in spec.quants}
    gs = {g.label: g for g in spec.gemms}
    if args.op in qs:
        sub = Spec(spec.name, spec.desc, [qs[args.op]], [], spec.nvfp4)
    elif args.op in gs:
        g = gs[args.op]
        sub = Spec(spec.name, spec.desc, [qs[n] for n in dict.fromkeys((g.a[0], g.b[0]))], [g],
                   spec.nvfp4)
    else:
        raise SystemExit(f"--op must be one of {sorted(qs) + sorted(gs)}")
    device = torch.device("cuda", 0)
    st = Step(sub, device)
    if sub.gemms:
        st.run()   # quantize the operands once
        g = sub.gemms[0]
        qa, sa = st.operand(g.a)
        qb, sb = st.operand(g.b)
        if sub.nvfp4:
            ka, kb = st.tensor_exp(g.a), st.tensor_exp(g.b)
            fn = lambda: mx.nvfp4_gemm(qa, sa, ka, qb, sb, kb, g.M, g.N, g.K, c=st.outs[g.label],
                                       workspace=st.ws)
        else:
            fn = lambda: mx.mxfp4_gemm(qa, sa, qb, sb, g.M, g.N, g.K, c=st.outs[g.label],
                                       workspace=st.ws)
        work, unit = sub.gemm_flops()[0] / 1e12, "TFLOP/s"
    else:
        q = sub.quants[0]
        qr, sr, qc, sc = st.bufs[q.name]
        x = st.inputs[q.name]
        prow, pcol = st.params[q.name]
        fn = lambda: mx.mxfp4_quantize(x, prow, pcol, q_row=qr, s_row=sr, q_col=qc, s_col=sc)
        work, unit = sub.quant_bytes()[0] / 1e9, "GB/s"
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    if mx.device_status() != 0:
        raise RuntimeError("a bounded device-side wait ran out")
    print(json.dumps({"op": args.op, "workload": args.workload, "ms": ms,
                      "rate": work / (ms / 1e3), "unit": unit, "launches": args.steps}), flush=True)
    return 0


def measure_step_config(name: str, steps: int, device) -> dict:
    """A training-step configuration other than the headline, measured after
    it. Before each step a 512 MB buffer is rewritten and read back (cold L2:
    the tiny step would otherwise run from L2). The step time is a CUDA-graph
    replay of the whole step (no host launch gaps, which would dominate the
    tiny step); the per-launch times come from eager steps with CUDA events
    around each launch. Medians over `steps` steps after 3 warm-up steps."""
    import torch

    spec = make_spec(name)
    st = Step(spec, device)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=device)
    for _ in range(3):
        st.run()
    torch.cuda.synchronize()
    per = [[] for _ in range(st.ops)]
    for _ in range(steps):
        flush_l2(flush)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(st.ops + 1)]
        st.run(events=ev)
        torch.cuda.synchronize()
        for j in range(st.ops):
            per[j].append(ev[j].elapsed_time(ev[j + 1]))
    g = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(g):
            st.run()
        replay = g.replay
        how = "graph replay of the step (value, ms_per_step)"
    except Exception:              # time the eager step instead; say so
        torch.cuda.synchronize()
        replay = st.run
        how = "eager step (graph capture failed) for value and ms_per_step"
    replay()
    whole = []
    for _ in range(steps):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        replay()
        e1.record()
        torch.cuda.synchronize()
        whole.append(e0.elapsed_time(e1))
    import gemm_pt_block_gb300 as mx
    if mx.device_status() != 0:
        raise RuntimeError("a bounded device-side wait ran out")
    ms = [statistics.median(t) for t in per]
    nq = len(spec.quants)
    labels, qwork, gwork = spec.labels(), spec.quant_bytes(), spec.gemm_flops()
    peaks, src = _peaks()
    fp4 = peaks.get("bf16_tflops", FALLBACK["bf16_tflops"]) * FP4_OVER_BF16
    hbm = peaks.get("hbm_gbs", FALLBACK["hbm_gbs"])
    step_ms = statistics.median(whole)
    gt = sum(gwork) / (sum(ms[nq:]) / 1e3) / 1e12
    qg = sum(qwork) / (sum(ms[:nq]) / 1e3) / 1e9
    return {"workload": spec.desc, "value": sum(gwork) / (step_ms / 1e3) / 1e12, "unit": "TFLOP/s",
            "ms_per_step": step_ms, "steps": steps,
            "gemm": {"tflops": gt, "frac_of_fp4_peak": gt / fp4, "ms": dict(zip(labels[nq:], ms[nq:]))},
            "quantize": {"gbs": qg, "frac_of_hbm": qg / hbm, "ms": dict(zip(labels[:nq], ms[:nq]))},
            "timing": how + " and eager per-launch CUDA events (parts), L2 flushed before each "
                      "step; peaks as in the headline (" + src + ")"}


def measure_configs(steps: int, device) -> dict:
    """The pages' other configurations, measured briefly after the headline
    step so that one benchmark line carries all five: the tiny layer (X, W
    [512, 1024], outlier columns, Y = Xq Wq^T), the 2D-block consistency
    check (W [4096, 4096] dual 32x32 in one pass, with its checks), the
    Llama-3.1-8B-shaped MLP up-projection step, and the square sweep (the
    quantizer variants and the n^3 GEMM, n = 1024..16384), the sweep's points
    condensed to fractions of their rooflines."""
    out = {"tiny": measure_step_config("tiny", steps, device)}
    two = measure_2d(steps, 3)
    out["2d-blocks"] = {k: two[k] for k in ("value", "unit", "ms_per_step", "steps", "checks")}
    out["2d-blocks"].update(workload=two["config"]["workload"], frac_of_hbm=two["roofline"]["frac"],
                            l2=two["config"]["l2"])
    out["8b-mlp-up"] = measure_step_config("8b-mlp-up", steps, device)
    pts = []
    sweep_points(3, pts.append)
    quant, gemm = {}, {}
    for p in pts:
        if "gbs" in p:
            quant.setdefault(p["sweep"], {})[str(p["n"])] = round(p["frac_of_hbm"], 3)
        else:
            gemm[str(p["n"])] = {"tflops": round(p["tflops"], 1), "frac_of_fp4_peak": round(p["frac_of_fp4_peak"], 3)}
    out["sweep"] = {"quantize_frac_of_hbm": quant, "gemm_n3": gemm,
                    "what": "square bf16 inputs ~ t(3); per point the median of 3 launches, L2 flushed "
                            "before each; `bench.py --sweep` prints every point in full"}
    return out


def flush_l2(buf):
    """Cold-L2 start for the next launch: rewrite a buffer larger than L2, then
    read it back, so none of the next launch's inputs are in L2 and the
    rewrite's dirty lines are written back here rather than inside the next
    launch's timed region."""
    import torch

    buf.fill_(1)
    buf.view(torch.int32).max()


def run_2d(args):
    """`--workload 2d-blocks`: prints measure_2d's line; fails if the 32x32
    blocks are not transposition-invariant."""
    line = measure_2d(args.steps, args.warmup)
    print(json.dumps(line), flush=True)
    c = line["checks"]
    if not (c["codes_transposition_invariant"] and c["scales_transposition_invariant"]
            and c["scale_mismatch_fraction_32x32"] == 0.0):
        raise RuntimeError("32x32 blocks are not transposition-invariant")
    return 0


def measure_2d(steps: int, warmup: int) -> dict:
    """The 2D-block consistency workload: W [4096, 4096] ~ N(0, 0.02) quantized
    in 32x32 blocks (round-up scales, nearest-even) in both orientations in one
    pass, timed with L2 flushed before each launch (W is 33.5 MB, smaller than
    L2); then checked in the same run: the column-wise codes and scales are
    exactly the transposes of the row-wise ones, and the same tensor in 1x32
    blocks gives the fraction of elements whose row-wise and column-wise scales
    differ (zero for 32x32 blocks). Scales are written in the tensor-core
    layout the GEMM consumes and read back into row-major order for the
    checks."""
    import torch
    import gemm_pt_block_gb300 as mx

    spec = make_spec(TWO_D)
    q = spec.quants[0]
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    x = gen_input(q, device)
    out = mx.mxfp4_quantize(x, q.prow, q.pcol)
    kw = dict(q_row=out[0], s_row=out[1], q_col=out[2], s_col=out[3])
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=device)
    for _ in range(max(warmup, 3)):
        mx.mxfp4_quantize(x, q.prow, q.pcol, **kw)
    times = []
    with ClockSampler(0) as clk:
        for _ in range(steps):
            flush_l2(flush)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            mx.mxfp4_quantize(x, q.prow, q.pcol, **kw)
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
    if mx.device_status() != 0:
        raise RuntimeError("a bounded device-side wait ran out")
    ms = statistics.median(times)
    gbs = spec.quant_bytes()[0] / (ms / 1e3) / 1e9
    peaks, src = _peaks()
    hbm = peaks.get("hbm_gbs", FALLBACK["hbm_gbs"])

    def codes(t):
        return torch.stack([t & 15, t >> 4], dim=-1).reshape(t.shape[0], -1)

    def rowmajor(s, rows):                  # tensor-core layout -> [rows, K/32]
        nkb = s.numel() // rows
        r = torch.arange(rows, device=s.device).view(-1, 1)
        kb = torch.arange(nkb, device=s.device).view(1, -1)
        off = (((r // 128) * (nkb // 4) + kb // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4
               + kb % 4)
        return s.reshape(-1)[off]

    def scale_map(s, k):                    # per-element scale, [rows, k]
        return rowmajor(s, s.numel() * 32 // k).repeat_interleave(32, dim=1)

    same_codes = torch.equal(codes(out[0]), codes(out[2]).T)
    srow, scol = scale_map(out[1], q.cols), scale_map(out[3], q.rows)
    same_scales = torch.equal(srow, scol.T)
    p1 = replace(q.prow, block=mx.BLOCK_1X32)
    o1 = mx.mxfp4_quantize(x, p1, p1)
    mism_1x32 = (scale_map(o1[1], q.cols) != scale_map(o1[3], q.rows).T).double().mean().item()
    mism_32x32 = (srow != scol.T).double().mean().item()
    line = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": steps,
        "warmup": max(warmup, 3), "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e2m1", "data": "synthetic",
        "config": bench_config(spec, 1),
        "roofline": {"bound": "hbm", "kernel": "quant_tile_kernel (weights profile)", "achieved": gbs,
                     "peak": hbm, "unit": "GB/s", "frac": gbs / hbm, "traffic": None,
                     "peak_source": src, "bytes_model": "bf16 read + 2 x (0.5 B codes + 1/32 B scales)"},
        "checks": {"codes_transposition_invariant": same_codes,
                   "scales_transposition_invariant": same_scales,
                   "scale_mismatch_fraction_32x32": mism_32x32,
                   "scale_mismatch_fraction_1x32": mism_1x32},
        "gpu_launches": steps, "clocks": clk.summary(),
    }
    return line


def run_ceiling(args):
    """Context for the GEMM's roofline: the three 70B-layer GEMM shapes, timed
    alone with CUDA events as a short burst (20 launches) and a sustained run
    (1500 launches, ~2 s) with the SM clock, power and power-cap flag sampled
    every 50 ms; and cuBLAS's block-scaled FP4 GEMM (torch._scaled_mm with
    NVFP4 operands: E2M1, E4M3 scales per 16, bf16 out; MXFP4 where this torch
    supports it) on the same shapes, as a measured achievable rate. One JSON
    line per measurement."""
    import torch
    import gemm_pt_block_gb300 as mx

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)

    def clocked(fn, n):
        torch.cuda.synchronize()
        with ClockSampler(0, interval_ms=50) as clk:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(n):
                fn()
            e1.record()
            torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n, clk.summary()

    spec = make_spec("70b-layer")
    st = Step(spec, dev)
    st.run()
    torch.cuda.synchronize()
    for g in spec.gemms:
        qa, sa = st.operand(g.a)
        qb, sb = st.operand(g.b)
        fn = lambda: mx.mxfp4_gemm(qa, sa, qb, sb, g.M, g.N, g.K, c=st.outs[g.label], workspace=st.ws)
        for n in (20, 1500):
            ms, clk = clocked(fn, n)
            print(json.dumps({"ceiling": "mxfp4_gemm (this library, fp32 C)", "gemm": g.label,
                              "M": g.M, "N": g.N, "K": g.K, "launches": n, "ms": ms,
                              "tflops": 2.0 * g.M * g.N * g.K / (ms / 1e3) / 1e12, "clocks": clk}),
                  flush=True)
    del st
    torch.cuda.empty_cache()
    fp4 = getattr(torch, "float4_e2m1fn_x2", None)
    for g in spec.gemms:
        M, N, K = g.M, g.N, g.K
        for kind in ("nvfp4", "mxfp4"):
            try:
                if fp4 is None:
                    raise RuntimeError("this torch has no float4_e2m1fn_x2")
                a = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, device=dev).view(fp4)
                b = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device=dev).view(fp4)
                if kind == "nvfp4":
                    s_a = (torch.rand(M * K // 16, device=dev) + 0.5).to(torch.float8_e4m3fn)
                    s_b = (torch.rand(N * K // 16, device=dev) + 0.5).to(torch.float8_e4m3fn)
                else:
                    s_a = torch.randint(120, 134, (M * K // 32,), dtype=torch.uint8,
                                        device=dev).view(torch.float8_e8m0fnu)
                    s_b = torch.randint(120, 134, (N * K // 32,), dtype=torch.uint8,
                                        device=dev).view(torch.float8_e8m0fnu)
                fn = lambda: torch._scaled_mm(a, b.t(), s_a, s_b, out_dtype=torch.bfloat16)
                fn()
                for n in (20, 1500):
                    ms, clk = clocked(fn, n)
                    print(json.dumps({"ceiling": f"cuBLAS {kind} (torch._scaled_mm, bf16 C)",
                                      "gemm": g.label, "M": M, "N": N, "K": K, "launches": n,
                                      "ms": ms, "tflops": 2.0 * M * N * K / (ms / 1e3) / 1e12,
                                      "clocks": clk}), flush=True)
                del a, b, s_a, s_b
            except Exception as e:   # the torch build may not offer this scaling
                print(json.dumps({"ceiling": f"cuBLAS {kind} (torch._scaled_mm)", "gemm": g.label,
                                  "unavailable": repr(e).splitlines()[0][:200]}), flush=True)
    return 0


def run_sweep(args):
    """`--sweep`: one JSON line per point of sweep_points."""
    sweep_points(max(args.steps, 3), lambda d: print(json.dumps(d), flush=True))
    return 0


def sweep_points(steps: int, emit) -> None:
    """Quantizer throughput over the square sweep (algorithmic bytes / time,
    against the measured HBM copy peak), then the n^3 GEMM at each n; `emit`
    receives one dict per point. Between timed launches a 512 MB buffer is
    rewritten and read back (flush_l2) so every launch starts with a cold
    L2."""
    import torch
    import gemm_pt_block_gb300 as mx
    import synth

    P = mx.QuantParams
    peaks, src = _peaks()
    hbm = peaks.get("hbm_gbs", FALLBACK["hbm_gbs"])
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    for n in sorted(SQUARES.values()):
        x = synth.dev_student_t(n, n, 3.0, 1004, "cuda")
        mask = synth.sign_mask(1004)
        variants = []
        for rnd, rname in ((mx.ROUND_RTN, "rtn"), (mx.ROUND_SR, "sr")):
            for blk, sm, bname in ((mx.BLOCK_1X32, mx.SCALE_FLOOR, "1x32-floor"),
                                   (mx.BLOCK_32X32, mx.SCALE_ROUNDUP, "32x32-roundup")):
                for wht, wname in ((False, "norot"), (True, "rot")):
                    p = P(blk, sm, rnd, mx.LAYOUT_MMA, wht, mask if wht else 0, 1005, 0)
                    variants.append((f"row {rname} {bname} {wname}", p, None))
        for blk, sm, bname in ((mx.BLOCK_1X32, mx.SCALE_FLOOR, "1x32-floor"),
                               (mx.BLOCK_32X32, mx.SCALE_ROUNDUP, "32x32-roundup")):
            p = P(blk, sm, mx.ROUND_RTN, mx.LAYOUT_MMA)
            variants.append((f"dual rtn {bname} norot", p, p))
        for name, prow, pcol in variants:
            out = mx.mxfp4_quantize(x, prow, pcol)
            kw = dict(q_row=out[0], s_row=out[1], q_col=out[2], s_col=out[3])
            for _ in range(2):
                mx.mxfp4_quantize(x, prow, pcol, **kw)
            times = []
            for _ in range(steps):
                flush_l2(flush)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                mx.mxfp4_quantize(x, prow, pcol, **kw)
                e1.record()
                torch.cuda.synchronize()
                times.append(e0.elapsed_time(e1))
            ms = statistics.median(times)
            byts = n * n * (2 + ((prow is not None) + (pcol is not None)) * (0.5 + 1 / 32))
            gbs = byts / (ms / 1e3) / 1e9
            emit({"sweep": name, "n": n, "ms": ms, "gbs": gbs, "frac_of_hbm": gbs / hbm,
                  "hbm_peak_source": src, "l2": "flushed (512 MB rewrite and read-back) before each launch"})
            del out, kw
        # the n^3 GEMM on 1x32 floor nearest-even operands (A, B ~ t(3))
        pg = P(mx.BLOCK_1X32, mx.SCALE_FLOOR, mx.ROUND_RTN, mx.LAYOUT_MMA)
        b = synth.dev_student_t(n, n, 3.0, 1104, "cuda")
        qa, sa, _, _ = mx.mxfp4_quantize(x, pg)
        qb, sb, _, _ = mx.mxfp4_quantize(b, pg)
        del b
        c = torch.empty(n, n, device="cuda")
        ws = torch.empty(mx.gemm_workspace_size(n, n, n), dtype=torch.uint8, device="cuda")
        for _ in range(2):
            mx.mxfp4_gemm(qa, sa, qb, sb, n, n, n, c=c, workspace=ws)
        times = []
        for _ in range(steps):
            flush_l2(flush)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            mx.mxfp4_gemm(qa, sa, qb, sb, n, n, n, c=c, workspace=ws)
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        ms = statistics.median(times)
        tflops = 2.0 * n ** 3 / (ms / 1e3) / 1e12
        fp4 = peaks.get("bf16_tflops", FALLBACK["bf16_tflops"]) * FP4_OVER_BF16
        emit({"sweep": "gemm n^3 (1x32 floor nearest-even operands, scale images)", "n": n,
              "ms": ms, "tflops": tflops, "frac_of_fp4_peak": tflops / fp4,
              "fp4_peak_source": f"derived: {src} bf16_tflops x {FP4_OVER_BF16:g}",
              "l2": "flushed (512 MB rewrite and read-back) before each launch"})
        del qa, sa, qb, sb, c, ws, x
    if mx.device_status() != 0:
        raise RuntimeError("a bounded device-side wait ran out")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="70b-layer", choices=WORKLOADS)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other configurations (tiny, 2d-blocks, 8b-mlp-up, sweep) that the "
                         "default run measures after the headline step")
    ap.add_argument("--sweep", action="store_true",
                    help="quantizer sweep on square bf16 inputs n = 1024..16384: eight row-wise "
                         "variants ({RTN, SR} x {1x32 floor, 32x32 round-up} x {no rotation, "
                         "random-sign rotation}) and both dual-orientation block types; one JSON "
                         "line per point (L2 flushed between launches)")
    ap.add_argument("--oracle-sample", type=int, default=None, help=argparse.SUPPRESS)
    ap.add_argument("--ceiling", action="store_true",
                    help="time the 70B GEMM shapes alone (burst and sustained, with clocks) and "
                         "cuBLAS's block-scaled FP4 GEMM on the same shapes; one JSON line each")
    ap.add_argument("--op", default=None,
                    help="profiling aid: allocate and time only this operation of the workload's "
                         "step (a quantizer name such as dY, or a GEMM label such as Fprop); prints "
                         "a short JSON line instead of the benchmark line")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.oracle_sample:
        return run_oracle_sample(args)
    if args.workload == TWO_D:
        return run_2d(args)
    if args.op:
        return run_op(args)
    if args.sweep:
        return run_sweep(args)
    if args.ceiling:
        return run_ceiling(args)

    import torch

    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)

    import gemm_pt_block_gb300 as mx
    from gemm_pt_block_gb300 import build as mxbuild

    if not os.path.exists(mx.lib_path()):
        mxbuild.build()
    mx.lib()

    spec = make_spec(args.workload)
    st = Step(spec, device)
    qwork, gwork = spec.quant_bytes(), spec.gemm_flops()
    nq = len(qwork)
    torch.cuda.synchronize()

    def barrier():
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        st.run()
    barrier()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(st.ops + 1)]
           for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        barrier()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for i in range(args.steps):
            st.run(events=evs[i])
        t1.record()
        barrier()
    total_ms = max_over_ranks(t0.elapsed_time(t1), ws, device)
    ms_step = total_ms / args.steps
    per_launch = [statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(args.steps))
                  for j in range(st.ops)]
    if mx.device_status() != 0:
        raise RuntimeError("a bounded device-side wait ran out during the benchmark")

    peaks, peak_src = _peaks()
    # The GEMMs run inside a step of a few ms, not a seconds-long loop: the
    # burst bf16 rate is the denominator, times the nominal FP4 : BF16 ratio.
    fp4_peak = peaks.get("bf16_tflops", FALLBACK["bf16_tflops"]) * FP4_OVER_BF16
    hbm_peak = peaks.get("hbm_gbs", FALLBACK["hbm_gbs"])
    q_ms, g_ms = per_launch[:nq], per_launch[nq:]
    labels = spec.labels()
    gemm_tflops = sum(gwork) / (sum(g_ms) / 1e3) / 1e12
    quant_gbs = sum(qwork) / (sum(q_ms) / 1e3) / 1e9
    value = job_rate(sum(gwork), ws, ms_step) / 1e12

    # Dominant kernel by share of the step: the GEMM (per-launch average).
    achieved = statistics.mean(f / (m / 1e3) / 1e12 for f, m in zip(gwork, g_ms))
    tr = _traffic_record()
    traffic = None
    if tr is not None and tr.get("workload") == args.workload:
        traffic = float(tr["dram_bytes_per_launch"])
    clocks = clk.summary()
    roofline = {"bound": "tensor", "kernel": "mxf4_gemm_pair_kernel" + ("<NVFP4>" if spec.nvfp4 else ""),
                "achieved": achieved,
                "peak": fp4_peak, "unit": "TFLOP/s", "frac": achieved / fp4_peak, "traffic": traffic,
                "peak_source": f"derived: {peak_src} bf16_tflops (burst) x {FP4_OVER_BF16:g}, the nominal "
                               f"dense FP4:BF16 ratio; no FP4 rate is measured directly",
                "traffic_source": ("ncu record profiles/gemm_traffic.txt (dram__bytes_read.sum + "
                                   "dram__bytes_write.sum, mean per GEMM launch of this workload), "
                                   "taken on this gemm.cu source") if traffic is not None else None,
                "nominal": {"peak": NOMINAL_FP4_TFLOPS, "frac": achieved / NOMINAL_FP4_TFLOPS,
                            "sm_mhz_median": clocks.get("sm_mhz"),
                            "gemm_mcycles_per_launch": (statistics.mean(g_ms) * clocks["sm_mhz"] / 1e3
                                                        if clocks.get("sm_mhz") else None),
                            "note": "NVIDIA's dense FP4 figure for one GB300 (context); the SM clock "
                                    "median over the timed region and GEMM time x clock in Mcycles"}}
    share = {lab: m / ms_step for lab, m in zip(labels, per_launch)}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e2m1", "data": "synthetic",
        "config": bench_config(spec, ws),
        "parts": {
            "gemm": {"tflops": gemm_tflops, "frac_of_fp4_peak": gemm_tflops / fp4_peak,
                     "ms": dict(zip(labels[nq:], g_ms))},
            "quantize": {"gbs": quant_gbs, "frac_of_hbm": quant_gbs / hbm_peak,
                         "ms": dict(zip(labels[:nq], q_ms)),
                         "gbs_each": {lab: b / (m / 1e3) / 1e9 for lab, b, m in zip(labels[:nq], qwork, q_ms)},
                         "bytes_model": "bf16 read + per orientation 0.5 B codes + "
                                        + ("1/16" if spec.nvfp4 else "1/32") + " B scales per element"},
            "share_of_step": share,
            "peaks": {"fp4_tflops": fp4_peak, "hbm_gbs": hbm_peak, "source": peak_src,
                      "fp4_note": "bf16 burst x 6 (derived)"},
        },
        "roofline": roofline,
        "gpu_launches": st.launches * args.steps,
        "clocks": clocks,
    }
    line["graph"] = measure_graph(st, max(3, args.steps))
    if not args.no_e2e:
        # at least 20 pipelined steps (at most 40), so the pipeline's fill
        # (the first step's copy-in, compute and copy-out, not overlapped)
        # weighs little in the mean; the count is reported in the object
        line["e2e"] = measure_e2e(st, min(max(args.steps, 20), 40), ws)
    if len(spec.gemms) == 3 and not spec.nvfp4 and not args.no_e2e:
        line["autograd_linear"] = measure_linear(spec, st, max(1, min(args.steps, 5)))
    if ws == 1 and args.workload == "70b-layer" and not args.no_configs:
        del st
        torch.cuda.empty_cache()
        try:
            line["other_configs"] = measure_configs(max(3, min(args.steps, 10)), device)
        except Exception as e:     # the headline line still prints; the failure is in it
            torch.cuda.synchronize()
            line["other_configs"] = {"unavailable": (str(e).splitlines() or [repr(e)])[0][:300]}
    if not args.no_cpu_baseline and rank == 0 and ws == 1:
        sample = OracleSample(spec, 4096)
        dt = sample.run()
        line["cpu_baseline"] = {"value": sample.flops / dt / 1e12, "unit": "TFLOP/s",
                                "cores": sample.threads, "kind": "oracle", "sample": sample.desc,
                                "seconds": dt, "quantize_gbs": sample.qbytes / dt / 1e9}
        # the same sample on one core, as the CPU-baseline plan asks
        one = run_single_thread_oracle(args.workload)
        if one is not None:
            line["cpu_baseline"]["single_thread"] = one
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

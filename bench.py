"""Benchmark of the fused weight-gradient GEMM + AdamW step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload mlp_down|attn_proj|linear|moe|fp8]

One step is one pass of the whole fused path over one batch of synthetic
input: dW = X^T dY with the AdamW update of W, m, v in the GEMM's epilogue.
The default workload is the Llama-style MLP down-projection (K = 8192
tokens, d_in = 14336, d_out = 4096, bf16 X / dY, fp32 W / m / v, AdamW
step t = 4 onward).  ``value`` is TFLOP/s = 2 M N K / (device time per step),
with inputs resident in HBM; ``e2e`` is the same metric through the C ABI
with pinned host buffers: every step copies its X and dY in and its updated
W out inside the timed region, the upload of the next step and the read-back
of the previous one overlapping the current step (``sequential_value``: the
same with each step alone).

Multi-GPU: the path is replicated (each rank runs its own full workload, no
collective on the data path); value sums over ranks and the time is the max
over ranks.  ``--impl reference`` times the fp64 CPU oracle on the host cores
on a bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as wl  # noqa: E402

METRIC = "fused wgrad+AdamW TFLOP/s and % of roofline; grad_W HBM bytes (must be 0)"
UNIT = "TFLOP/s"
L2_FLUSH_BYTES = 512 << 20
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except OSError:
        return dict(PEAKS_FALLBACK), "fallback"


# The sources the fused kernel and its launch are built from.
FUSED_SOURCES = ("forge_api.cu", "forge_kernel.cuh", "forge_launch.cuh", "forge_ptx.cuh",
                 "kernels_bf16.cu", "kernels_e4m3.cu", "kernels_pair_bf16.cu",
                 "kernels_pair_e4m3.cu")


def csrc_digest():
    """sha256 over the fused kernel's sources (file name + content, sorted)."""
    import hashlib
    d = os.path.join(ROOT, "weight_grad_gemm_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(FUSED_SOURCES):
        h.update(f.encode())
        with open(os.path.join(d, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def profile_summary():
    """Per-launch DRAM traffic of the fused kernel from the committed ncu
    summary, or None when the kernel sources changed since that capture."""
    p = os.path.join(ROOT, "profiles", "fused_adamw_mlp_down.json")
    try:
        with open(p) as f:
            doc = json.load(f)
    except OSError:
        return None
    return doc if doc.get("csrc_sha256") == csrc_digest() else None


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ["clocks.sm", "clocks.max.sm", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == len(self.FIELDS):
                self.samples.append(parts)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm = [float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        reasons = sorted({self.NAMES[i] for s in self.samples for i in range(4)
                          if s[2 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.samples)}


# ---------------------------------------------------------------- workloads

class Dense:
    """One fused wgrad+AdamW call per step on a [K, N] x [K, M] problem."""

    def __init__(self, wk: wl.Workload, dev, state_dtype=torch.float32):
        self.wk = wk
        self.dev = dev
        K, N, M = wk.K, wk.N, wk.M
        self.X = wl.activations(K, N, wl.seed_of(wk.name, "X"), device=dev)
        self.D = wl.activations(K, M, wl.seed_of(wk.name, "dY"), device=dev)
        self.W = wl.randn((N, M), wl.seed_of(wk.name, "W"), device=dev, std=0.02)
        self.m = torch.zeros((N, M), dtype=state_dtype, device=dev)
        self.v = torch.zeros((N, M), dtype=state_dtype, device=dev)
        self.hp = wk.adam.f32()
        # the state is warmed by the steps before the timed one (t = first_step)
        self.t = 1
        while self.t < wk.first_step:
            self.step()
        self.flops = wk.flops
        self.params = N * M
        es = 4 if state_dtype == torch.float32 else 2
        # algorithmic bytes: X and dY read once, W read+write, m and v read+write
        self.bytes = (K * N + K * M) * 2 + N * M * (8 + 4 * es)
        # the fused kernel, plus a staging copy per operand whose rows are not
        # a multiple of 16 bytes
        self.launches = 1 + int((2 * N) % 16 != 0) + int((2 * M) % 16 != 0)

    peak_key = "bf16"
    opt = "AdamW"

    def step(self, X=None, D=None, stream=None):
        import weight_grad_gemm_gb300 as fg
        hp = self.hp
        fg.forge_wgrad_adamw(self.X if X is None else X, self.D if D is None else D, self.W,
                             self.m, self.v, lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2, eps=hp.eps,
                             wd=hp.wd, step=self.t, stream=stream)
        self.t += 1

    def inputs(self):
        return [self.X, self.D]

    def step_with(self, ins, stream=None):
        self.step(ins[0], ins[1], stream=stream)

    def result(self):
        return self.W


class Backward(Dense):
    """The MLP down-projection's whole backward-and-update step through
    forge_backward_adamw: dX = dY Wb^T from the forward's bf16 weight copy,
    then the fused dW + AdamW, ordered on one stream."""

    def __init__(self, dev, state_dtype=torch.float32):
        super().__init__(wl.MLP_DOWN, dev, state_dtype)
        wk = self.wk
        K, N, M = wk.K, wk.N, wk.M
        self.Wb = self.W.to(torch.bfloat16)
        self.dX = torch.empty((K, N), dtype=torch.bfloat16, device=dev)
        self.flops = 2 * wk.flops
        # the input gradient reads dY and Wb and writes dX
        self.bytes += 2 * (K * M + N * M + K * N)
        self.launches = 2
        self.wk = wl.Workload(f"backward K={K} d_in={N} d_out={M} (dX = dY W^T, then fused "
                              "dW + AdamW)", K=K, N=N, M=M)

    def step(self, X=None, D=None, stream=None):
        import weight_grad_gemm_gb300 as fg
        if not hasattr(self, "Wb"):  # the warm-up steps of the constructor
            return Dense.step(self, X, D, stream)
        hp = self.hp
        fg.forge_backward_adamw(self.X if X is None else X, self.D if D is None else D, self.W,
                                self.m, self.v, self.dX, Wb=self.Wb, lr=hp.lr, beta1=hp.beta1,
                                beta2=hp.beta2, eps=hp.eps, wd=hp.wd, step=self.t, stream=stream)
        self.t += 1

    def parts_us(self, stream, flush, reps=5):
        """Median device time of the input gradient and of the fused call."""
        import weight_grad_gemm_gb300 as fg
        a, b = [], []
        for _ in range(reps):
            flush.zero_()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            ev[0].record(stream)
            fg.forge_dgrad(self.D, self.Wb, self.dX, stream=stream)
            ev[1].record(stream)
            Dense.step(self, stream=stream)
            ev[2].record(stream)
            ev[2].synchronize()
            a.append(ev[0].elapsed_time(ev[1]) * 1e3)
            b.append(ev[1].elapsed_time(ev[2]) * 1e3)
        return float(np.median(a)), float(np.median(b))


class AttnSet:
    """The four attention projections of one layer (d_in 4096, d_out 4096,
    1024, 1024, 4100; K = 16384), one AdamW step each per step, all reading
    the same X: one multi-problem call, whose single launch walks the four
    problems' tiles (a d_out = 1024 projection alone fills only 64 of the 76
    CTA pairs).  d_out = 4100 has 8200-byte dY rows, which the library stages
    into 16-byte rows first."""

    peak_key = "bf16"
    opt = "AdamW"

    def __init__(self, dev, state_dtype=torch.float32):
        self.parts = [Dense(wk, dev, state_dtype) for wk in wl.ATTN_PROJ]
        shared = self.parts[0].X
        for p in self.parts[1:]:
            p.X = shared  # one activation tensor feeds all four projections
        self.wk = wl.Workload("attn_proj K=16384 d_in=4096 d_out={4096,1024,1024,4100}",
                              K=16384, N=4096, M=sum(wl.ATTN_OUTS))
        self.flops = sum(p.flops for p in self.parts)
        self.params = sum(p.params for p in self.parts)
        self.bytes = sum(p.bytes for p in self.parts)
        # the fused launch and the staging copy of the 4100-wide dY
        self.launches = 1 + sum(p.launches - 1 for p in self.parts)
        self.t = self.parts[0].t

    def _call(self, X, Ds, stream):
        import weight_grad_gemm_gb300 as fg
        ps = self.parts
        hp = ps[0].hp  # the four projections share their hyperparameters
        fg.forge_wgrad_adamw_multi(X, Ds, [p.W for p in ps], [p.m for p in ps],
                                   [p.v for p in ps], lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2,
                                   eps=hp.eps, wd=hp.wd, step=self.t, stream=stream)
        self.t += 1

    def step(self, stream=None):
        self._call(self.parts[0].X, [p.D for p in self.parts], stream)

    def inputs(self):
        return [self.parts[0].X] + [p.D for p in self.parts]

    def step_with(self, ins, stream=None):
        self._call(ins[0], list(ins[1:]), stream)

    def result(self):
        return self.parts[0].W


class MoE:
    """Grouped call over 8 experts [14336, 4096]; the step cycles through the
    six seeded top-2 Zipf(1.2) routings (four empty experts on even steps).
    `wk` = MOE_SMALL: the same layer shapes with two experts of 4096 routed
    rows each (top-2 over two experts), about 3 GB on the device, the case a
    full ncu capture of the grouped kernel runs on; MOE_DECAY: two experts
    without tokens, the decay-only epilogue alone (2.8 GB of state read and
    written, bound by HBM)."""

    peak_key = "bf16"
    opt = "AdamW"

    def __init__(self, dev, state_dtype=torch.float32, wk=None):
        wk = wl.MOE if wk is None else wk
        small = wk is not wl.MOE
        self.wk = wk
        E, N, M = wk.experts, wk.N, wk.M
        offs = []
        for t in range(1, wk.steps + 1):
            zero = (wl.moe_zero_experts(wl.seed_of(wk.name, "zero", t), E)
                    if t % 2 == 0 and not small else ())
            c = wl.zipf_top2_counts(wl.seed_of(wk.name, "route", t), tokens=wk.K // 2,
                                    experts=E, zero_experts=zero)
            offs.append(torch.from_numpy(wl.offsets_from_counts(c).astype(np.int32)).to(dev))
        self.offs = offs
        T = int(offs[0][-1])
        self.X = wl.activations(T, N, wl.seed_of(wk.name, "X"), device=dev)
        self.D = wl.activations(T, M, wl.seed_of(wk.name, "dY"), device=dev)
        self.W = wl.randn((E, N, M), wl.seed_of(wk.name, "W"), device=dev, std=0.02)
        self.m = wl.randn((E, N, M), wl.seed_of(wk.name, "m"), device=dev, std=1e-3).to(state_dtype)
        self.v = (wl.randn((E, N, M), wl.seed_of(wk.name, "v"), device=dev, std=1e-3) ** 2).to(
            state_dtype)
        self.hp = wk.adam.f32()
        self.t = 1
        self.flops = 2.0 * N * M * T
        self.params = E * N * M
        es = 4 if state_dtype == torch.float32 else 2
        self.bytes = 2 * (T * N + T * M) + E * N * M * (8 + 4 * es)
        self.launches = 1

    def step(self, stream=None, X=None, D=None):
        import weight_grad_gemm_gb300 as fg
        hp = self.hp
        off = self.offs[(self.t - 1) % len(self.offs)]
        fg.forge_grouped_wgrad_adamw(self.X if X is None else X, self.D if D is None else D,
                                     self.W, self.m, self.v, off, lr=hp.lr, beta1=hp.beta1,
                                     beta2=hp.beta2, eps=hp.eps, wd=hp.wd, step=self.t,
                                     stream=stream)
        self.t += 1

    def inputs(self):
        return [self.X, self.D]

    def step_with(self, ins, stream=None):
        self.step(stream=stream, X=ins[0], D=ins[1])

    def result(self):
        return self.W


class Fp8:
    """X, dY [32768, 8192] e4m3 with per-tensor scales; AdamW or SGD momentum."""

    peak_key = "fp8"

    def __init__(self, dev, state_dtype=torch.float32, opt="AdamW"):
        wk = wl.FP8
        self.wk = wk
        K, N, M = wk.K, wk.N, wk.M
        self.X, sx = wl.quantize_e4m3(wl.with_outliers((K, N), wl.seed_of(wk.name, "X"), dev))
        self.D, sy = wl.quantize_e4m3(wl.with_outliers((K, M), wl.seed_of(wk.name, "dY"), dev))
        self.scales = torch.tensor([sx, sy], dtype=torch.float32, device=dev)
        self.W = wl.randn((N, M), wl.seed_of(wk.name, "W"), device=dev, std=0.02)
        self.m = wl.randn((N, M), wl.seed_of(wk.name, "m"), device=dev, std=1e-3).to(state_dtype)
        self.v = (wl.randn((N, M), wl.seed_of(wk.name, "v"), device=dev, std=1e-3) ** 2).to(
            state_dtype)
        self.opt = opt
        self.hp = wk.adam.f32() if opt == "AdamW" else wl.FP8_SGD.f32()
        self.t = 1
        self.flops = wk.flops
        self.params = N * M
        es = 4 if state_dtype == torch.float32 else 2
        nst = 2 if opt == "AdamW" else 1
        self.bytes = (K * N + K * M) + N * M * (8 + 2 * nst * es)
        self.launches = 1

    def step(self, stream=None, X=None, D=None):
        import weight_grad_gemm_gb300 as fg
        hp = self.hp
        X = self.X if X is None else X
        D = self.D if D is None else D
        if self.opt == "AdamW":
            fg.forge_wgrad_adamw(X, D, self.W, self.m, self.v, lr=hp.lr, beta1=hp.beta1,
                                 beta2=hp.beta2, eps=hp.eps, wd=hp.wd, step=self.t,
                                 scales=self.scales, stream=stream)
        else:
            fg.forge_wgrad_sgdm(X, D, self.W, self.m, lr=hp.lr, momentum=hp.momentum, wd=hp.wd,
                                scales=self.scales, stream=stream)
        self.t += 1

    def inputs(self):
        return [self.X, self.D]

    def step_with(self, ins, stream=None):
        self.step(stream=stream, X=ins[0], D=ins[1])

    def result(self):
        return self.W


class Fp8Quant(Fp8):
    """The fp8 path from fp32 activations: every step quantises X and dY
    [32768, 8192] with the library (amax pass + e4m3 codes, two launches
    each), then runs the fused e4m3 AdamW call on the codes and scales."""

    def __init__(self, dev, state_dtype=torch.float32):
        super().__init__(dev, state_dtype, "AdamW")
        wk = self.wk
        K, N, M = wk.K, wk.N, wk.M
        self.xf = wl.with_outliers((K, N), wl.seed_of(wk.name, "X"), dev)
        self.yf = wl.with_outliers((K, M), wl.seed_of(wk.name, "dY"), dev)
        self.X = torch.empty((K, N), dtype=torch.float8_e4m3fn, device=dev)
        self.D = torch.empty((K, M), dtype=torch.float8_e4m3fn, device=dev)
        # two passes over each fp32 input (amax, then codes) and the codes written
        self.quant_bytes = 9 * (K * N + K * M)
        self.bytes += self.quant_bytes
        self.launches = 5
        self.wk = wl.Workload(f"fp8_quant K={K} d_in={N} d_out={M} (fp32 X, dY quantised to "
                              "e4m3 each step)", K=K, N=N, M=M)

    def quantize(self, xf, yf, stream=None):
        import weight_grad_gemm_gb300 as fg
        fg.forge_quantize_e4m3(xf, self.X, self.scales[0:1], stream=stream)
        fg.forge_quantize_e4m3(yf, self.D, self.scales[1:2], stream=stream)

    def step(self, stream=None, X=None, D=None):
        self.quantize(self.xf if X is None else X, self.yf if D is None else D, stream)
        super().step(stream=stream)

    def inputs(self):
        return [self.xf, self.yf]

    def parts_us(self, stream, flush, reps=5):
        """Median device time of the quantisation and of the fused call."""
        q, f = [], []
        for _ in range(reps):
            flush.zero_()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            ev[0].record(stream)
            self.quantize(self.xf, self.yf, stream)
            ev[1].record(stream)
            Fp8.step(self, stream=stream)
            ev[2].record(stream)
            ev[2].synchronize()
            q.append(ev[0].elapsed_time(ev[1]) * 1e3)
            f.append(ev[1].elapsed_time(ev[2]) * 1e3)
        return float(np.median(q)), float(np.median(f))


class OwnerStep(Dense):
    """The data-parallel path with sharded optimizer state on the MLP
    down-projection shapes: each step writes this rank's partial dW (fp32) with
    forge_wgrad_only, sums the ranks' partials with a reduce-scatter (NCCL,
    only when several ranks run; one rank owns every row), and applies the
    owner's AdamW to its rows with forge_owner_adamw.  The gradient makes a
    round trip through HBM here by construction (the collective needs it)."""

    def __init__(self, dev, state_dtype=torch.float32):
        super().__init__(wl.MLP_DOWN, dev, state_dtype)
        from weight_grad_gemm_gb300 import owner
        wk = self.wk
        K, N, M = wk.K, wk.N, wk.M
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.ranges = owner.owner_ranges(N, self.world)
        r0, r1 = self.ranges[self.rank]
        self.shard = (r0, r1)
        self.G = torch.empty((N, M), dtype=torch.float32, device=dev)
        es = 4 if state_dtype == torch.float32 else 2
        n_own = (r1 - r0) * M
        # operands once, the partial gradient written once and read back by
        # the collective or the owner, the owner's shard of W, m, v
        self.owner_bytes = n_own * (4 + 8 + 4 * es)
        self.bytes = (K * N + K * M) * 2 + N * M * 4 + self.owner_bytes
        self.launches = 2
        self.wk = wl.Workload(f"owner_mlp K={K} d_in={N} d_out={M} (partial dW, reduce-scatter "
                              f"over {self.world} rank(s), owner AdamW)", K=K, N=N, M=M)

    def step(self, X=None, D=None, stream=None):
        import weight_grad_gemm_gb300 as fg
        if not hasattr(self, "G"):  # the warm-up steps of the constructor
            return Dense.step(self, X, D, stream)
        from weight_grad_gemm_gb300 import owner
        hp = self.hp
        fg.forge_wgrad_only(self.X if X is None else X, self.D if D is None else D, self.G,
                            stream=stream)
        r0, r1 = self.shard
        G = owner.reduce_scatter_rows(self.G, self.ranges) if self.world > 1 else self.G[r0:r1]
        if r1 > r0:
            fg.forge_owner_adamw(G, self.W[r0:r1], self.m[r0:r1], self.v[r0:r1], lr=hp.lr,
                                 beta1=hp.beta1, beta2=hp.beta2, eps=hp.eps, wd=hp.wd,
                                 step=self.t, stream=stream)
        self.t += 1

    def parts_us(self, stream, flush, reps=5):
        """Median device time of the partial dW and of the owner's step."""
        import weight_grad_gemm_gb300 as fg
        hp = self.hp
        r0, r1 = self.shard
        a, b = [], []
        for _ in range(reps):
            flush.zero_()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            ev[0].record(stream)
            fg.forge_wgrad_only(self.X, self.D, self.G, stream=stream)
            ev[1].record(stream)
            fg.forge_owner_adamw(self.G[r0:r1], self.W[r0:r1], self.m[r0:r1], self.v[r0:r1],
                                 lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2, eps=hp.eps, wd=hp.wd,
                                 step=self.t, stream=stream)
            ev[2].record(stream)
            ev[2].synchronize()
            self.t += 1
            a.append(ev[0].elapsed_time(ev[1]) * 1e3)
            b.append(ev[1].elapsed_time(ev[2]) * 1e3)
        return float(np.median(a)), float(np.median(b))


class Unfused:
    """The unfused pair on the same inputs: cuBLAS bf16 matmul (fp32
    accumulate, rounded to bf16 on output), .float(), then PyTorch's fused
    AdamW step -- the gradient makes a round trip through HBM.  With
    fp32_out, cuBLAS writes the fp32 accumulator itself (no bf16 rounding,
    torch.mm with out_dtype float32), then the same AdamW step."""

    def __init__(self, job: Dense, fp32_out: bool = False):
        self.job = job
        self.fp32_out = fp32_out
        self.W = torch.nn.Parameter(job.W.clone())
        hp = job.hp
        self.opt = torch.optim.AdamW([self.W], lr=hp.lr, betas=(hp.beta1, hp.beta2), eps=hp.eps,
                                     weight_decay=hp.wd, fused=True)
        self.opt.state[self.W] = {
            "step": torch.tensor(float(job.t - 1), device=job.W.device),
            "exp_avg": job.m.float().clone(), "exp_avg_sq": job.v.float().clone()}
        self.flops = job.flops
        self.params = job.params
        self.bytes = job.bytes
        self.wk = job.wk
        self.X = job.X
        self.D = job.D

    def step(self, X=None, D=None, stream=None):
        j = self.job
        Xt = (j.X if X is None else X).t()
        D = j.D if D is None else D
        if self.fp32_out:
            self.W.grad = torch.mm(Xt, D, out_dtype=torch.float32)
        else:
            self.W.grad = torch.matmul(Xt, D).float()
        self.opt.step()

    def inputs(self):
        return [self.X, self.D]

    def step_with(self, ins, stream=None):
        self.step(ins[0], ins[1], stream=stream)

    def result(self):
        return self.W


WORKLOADS = {
    "mlp_down": lambda dev, st: Dense(wl.MLP_DOWN, dev, st),
    "attn_proj": lambda dev, st: AttnSet(dev, st),
    "linear": lambda dev, st: Dense(wl.LINEAR, dev, st),
    "moe": lambda dev, st: MoE(dev, st),
    "moe_small": lambda dev, st: MoE(dev, st, wl.MOE_SMALL),
    "moe_decay": lambda dev, st: MoE(dev, st, wl.MOE_DECAY),
    "fp8": lambda dev, st: Fp8(dev, st, "AdamW"),
    "fp8_sgdm": lambda dev, st: Fp8(dev, st, "SGD"),
    "fp8_quant": lambda dev, st: Fp8Quant(dev, st),
    "backward": lambda dev, st: Backward(dev, st),
    "owner_mlp": lambda dev, st: OwnerStep(dev, st),
}


# ---------------------------------------------------------------- CPU oracle leg

def oracle_sample(job_X, job_D, job_W, job_m, job_v, hp, step, rows, scales=(1.0, 1.0)):
    """The oracle (fp64 CPU) on `rows` output rows of the workload: the
    contraction over all K for those rows and the AdamW step on them."""
    import oracle
    G = oracle.wgrad(job_X, job_D, rows=rows, scales=scales)
    oracle.adamw(G, job_W[rows], job_m[rows], job_v[rows], lr=hp.lr, beta1=hp.beta1,
                 beta2=hp.beta2, eps=hp.eps, wd=hp.wd, step=step)


# The contraction the CPU oracle times for each workload (see oracle_case).
ORACLE_SPECS = {"mlp_down": wl.MLP_DOWN, "backward": wl.MLP_DOWN, "owner_mlp": wl.MLP_DOWN,
                "attn_proj": wl.ATTN_PROJ[0],
                "linear": wl.LINEAR, "fp8": wl.FP8, "fp8_sgdm": wl.FP8, "fp8_quant": wl.FP8,
                "moe": wl.MOE, "moe_small": wl.MOE_SMALL, "moe_decay": wl.MOE_DECAY}


def oracle_case(workload):
    """The contraction the oracle times for a workload, on host copies of
    seeded inputs: the attention set by its widest projection, the MoE
    layers by one expert of their average token count, the fp8 workloads
    with e4m3 inputs and their scales.  Returns (workload spec, X, dY,
    scales, K, N, M)."""
    import oracle
    wk = ORACLE_SPECS[workload]
    K, N, M = wk.K // max(wk.experts, 1), wk.N, wk.M
    scales = (1.0, 1.0)
    if wk is wl.FP8:
        Xq, sx = wl.quantize_e4m3(wl.with_outliers((K, N), wl.seed_of(wk.name, "X8")))
        Dq, sy = wl.quantize_e4m3(wl.with_outliers((K, M), wl.seed_of(wk.name, "dY8")))
        X, D, scales = oracle.as_bits(Xq), oracle.as_bits(Dq), (sx, sy)
    else:
        X = oracle.as_bits(wl.activations(K, N, wl.seed_of(wk.name, "X")))
        D = oracle.as_bits(wl.activations(K, M, wl.seed_of(wk.name, "dY")))
    return wk, X, D, scales, K, N, M


def host_copies(job):
    import oracle
    X = oracle.as_bits(job.X.cpu())
    D = oracle.as_bits(job.D.cpu())
    W = job.W.float().cpu().numpy()
    m = job.m.float().cpu().numpy()
    v = job.v.float().cpu().numpy()
    return X, D, W, m, v


def cpu_baseline(job, workload, target_s=15.0):
    """The oracle's rate on the host cores: a dense job's own inputs and
    state, else the workload's oracle case (seeded inputs, warm state)."""
    import oracle
    oracle.build()
    scales = (1.0, 1.0)
    if type(job) is Dense:
        X, D, W, m, v = host_copies(job)
        K, N, M = job.wk.K, job.wk.N, job.wk.M
        hp, t = job.hp, job.t
    else:
        wk, X, D, scales, K, N, M = oracle_case(workload)
        rng = np.random.default_rng(0)
        W = (rng.standard_normal((N, M)) * 0.02).astype(np.float32)
        m = (rng.standard_normal((N, M)) * 1e-3).astype(np.float32)
        v = (rng.standard_normal((N, M)) * 1e-3).astype(np.float32) ** 2
        hp, t = wk.adam.f32(), 4
    oracle_sample(X, D, W, m, v, hp, t, list(range(2)), scales)  # warm caches and threads
    rows = list(range(32))
    t0 = time.perf_counter()
    oracle_sample(X, D, W, m, v, hp, t, rows, scales)
    t_cal = time.perf_counter() - t0
    n = int(max(32, min(N, 32 * target_s / max(t_cal, 1e-3))))
    rows = list(range(n))
    t0 = time.perf_counter()
    oracle_sample(X, D, W, m, v, hp, t, rows, scales)
    dt = time.perf_counter() - t0
    flops = 2.0 * n * M * K
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle", "seconds": dt,
            "sample": f"{n} of {N} output rows (all {M} columns, full K={K}) of dW + AdamW, "
                      f"fp64 C oracle with OpenMP"}


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    wk, X, D, scales, K, N, M = oracle_case(args.workload)
    hp = wk.adam.f32()
    rng = np.random.default_rng(0)
    # state rows only for the sampled output rows (the rest is never touched)
    total_budget_s = 150.0
    t0 = time.perf_counter()
    oracle_sample(X, D, (rng.standard_normal((1, M)) * 0.02).astype(np.float32),
                  np.zeros((1, M), np.float32), np.zeros((1, M), np.float32), hp, wk.first_step,
                  [0], scales)
    t1 = max(time.perf_counter() - t0, 1e-4)
    rows_per_step = int(max(1, min(N, total_budget_s / (args.steps + args.warmup) / t1)))
    Wr = (rng.standard_normal((rows_per_step, M)) * 0.02).astype(np.float32)
    mr = (rng.standard_normal((rows_per_step, M)) * 1e-3).astype(np.float32)
    vr = (rng.standard_normal((rows_per_step, M)) * 1e-3).astype(np.float32) ** 2
    rows = list(range(rows_per_step))
    for _ in range(args.warmup):
        oracle_sample(X, D, Wr, mr, vr, hp, wk.first_step, rows, scales)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample(X, D, Wr, mr, vr, hp, wk.first_step, rows, scales)
    dt = (time.perf_counter() - t0) / args.steps
    value = 2.0 * rows_per_step * M * K / dt / 1e12
    cores = len(os.sched_getaffinity(0))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wk.name, "K": K, "d_in": N, "d_out": M,
                   "sample_rows_per_step": rows_per_step},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{rows_per_step} of {N} output rows per step (all {M} "
                                   f"columns, full K={K}) of dW + AdamW"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- ranks

def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of every rank's x (the slowest rank's time); x itself on
    one rank.  Works on any initialised process group (NCCL with a CUDA
    device, gloo with the CPU)."""
    if world <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(flops_per_rank: float, world: int, ms: float) -> float:
    """TFLOP/s of the whole job: every replica does flops_per_rank per step,
    and the step takes the slowest rank's ms."""
    return flops_per_rank * world / (ms * 1e-3) / 1e12


# ---------------------------------------------------------------- ncu

def _csv_rows(path):
    import csv
    with open(path) as f:
        return [r for r in csv.reader(f) if r]


# Workloads that hold too much device memory for a full (multi-pass) ncu
# capture: their --ncu run stops after the one-pass launch list.
FULL_CAPTURE_TOO_LARGE = {"moe"}
# the kernel a workload's full capture targets, where it is not the fused one
CAPTURE_KERNEL = {"owner_mlp": "forge_owner"}


def run_ncu(args):
    """Profile the workload with ncu, following the pool's rules: the plain
    command first (it must exit 0), then a one-pass launch list, then one
    full capture of the first fused-kernel launch after the warm-up, all with
    --clock-control none.  Prints a JSON summary; for the MLP workload it also
    refreshes profiles/fused_adamw_mlp_down.json (the digest and traffic the
    timed runs report)."""
    import subprocess
    out = os.path.abspath(args.ncu)
    os.makedirs(out, exist_ok=True)
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "2", "--warmup", "3",
           "--no-cpu-baseline", "--no-per-config", "--e2e-steps", "1", "--workload",
           args.workload, "--state", args.state]
    subprocess.run(cmd, check=True, stdout=subprocess.DEVNULL)
    launches = os.path.join(out, "launches.csv")
    subprocess.run(["ncu", "--metrics", "gpu__time_duration.sum", "--clock-control", "none",
                    "--csv", "--log-file", launches, *cmd], check=True,
                   stdout=subprocess.DEVNULL)
    rows = _csv_rows(launches)
    start = next(i for i, r in enumerate(rows) if "Kernel Name" in r)
    hdr, rows = rows[start], rows[start + 1:]
    ki, mi, vi = hdr.index("Kernel Name"), hdr.index("Metric Name"), hdr.index("Metric Value")
    per = {}
    for r in rows:
        if len(r) > vi and r[mi] == "gpu__time_duration.sum":
            name = r[ki].split("(")[0]
            n, t = per.get(name, (0, 0.0))
            per[name] = (n + 1, t + float(r[vi].replace(",", "")))
    total = sum(t for _, t in per.values()) or 1.0
    table = [{"kernel": k, "launches": n, "total_us": t / 1e3, "share": t / total}
             for k, (n, t) in sorted(per.items(), key=lambda kv: -kv[1][1])]
    # the first fused launch after the state-warming steps (the owner's step
    # for the owner workload)
    kernel = CAPTURE_KERNEL.get(args.workload, "forge_wgrad")
    # a full capture replays the launch about forty times, saving and
    # restoring device memory around each pass: only on workloads of a few GB
    # (the MoE layer has the two-expert `moe_small` case for it)
    if args.workload in FULL_CAPTURE_TOO_LARGE:
        print(json.dumps({"workload": args.workload, "kernel": kernel, "launches": table,
                          "capture": None, "csrc_sha256": csrc_digest()}))
        return 0
    rep = os.path.join(out, "prof")
    subprocess.run(["ncu", "--set", "full", "--clock-control", "none", "-k",
                    f"regex:{kernel}", "-s", "3", "-c", "1", "-f", "-o", rep, *cmd], check=True,
                   stdout=subprocess.DEVNULL)
    raw = os.path.join(out, "prof_raw.csv")
    with open(raw, "w") as f:
        subprocess.run(["ncu", "-i", rep + ".ncu-rep", "--page", "raw", "--csv"], check=True,
                       stdout=f)
    hdr, units, vals = _csv_rows(raw)[:3]  # the raw page: names, units, one launch

    def metric(name):
        return float(vals[hdr.index(name)].replace(",", "")) if name in hdr else None

    def scaled(name):  # bytes, whatever unit ncu chose
        v = metric(name)
        scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
        return None if v is None else v * scale.get(units[hdr.index(name)], 1)

    rd, wr = scaled("dram__bytes_read.sum"), scaled("dram__bytes_write.sum")
    summary = {
        "workload": args.workload, "kernel": kernel, "launches": table,
        "capture": {"gpu_time_us": metric("gpu__time_duration.sum"),
                    "dram_bytes_read": rd, "dram_bytes_write": wr,
                    "tensor_active_pct": metric(
                        "sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active"),
                    "dram_throughput_pct": metric(
                        "gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed")},
        "csrc_sha256": csrc_digest(),
    }
    if args.workload == "mlp_down" and args.state == "f32" and rd is not None:
        p = os.path.join(ROOT, "profiles", "fused_adamw_mlp_down.json")
        with open(p) as f:
            doc = json.load(f)
        doc.update({"csrc_sha256": summary["csrc_sha256"], "dram_bytes_read": int(rd),
                    "dram_bytes_write": int(wr), "dram_bytes_per_launch": int(rd + wr),
                    "gpu_time_us_under_ncu": summary["capture"]["gpu_time_us"]})
        with open(p, "w") as f:
            json.dump(doc, f, indent=1)
    print(json.dumps(summary))
    return 0


# ---------------------------------------------------------------- end to end

def e2e_sequential(job, ins_h, res_h, dev, stream, flush, steps):
    """Milliseconds per step with each step alone: copy in, step, copy out."""
    ins_d = [torch.empty_like(h, device=dev) for h in ins_h]
    times = []
    for i in range(steps + 2):
        flush.zero_()
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        with torch.cuda.stream(stream):
            for d, h in zip(ins_d, ins_h):
                d.copy_(h, non_blocking=True)
            job.step_with(ins_d, stream=stream)
            res_h.copy_(job.result(), non_blocking=True)
        b.record(stream)
        b.synchronize()
        if i >= 2:
            times.append(a.elapsed_time(b))
    return float(np.mean(times)) if times else float("nan")


def e2e_pipelined(job, ins_h, res_h, dev, stream, steps):
    """Milliseconds per step over `steps` back-to-back steps, each with its
    own host->device copy of the inputs and device->host copy of the updated
    parameters.  The upload of step i+1 (double-buffered inputs, its own
    stream) overlaps step i; step i's parameters are snapshotted on the
    device right after it and read back on a third stream while step i+1
    runs (the next step updates W in place)."""
    res = job.result()
    bufs = [[torch.empty_like(h, device=dev) for h in ins_h] for _ in range(2)]
    snap = torch.empty_like(res)
    up = torch.cuda.Stream(dev)
    down = torch.cuda.Stream(dev)

    def run(n):
        ready = [torch.cuda.Event() for _ in range(2)]
        used = [torch.cuda.Event() for _ in range(2)]
        taken, read = torch.cuda.Event(), torch.cuda.Event()
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        up.wait_event(a)
        down.wait_event(a)
        for i in range(n):
            k = i % 2
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(used[k])  # step i-2 is done with this buffer
                for d, h in zip(bufs[k], ins_h):
                    d.copy_(h, non_blocking=True)
                ready[k].record(up)
            stream.wait_event(ready[k])
            job.step_with(bufs[k], stream=stream)
            used[k].record(stream)
            if i >= 1:
                stream.wait_event(read)  # the previous read-back is done with the snapshot
            with torch.cuda.stream(stream):
                snap.copy_(res, non_blocking=True)
            taken.record(stream)
            with torch.cuda.stream(down):
                down.wait_event(taken)
                res_h.copy_(snap, non_blocking=True)
                read.record(down)
        stream.wait_event(read)
        b.record(stream)
        b.synchronize()
        return a.elapsed_time(b) / max(n, 1)

    run(2)  # warm-up
    return run(steps)


# ---------------------------------------------------------------- our arm

# ---------------------------------------------------------------- timing helpers

def measure_e4m3_peak(dev, n=8192, reps=10):
    """Dense e4m3 rate of this GPU in TFLOP/s: cuBLAS through torch._scaled_mm
    on n^3 (fp32 accumulate, bf16 out, unit scales), best of `reps` launches
    timed with CUDA events.  None if the call is unavailable."""
    try:
        a = torch.randn((n, n), device=dev).to(torch.float8_e4m3fn)
        b = torch.randn((n, n), device=dev).to(torch.float8_e4m3fn).t()  # column-major
        one = torch.ones((), device=dev)
        for _ in range(3):
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        best = float("inf")
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
            e1.record()
            e1.synchronize()
            best = min(best, e0.elapsed_time(e1))
        del a, b
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    except (RuntimeError, TypeError, AttributeError):
        return None


def resident_bytes(job):
    """Bytes of the device tensors a job keeps (inputs and state), each
    storage counted once."""
    seen, total = set(), 0
    objs = [job] + list(getattr(job, "parts", []))
    for o in objs:
        for t in vars(o).values():
            if isinstance(t, torch.Tensor) and t.is_cuda:
                key = t.untyped_storage().data_ptr()
                if key not in seen:
                    seen.add(key)
                    total += t.untyped_storage().nbytes()
    return total


def job_dtype(job):
    return "e4m3" if getattr(job, "peak_key", "bf16") == "fp8" else "bf16"


def l2_note(job):
    return (f"flushed between steps (512 MiB write); inputs+state "
            f"{resident_bytes(job) / 1e9:.2f} GB > 129 MB L2")


def time_steps(job, steps, warmup, dev, local, flush, barrier):
    """W untimed steps, then `steps` steps each bracketed by CUDA events on
    the launch stream, L2 flushed before each (outside the events), clocks
    sampled throughout.  Returns (per-step ms list, clock record, wall s)."""
    import weight_grad_gemm_gb300 as fg
    stream = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        job.step()
    torch.cuda.synchronize(dev)
    if fg.forge_get_device_status() != fg.FORGE_OK:
        raise RuntimeError("device status not OK after warm-up")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for i in range(steps):
        flush.zero_()  # evict L2 between steps (outside the timed events)
        starts[i].record(stream)
        job.step(stream=stream)
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    wall = time.perf_counter() - wall0
    time.sleep(0.2)
    clk = clocks.stop()
    if fg.forge_get_device_status() != fg.FORGE_OK:
        raise RuntimeError("device status not OK after the timed region")
    return [s.elapsed_time(e) for s, e in zip(starts, ends)], clk, wall


def roofline_of(job, ms, peaks, peak_src, e4m3_peak):
    """The roofline record of a job's step time: tensor-bound against the
    peak of its own input type (bf16: the measured burst peak; e4m3: the
    rate measured in this run, else the bf16 peak times the nominal fp8/bf16
    ratio of 2), or HBM-bound against the measured copy bandwidth when its
    algorithmic bytes take longer than its FLOP."""
    peak_tf = peaks["bf16_tflops"]
    peak_note = f"bf16_tflops burst, {peak_src}"
    sustained_ratio = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) / peaks["bf16_tflops"]
    if getattr(job, "peak_key", "bf16") == "fp8":
        if e4m3_peak:
            peak_tf = e4m3_peak
            peak_note = "e4m3 dense, measured in this run (torch._scaled_mm 8192^3, best of 10)"
        else:
            peak_tf = peaks["bf16_tflops"] * 2.0
            peak_note = f"bf16_tflops burst x 2 (nominal fp8/bf16), {peak_src}"
    bw = peaks["hbm_gbs"]
    kernel_tf = job.flops / (ms * 1e-3) / 1e12
    t_tensor = job.flops / (peak_tf * 1e12)
    t_hbm = job.bytes / (bw * 1e9)
    if t_tensor >= t_hbm:
        r = {"bound": "tensor", "achieved": kernel_tf, "peak": peak_tf, "unit": "TFLOP/s",
             "frac": kernel_tf / peak_tf, "peak_source": peak_note,
             # the same against the power-capped (seconds-long) cuBLAS rate
             "frac_sustained": kernel_tf / (peak_tf * sustained_ratio)}
    else:
        gbs = job.bytes / (ms * 1e-3) / 1e9
        r = {"bound": "hbm", "achieved": gbs, "peak": bw, "unit": "GB/s", "frac": gbs / bw,
             "peak_source": f"hbm_gbs, {peak_src}"}
    return r, max(t_tensor, t_hbm) / (ms * 1e-3)


# The large configurations timed after the headline in the same process (the
# headline is the MLP down-projection): (label, workload, state dtype, steps
# rounded up to a multiple of this, so the MoE layer runs whole routing cycles).
PER_CONFIG = [
    ("attn_proj f32 state", "attn_proj", torch.float32, 1),
    ("attn_proj bf16 state", "attn_proj", torch.bfloat16, 1),
    ("moe f32 state, 6-step routing cycle", "moe", torch.float32, 6),
    ("moe bf16 state, 6-step routing cycle", "moe", torch.bfloat16, 6),
    ("fp8 e4m3 AdamW", "fp8", torch.float32, 1),
    ("fp8 e4m3 SGD-momentum", "fp8_sgdm", torch.float32, 1),
]


def per_config_lines(args, dev, local, flush, barrier, world, peaks, peak_src, e4m3_peak):
    out = {}
    for label, name, st, cycle in PER_CONFIG:
        try:
            out[label] = per_config_line(args, dev, local, flush, barrier, world, peaks, peak_src,
                                         e4m3_peak, name, st, cycle)
        except Exception as exc:
            # on one GPU a configuration's failure must not lose the headline
            # line; with several ranks it must end every rank (the others
            # would wait at the next barrier)
            if world > 1:
                raise
            out[label] = {"error": f"{type(exc).__name__}: {exc}"[:300]}
        torch.cuda.empty_cache()
    return out


def per_config_line(args, dev, local, flush, barrier, world, peaks, peak_src, e4m3_peak, name,
                    st, cycle):
    """One per-config entry: the workload set up, timed like the headline
    (whole routing cycles for the MoE layer) and its roofline record."""
    job = WORKLOADS[name](dev, st)
    steps = -(-args.steps // cycle) * cycle
    per_ms, clk, wall = time_steps(job, steps, args.warmup, dev, local, flush, barrier)
    ms = max_over_ranks(float(sum(per_ms)), world, dev) / steps
    roof, pct = roofline_of(job, ms, peaks, peak_src, e4m3_peak)
    line = {
        "workload": job.wk.name, "dtype": job_dtype(job),
        "state": "f32" if st == torch.float32 else "bf16",
        "steps": steps, "warmup": args.warmup, "ms_per_step": ms,
        "value": whole_job_rate(job.flops, world, ms), "unit": UNIT,
        "pct_roofline": pct, "roofline": roof,
        "updates_per_s": job.params * world / (ms * 1e-3),
        "gpu_launches": steps * getattr(job, "launches", 1),
        "l2": l2_note(job), "clocks": clk, "wall_s_timed_region": wall}
    del job
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours",
                    choices=["ours", "reference", "unfused", "unfused_f32"])
    ap.add_argument("--workload", default="mlp_down", choices=sorted(WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--state", default="f32", choices=["f32", "bf16"],
                    help="optimizer state type (default fp32, the headline workload)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only the chosen workload (by default the MLP down-projection "
                         "line also times the attention set, the MoE layer and the fp8 "
                         "workloads into its per_config object)")
    ap.add_argument("--ncu", metavar="DIR",
                    help="profile instead of timing: run the workload plainly, then under "
                         "ncu (launch list, then one full capture of the fused kernel), "
                         "write the raw reports to DIR and print the summary as JSON")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.ncu:
        return run_ncu(args)
    if args.impl == "reference":
        return run_reference(args)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    import weight_grad_gemm_gb300 as fg
    fg.lib()  # fails loudly if the CUDA library is not built

    job = WORKLOADS[args.workload](dev, torch.float32 if args.state == "f32" else torch.bfloat16)
    if args.impl in ("unfused", "unfused_f32"):
        if not isinstance(job, Dense):
            ap.error("--impl unfused is defined for the dense workloads")
        job = Unfused(job, fp32_out=args.impl == "unfused_f32")
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    per_step_ms, clk, wall = time_steps(job, args.steps, args.warmup, dev, local, flush, barrier)
    total_ms = max_over_ranks(float(sum(per_step_ms)), world, dev)
    ms = total_ms / args.steps
    value = whole_job_rate(job.flops, world, ms)

    # end to end through the C ABI with pinned host buffers: every step's
    # inputs are copied in and its updated parameters copied out
    ins_h = [t.cpu().pin_memory() for t in job.inputs()]
    res_h = torch.empty(job.result().shape, dtype=job.result().dtype).pin_memory()
    e2e_seq_ms = max_over_ranks(e2e_sequential(job, ins_h, res_h, dev, stream, flush,
                                               args.e2e_steps), world, dev)
    e2e_ms = max_over_ranks(e2e_pipelined(job, ins_h, res_h, dev, stream, args.e2e_steps),
                            world, dev)
    h2d = sum(h.numel() * h.element_size() for h in ins_h)
    d2h = res_h.numel() * res_h.element_size()

    peaks, peak_src = load_peaks()
    per_config = (args.workload == "mlp_down" and args.impl == "ours" and
                  not args.no_per_config)
    needs_e4m3 = per_config or getattr(job, "peak_key", "bf16") == "fp8"
    e4m3_peak = measure_e4m3_peak(dev) if args.impl == "ours" and needs_e4m3 else None
    roofline, pct = roofline_of(job, ms, peaks, peak_src, e4m3_peak)
    peak_tf = roofline["peak"] if roofline["bound"] == "tensor" else peaks["bf16_tflops"]
    bw = peaks["hbm_gbs"]
    prof = profile_summary() if (args.workload == "mlp_down" and args.state == "f32" and
                                 args.impl == "ours") else None
    traffic = prof.get("dram_bytes_per_launch") if prof else None
    gradw = prof.get("grad_w_hbm_bytes") if prof else None
    roofline["traffic"] = traffic

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "impl": args.impl,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": job_dtype(job), "data": "synthetic",
        "config": {"workload": job.wk.name + f" {getattr(job, 'opt', 'AdamW')} {args.state} state",
                   "K": job.wk.K, "d_in": job.wk.N, "d_out": job.wk.M,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": l2_note(job)},
        "pct_roofline": pct,
        "e4m3_peak_tflops": e4m3_peak,
        "updates_per_s": job.params * world / (ms * 1e-3),
        "grad_w_hbm_bytes": gradw,
        "roofline": roofline,
        "e2e": {"value": whole_job_rate(job.flops, world, e2e_ms), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms, "pipelined": True,
                "sequential_value": whole_job_rate(job.flops, world, e2e_seq_ms)},
        "gpu_launches": args.steps * getattr(job, "launches", 1) if args.impl == "ours" else 0,
        "clocks": clk,
        "wall_s_timed_region": wall,
    }
    if isinstance(job, Backward):
        d_us, f_us = job.parts_us(stream, flush)
        wk = job.wk
        tf = 2.0 * wk.K * wk.N * wk.M / (d_us * 1e-6) / 1e12
        line["dgrad"] = {"us": d_us, "fused_us": f_us, "bound": "tensor", "achieved": tf,
                         "peak": peak_tf, "unit": "TFLOP/s", "frac": tf / peak_tf}
    if isinstance(job, OwnerStep):
        d_us, o_us = job.parts_us(stream, flush)
        gbs = job.owner_bytes / (o_us * 1e-6) / 1e9
        line["owner"] = {"wgrad_only_us": d_us, "owner_adamw_us": o_us, "bound": "hbm",
                         "achieved": gbs, "peak": bw, "unit": "GB/s", "frac": gbs / bw,
                         "bytes": job.owner_bytes,
                         "collective": "reduce_scatter_tensor (NCCL)" if world > 1 else
                         "none (one rank owns every row)"}
    if isinstance(job, Fp8Quant):
        q_us, f_us = job.parts_us(stream, flush)
        gbs = job.quant_bytes / (q_us * 1e-6) / 1e9
        line["quantize"] = {"us": q_us, "fused_us": f_us, "bound": "hbm", "achieved": gbs,
                            "peak": bw, "unit": "GB/s", "frac": gbs / bw,
                            "bytes": job.quant_bytes}
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.impl == "ours":
        line["cpu_baseline"] = cpu_baseline(job, args.workload)
    if per_config:
        # the headline's own tensors are not needed any more
        del job, ins_h, res_h
        torch.cuda.empty_cache()
        line["per_config"] = per_config_lines(args, dev, local, flush, barrier, world, peaks,
                                              peak_src, e4m3_peak)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

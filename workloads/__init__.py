"""Seeded synthetic inputs for the fused weight-gradient + optimizer path.

This module serves both the CUDA path and the oracle.  It draws random
tensors and routing decisions and quantizes fp8 inputs; it holds none of the
method's arithmetic (no contraction, no optimizer step).

Workloads (shapes, value distributions and hyperparameters):

* ``linear``   -- one linear layer, X [512, 256], dY [512, 256] bf16 with
  entries N(0,1)*0.05, W [256, 256] fp32 N(0, 0.02), m = v = 0, AdamW
  lr 1e-3, betas (0.9, 0.999), eps 1e-8, wd 0.01, 10 steps with fresh X, dY.
* ``mlp_down`` -- Llama-style MLP down-projection wgrad: K = 8192 tokens,
  d_in = 14336, d_out = 4096; X, dY bf16 N(0,1)/sqrt(d) (d = that tensor's
  feature width); W fp32 N(0, 0.02); fp32 m, v warmed by 3 prior steps; the
  timed step is t = 4.
* ``attn_proj`` -- four wgrads at d_in = 4096, d_out in {4096, 1024, 1024,
  4100}, K = 16384, bf16 N(0,1)/sqrt(d), AdamW wd = 0.1, fp32 state and
  again bf16 m/v state.
* ``moe``      -- 8 experts of W [14336, 4096] fp32; 16384 tokens routed
  top-2 (two distinct experts per token) with Zipf(1.2) expert popularity
  (p proportional to r^-1.2 over a per-step seeded permutation of ranks); on
  steps 2, 4, 6 a seeded set of 4 experts receives no tokens; packed X
  [32768, 14336], dY [32768, 4096] bf16; 6 AdamW steps.
* ``fp8``      -- X, dY [32768, 8192] N(0,1) with 0.1% of entries set to
  +-20 (seeded positions and signs), quantized to e4m3 with the per-tensor
  scale amax / 448; AdamW (the ``linear`` hyperparameters) and SGD momentum
  0.9, lr 1e-2, wd 0.

No public dataset is involved; everything is drawn from seeded generators.
"""
from __future__ import annotations

import math
import zlib
from dataclasses import dataclass, field

import numpy as np
import torch

E4M3_MAX = 448.0


def seed_of(*parts) -> int:
    """Stable 31-bit seed from (workload, step, tensor name, ...)."""
    return zlib.crc32("/".join(str(p) for p in parts).encode()) & 0x7FFFFFFF


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def randn(shape, seed, device="cpu", std=1.0, dtype=torch.float32):
    """N(0, std^2) in fp32, rounded once to ``dtype``."""
    g = _gen(device, seed)
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def activations(K, width, seed, device="cpu", scale=None, dtype=torch.bfloat16):
    """Token-major activations / output grads [K, width]: N(0,1) * scale
    (default 1/sqrt(width)), rounded to ``dtype``."""
    s = (1.0 / math.sqrt(width)) if scale is None else scale
    return randn((K, width), seed, device, std=s, dtype=dtype)


def with_outliers(shape, seed, device="cpu", frac=1e-3, value=20.0):
    """N(0,1) fp32 with a seeded fraction ``frac`` of entries set to +-value."""
    t = randn(shape, seed, device)
    numel = t.numel()
    if numel == 0:
        return t
    g = _gen(device, seed ^ 0x5A5A5A5)
    n_out = max(1, int(round(numel * frac)))
    idx = torch.randint(0, numel, (n_out,), generator=g, device=device)
    sign = torch.randint(0, 2, (n_out,), generator=g, device=device).to(torch.float32) * 2 - 1
    t.view(-1)[idx] = sign * value
    return t


def quantize_e4m3(t: torch.Tensor):
    """Per-tensor scale s = amax / 448 and codes = RNE(t / s) in e4m3fn.
    Returns (codes, s) with s a python float (fp32 value)."""
    amax = float(t.abs().max()) if t.numel() else 0.0
    s = float(np.float32(amax / E4M3_MAX)) if amax > 0 else 1.0
    codes = (t / s).to(torch.float8_e4m3fn)
    return codes, s


def zipf_top2_counts(seed, tokens=16384, experts=8, topk=2, zipf_s=1.2, zero_experts=()):
    """Tokens per expert for top-k routing without replacement.

    Expert popularity is Zipf(zipf_s) over a seeded permutation of ranks;
    experts in ``zero_experts`` have probability 0.  Each token draws
    ``topk`` distinct experts (successive draws without replacement).
    Returns an int64 numpy array of counts (sum = tokens * topk)."""
    rng = np.random.default_rng(seed)
    ranks = rng.permutation(experts) + 1
    p = ranks.astype(np.float64) ** (-zipf_s)
    for e in zero_experts:
        p[e] = 0.0
    active = int((p > 0).sum())
    if active < topk:
        raise ValueError("fewer active experts than top-k")
    p = p / p.sum()
    # Gumbel-top-k draws k distinct experts with the successive-sampling law.
    logp = np.where(p > 0, np.log(np.where(p > 0, p, 1.0)), -np.inf)
    gumbel = rng.gumbel(size=(tokens, experts))
    choice = np.argsort(-(logp[None, :] + gumbel), axis=1)[:, :topk]
    return np.bincount(choice.reshape(-1), minlength=experts).astype(np.int64)


def moe_zero_experts(seed, experts=8, n_zero=4):
    rng = np.random.default_rng(seed)
    return tuple(sorted(rng.choice(experts, size=n_zero, replace=False).tolist()))


def offsets_from_counts(counts):
    off = np.zeros(len(counts) + 1, np.int64)
    off[1:] = np.cumsum(counts)
    return off


@dataclass
class AdamHP:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    wd: float = 0.01

    def f32(self):
        """Hyperparameters as the fp32 values the library receives."""
        return AdamHP(*(float(np.float32(x)) for x in (self.lr, self.beta1, self.beta2,
                                                      self.eps, self.wd)))


@dataclass
class SgdHP:
    lr: float = 1e-2
    momentum: float = 0.9
    wd: float = 0.0

    def f32(self):
        return SgdHP(*(float(np.float32(x)) for x in (self.lr, self.momentum, self.wd)))


@dataclass
class Workload:
    name: str
    K: int
    N: int  # d_in
    M: int  # d_out
    adam: AdamHP = field(default_factory=AdamHP)
    steps: int = 1
    first_step: int = 1
    experts: int = 0

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K


LINEAR = Workload("linear K=512 d_in=256 d_out=256", K=512, N=256, M=256, steps=10)
MLP_DOWN = Workload("mlp_down K=8192 d_in=14336 d_out=4096", K=8192, N=14336, M=4096,
                    first_step=4)
ATTN_OUTS = (4096, 1024, 1024, 4100)
ATTN_PROJ = [Workload(f"attn_proj K=16384 d_in=4096 d_out={m}", K=16384, N=4096, M=m,
                      adam=AdamHP(wd=0.1)) for m in ATTN_OUTS]
MOE = Workload("moe E=8 tokens=16384 top2 d_in=14336 d_out=4096", K=32768, N=14336, M=4096,
               steps=6, experts=8)
MOE_SMALL = Workload("moe_small E=2 tokens=4096 top2 d_in=14336 d_out=4096", K=8192, N=14336,
                     M=4096, steps=1, experts=2)
MOE_DECAY = Workload("moe_decay E=2 tokens=0 d_in=14336 d_out=4096", K=0, N=14336, M=4096,
                     steps=1, experts=2)
FP8 = Workload("fp8 K=32768 d_in=8192 d_out=8192", K=32768, N=8192, M=8192)
FP8_SGD = SgdHP(lr=1e-2, momentum=0.9, wd=0.0)

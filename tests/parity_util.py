"""Comparison rules between the CUDA path and the fp64 oracle.

Tolerances (the contract of the fused path):
* dW: relative Frobenius error <= 2e-3 for bf16 inputs, <= 3e-2 for e4m3.
  Both paths see identical inputs (the fp8 codes and scales), so the only
  difference is fp32 accumulation; a tighter diagnostic bound (1e-5) is
  also asserted, which any dropped k-block, tile or operand slip breaks.
* fp32 state (m, v, momentum): elementwise |error| <= 2e-3 * rms(oracle).
* bf16 state: the stored value must be the round-to-nearest-even bf16 of the
  oracle's exact value, except that the other bracketing bf16 value is
  accepted where the exact value lies within ``band`` (relative) of the
  midpoint between them -- fp32 arithmetic on the GPU cannot decide such
  near-ties the way fp64 does.  The count of such elements is returned.
* W: |error| <= 1e-2 * lr wherever |g| > 1e-2 * rms(g) (per tensor; per
  expert in the grouped call; where an expert has g = 0 the mask is
  |m_exact| > 1e-2 * rms(m_exact)).
"""
import numpy as np

import oracle

DW_TOL = {"bf16": 2e-3, "e4m3": 3e-2}
DW_DIAG_TOL = 1e-5
STATE_TOL = 2e-3
W_TOL = 1e-2
BF16_TIE_BAND = 2.0 ** -14


def rms(x):
    x = np.asarray(x, dtype=np.float64)
    return float(np.sqrt(np.mean(x * x))) if x.size else 0.0


def rel_fro(gpu, ref):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(gpu - ref)
    return num / den if den > 0 else num


def check_dw(gpu, ref, kind="bf16"):
    e = rel_fro(gpu, ref)
    assert e <= DW_TOL[kind], f"dW relative Frobenius error {e:.3e} > {DW_TOL[kind]}"
    assert e <= DW_DIAG_TOL, f"dW relative Frobenius error {e:.3e} > diagnostic {DW_DIAG_TOL}"
    return e


def check_state_f32(gpu, exact, name="state"):
    gpu = np.asarray(gpu, np.float64)
    exact = np.asarray(exact, np.float64)
    bound = STATE_TOL * rms(exact)
    err = np.max(np.abs(gpu - exact)) if gpu.size else 0.0
    assert err <= bound, f"{name}: max |error| {err:.3e} > 2e-3*rms = {bound:.3e}"
    return err


def check_state_bf16(gpu_bits, exact, name="state", band=BF16_TIE_BAND):
    gpu_bits = np.asarray(gpu_bits).astype(np.uint16).ravel()
    exact = np.asarray(exact, np.float64).ravel()
    rn = oracle.round_bf16(exact)
    bad = np.nonzero(gpu_bits != rn)[0]
    if bad.size == 0:
        return 0
    g = oracle.decode(gpu_bits[bad])
    r = oracle.decode(rn[bad])
    x = exact[bad]
    # the GPU value must be the other neighbour bracketing x ...
    lo = np.minimum(g, r)
    hi = np.maximum(g, r)
    bracket = (lo <= x) & (x <= hi)
    adjacent = np.abs(gpu_bits[bad].astype(np.int32) - rn[bad].astype(np.int32)) == 1
    # ... and x must sit within `band` of their midpoint
    near_tie = np.abs(x - (lo + hi) / 2) <= band * np.abs(x)
    ok = bracket & adjacent & near_tie
    assert ok.all(), (f"{name}: {int((~ok).sum())} bf16 values are not the rounding of the "
                      f"exact value (first: gpu {g[~ok][:3]}, exact {x[~ok][:3]})")
    return int(bad.size)


def check_W(gpu_W, exact_W, G, lr, m_exact=None, name="W"):
    gpu_W = np.asarray(gpu_W, np.float64)
    exact_W = np.asarray(exact_W, np.float64)
    G = np.asarray(G, np.float64)
    rg = rms(G)
    if rg > 0:
        mask = np.abs(G) > 1e-2 * rg
    else:
        assert m_exact is not None
        mm = np.asarray(m_exact, np.float64)
        mask = np.abs(mm) > 1e-2 * rms(mm)
    err = np.max(np.abs(gpu_W - exact_W)[mask]) if mask.any() else 0.0
    assert err <= W_TOL * lr, f"{name}: max |error| {err:.3e} > 1e-2*lr = {W_TOL * lr:.3e}"
    return err

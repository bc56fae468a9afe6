"""Comparison rules between the CUDA path and the fp64 oracle.

Tolerances (the contract of the fused path):
* dW: relative Frobenius error <= 2e-3 for bf16 inputs, <= 3e-2 for e4m3.
  Both paths see identical inputs (the fp8 codes and scales), so the only
  difference is fp32 accumulation; a tighter diagnostic bound (1e-5) is
  also asserted, which any dropped k-block, tile or operand slip breaks.
* fp32 state (m, v, momentum): elementwise |error| <= 2e-3 * rms(oracle);
  a diagnostic bound |error| <= 1e-5 * rms + 2^-20 |exact| is asserted too
  (fp32 arithmetic on the GPU sits far inside it; a wrong coefficient does
  not).
* bf16 state: the stored value must be the round-to-nearest-even bf16 of
  some y with |y - exact| within that same diagnostic band, i.e. the state
  contract applied before the rounding to storage.  Where the exact value is
  near a rounding midpoint, fp32 arithmetic may land on the other side, so
  the stored value may be the other bracketing neighbour; the count of such
  elements is returned.
* W: |error| <= 1e-2 * lr wherever |g| > 1e-2 * rms(g) (per tensor; per
  expert in the grouped call; where an expert has g = 0 the mask is
  |m_exact| > 1e-2 * rms(m_exact)).
* W on every element (diagnostic): W' recomputed in fp64 from the old W and
  the kernel's own stored m', v' must match the kernel's W' within the
  rounding of the epilogue's few fp32 operations and its approximate square
  root and reciprocal (2^-19 of the update plus 2^-21 |W|); with bf16 state
  the stored m', v' are the rounded copies of the values the update used,
  so the update term gets 2^-7.  This covers the parameters whose gradient
  is too small for the mask above, where the gradient's own fp32
  accumulation error would dominate a comparison with the oracle.
"""
import numpy as np

import oracle

DW_TOL = {"bf16": 2e-3, "e4m3": 3e-2}
DW_DIAG_TOL = 1e-5
STATE_TOL = 2e-3
W_TOL = 1e-2
STATE_DIAG_RMS = 1e-5
STATE_DIAG_REL = 2.0 ** -20


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


def _band(exact):
    exact = np.asarray(exact, np.float64)
    return STATE_DIAG_RMS * rms(exact) + STATE_DIAG_REL * np.abs(exact)


def check_state_f32(gpu, exact, name="state", diag=True):
    """Contract bound always; the tight diagnostic band when `diag` (it is
    calibrated for K up to about a thousand tokens, where fp32 accumulation
    error in g stays below it)."""
    gpu = np.asarray(gpu, np.float64)
    exact = np.asarray(exact, np.float64)
    if not gpu.size:
        return 0.0
    bound = STATE_TOL * rms(exact)
    err = np.abs(gpu - exact)
    assert err.max() <= bound, f"{name}: max |error| {err.max():.3e} > 2e-3*rms = {bound:.3e}"
    if diag:
        over = err > _band(exact)
        assert not over.any(), (f"{name}: {int(over.sum())} elements beyond the diagnostic band "
                                f"(worst {err.max():.3e}, rms {rms(exact):.3e})")
    return float(err.max())


def check_state_bf16(gpu_bits, exact, name="state", diag=True):
    """The stored bf16 must be the rounding of some value within the band of
    the exact value: the diagnostic band when `diag`, else the contract's
    2e-3 * rms."""
    gpu_bits = np.asarray(gpu_bits).astype(np.uint16).ravel()
    exact = np.asarray(exact, np.float64).ravel()
    rn = oracle.round_bf16(exact)
    bad = np.nonzero(gpu_bits != rn)[0]
    if bad.size == 0:
        return 0
    band = (_band(exact) if diag else np.full(exact.shape, STATE_TOL * rms(exact)))[bad]
    x = exact[bad]
    g = oracle.decode(gpu_bits[bad])
    lo = oracle.decode(oracle.round_bf16(x - band))
    hi = oracle.decode(oracle.round_bf16(x + band))
    ok = (lo <= g) & (g <= hi)
    assert ok.all(), (f"{name}: {int((~ok).sum())} bf16 values are not the rounding of a value "
                      f"within the band (first: gpu {g[~ok][:3]}, exact {x[~ok][:3]}, "
                      f"rms {rms(exact):.3e})")
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


def check_grad_from_m(m_gpu, m_old, G, beta1, name="g from m"):
    """Reconstruct the gradient the kernel used from m' = b1 m + (1-b1) g and
    compare it with the oracle's g: the dW contract (relative Frobenius
    <= 2e-3) and a diagnostic bound of 1e-4 for long contractions."""
    m_gpu = np.asarray(m_gpu, np.float64)
    m_old = np.asarray(m_old, np.float64)
    g = (m_gpu - beta1 * m_old) / (1.0 - beta1)
    e = rel_fro(g, G)
    assert e <= DW_TOL["bf16"], f"{name}: relative Frobenius {e:.3e} > {DW_TOL['bf16']}"
    assert e <= 1e-4, f"{name}: relative Frobenius {e:.3e} > diagnostic 1e-4"
    return e


def check_W_from_state(gpu_W, W_old, m_new, v_new, hp, step, state_bf16, name="W (all)"):
    """The diagnostic W bound over every element (module docstring).  m_new,
    v_new: the kernel's stored state (fp32 values or bf16 bits)."""
    dec = (lambda a: oracle.decode(np.asarray(a).astype(np.uint16))) if state_bf16 else \
        (lambda a: np.asarray(a, np.float64))
    m = dec(m_new).astype(np.float64).reshape(-1)
    v = dec(v_new).astype(np.float64).reshape(-1)
    W0 = np.asarray(W_old, np.float64).reshape(-1)
    got = np.asarray(gpu_W, np.float64).reshape(-1)
    lr, b1, b2, eps, wd = (float(hp.lr), float(hp.beta1), float(hp.beta2), float(hp.eps),
                           float(hp.wd))
    bc1 = 1.0 - b1 ** step
    bc2 = 1.0 - b2 ** step
    r = (m / bc1) / (np.sqrt(v / bc2) + eps)
    want = W0 * (1.0 - lr * wd) - lr * r
    upd = 2.0 ** -7 if state_bf16 else 2.0 ** -19
    bound = upd * lr * np.abs(r) + 2.0 ** -21 * np.maximum(np.abs(W0), np.abs(want)) + 1e-38
    err = np.abs(got - want)
    bad = err > bound
    assert not bad.any(), (f"{name}: {int(bad.sum())} of {err.size} elements off the update "
                           f"their own state implies (worst {err.max():.3e})")
    return float(err.max()) if err.size else 0.0

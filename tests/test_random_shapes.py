"""A seeded sweep of random problem shapes against the fp64 oracle: dense
AdamW and SGD-momentum calls over random K, d_in, d_out (aligned or not,
bf16 or e4m3 inputs, fp32 or bf16 state), grouped calls over random expert
counts, multi-problem calls over random problem counts and widths, and
dX = dY Wb^T over random shapes.  The shapes are drawn once from a fixed seed, so a failure
names a reproducible case; sizes stay small enough for the oracle."""
import numpy as np
import pytest

import oracle
from test_parity import (HP, adamw_ref, bf16_inputs, check_adamw, check_grouped, e4m3_inputs,
                         grouped_case, run_adamw, run_grouped, warm_state)

pytestmark = pytest.mark.gpu


def dense_cases(n=48, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        K = int(rng.choice([0, 1, int(rng.integers(2, 700))], p=[0.08, 0.08, 0.84]))
        N = int(rng.integers(1, 700))
        M = int(rng.integers(1, 900))
        kind = "e4m3" if rng.random() < 0.3 else "bf16"
        state_bf16 = bool(rng.random() < 0.4)
        out.append((i, K, N, M, kind, state_bf16))
    return out


def grouped_cases(n=16, seed=2025):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        E = int(rng.integers(1, 12))
        counts = rng.integers(0, 160, size=E)
        counts[rng.random(E) < 0.3] = 0
        N = int(rng.integers(8, 520))
        M = int(rng.integers(8, 600))
        kind = "e4m3" if rng.random() < 0.3 else "bf16"
        out.append((i, [int(c) for c in counts], N, M, kind))
    return out


@pytest.mark.parametrize("i,K,N,M,kind,state_bf16", dense_cases(),
                         ids=lambda v: str(v) if not isinstance(v, bool) else ("bf16st" if v else "f32st"))
def test_random_dense_adamw(cuda_device, i, K, N, M, kind, state_bf16):
    if kind == "bf16":
        X, D = bf16_inputs(K, N, M, 300 + i)
        sc = None
    else:
        X, D, sc = e4m3_inputs(K, N, M, 300 + i)
    W, m, v = warm_state(N, M, 400 + i, state_bf16)
    got = run_adamw(cuda_device, X, D, W, m, v, step=3, scales=sc)
    G = oracle.wgrad(X, D, scales=sc or (1.0, 1.0))
    ref = adamw_ref(G, W, m, v, step=3, **vars(HP))
    check_adamw(got, ref, G, HP.lr, state_bf16)


@pytest.mark.parametrize("i,counts,N,M,kind", grouped_cases(), ids=lambda v: str(v)[:24])
def test_random_grouped_adamw(cuda_device, i, counts, N, M, kind):
    X, D, off, W, m, v, sc = grouped_case(counts, N, M, 500 + i, kind=kind)
    got = run_grouped(cuda_device, X, D, off, W, m, v, step=2, scales=sc)
    check_grouped(got, X, D, off, W, m, v, 2, sc, False)


@pytest.mark.parametrize("i,K,N,M,kind,state_bf16", dense_cases(n=8, seed=2026),
                         ids=lambda v: str(v) if not isinstance(v, bool) else ("bf16st" if v else "f32st"))
def test_random_dense_sgdm(cuda_device, i, K, N, M, kind, state_bf16):
    import torch

    import weight_grad_gemm_gb300 as fg
    from parity_util import check_state_bf16, check_state_f32, rms
    from test_parity import dev_state, host_state, scales_dev
    if kind == "bf16":
        X, D = bf16_inputs(K, N, M, 600 + i)
        sc = None
    else:
        X, D, sc = e4m3_inputs(K, N, M, 600 + i)
    W, buf, _ = warm_state(N, M, 700 + i, state_bf16)
    lr, mu, wd = float(np.float32(1e-2)), float(np.float32(0.9)), float(np.float32(0.05))
    Wd, bd = dev_state(W, cuda_device), dev_state(buf, cuda_device)
    fg.forge_wgrad_sgdm(X.to(cuda_device), D.to(cuda_device), Wd, bd, lr=lr, momentum=mu, wd=wd,
                        scales=None if sc is None else scales_dev(sc, cuda_device))
    torch.cuda.synchronize()
    G = oracle.wgrad(X, D, scales=sc or (1.0, 1.0))
    ref = oracle.sgdm(G, W, buf, lr=lr, momentum=mu, wd=wd)
    if state_bf16:
        check_state_bf16(host_state(bd), ref["buf_exact"], "buf")
    else:
        check_state_f32(host_state(bd), ref["buf_exact"], "buf")
    err = np.max(np.abs(host_state(Wd).astype(np.float64) - ref["W_exact"]))
    assert err <= 2e-3 * lr * rms(ref["buf_exact"]) + 2 * np.finfo(np.float32).eps * 0.1


def multi_cases(n=6, seed=2027):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        P = int(rng.integers(1, 9))
        Ms = [int(rng.integers(1, 700)) for _ in range(P)]
        K = int(rng.integers(0, 400))
        N = int(rng.integers(1, 600))
        out.append((i, K, N, Ms, bool(rng.random() < 0.5)))
    return out


@pytest.mark.parametrize("i,K,N,Ms,state_bf16", multi_cases(), ids=lambda v: str(v)[:30])
def test_random_multi(cuda_device, i, K, N, Ms, state_bf16):
    from test_multi import case, run_multi
    X, Ds, states = case(K, N, Ms, 800 + i, state_bf16)
    got = run_multi(cuda_device, X, Ds, states, step=2)
    for D, (W, m, v), g in zip(Ds, states, got):
        G = oracle.wgrad(X, D)
        check_adamw(g, adamw_ref(G, W, m, v, step=2, **vars(HP)), G, HP.lr, state_bf16)


def dgrad_cases(n=8, seed=2028):
    rng = np.random.default_rng(seed)
    return [(i, int(rng.integers(1, 600)), int(rng.integers(1, 600)), int(rng.integers(1, 900)))
            for i in range(n)]


@pytest.mark.parametrize("i,K,N,M", dgrad_cases(), ids=lambda v: str(v))
def test_random_dgrad(cuda_device, i, K, N, M):
    import torch

    import weight_grad_gemm_gb300 as fg
    from test_dgrad import check_dx, inputs
    D, Wb = inputs(K, N, M, 900 + i, cuda_device)
    dX = torch.full((K, N), float("nan"), dtype=torch.bfloat16, device=cuda_device)
    fg.forge_dgrad(D, Wb, dX)
    torch.cuda.synchronize()
    check_dx(dX, oracle.dgrad(oracle.as_bits(D.cpu()), oracle.as_bits(Wb.cpu())))

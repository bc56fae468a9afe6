"""GPU parity of the multi-problem entry: several AdamW weight-gradient
steps sharing X, in one launch, against the fp64 oracle per problem, and
bitwise against one forge_wgrad_adamw call per problem where that call runs
on CTA pairs (d_out > 128).
"""
import numpy as np
import pytest
import torch

import oracle
import weight_grad_gemm_gb300 as fg
from test_parity import (HP, adamw_ref, bf16_inputs, check_adamw, dev_state, host_state,
                         warm_state)

pytestmark = pytest.mark.gpu

# d_out per problem: several pair tiles with ragged edges, one below a pair
# tile, one below a single tile, and 130 (260-byte dY rows: staged)
MS = [392, 136, 96, 260, 130]


def case(K, N, Ms, seed, state_bf16):
    X, _ = bf16_inputs(K, N, Ms[0], seed)
    Ds = [bf16_inputs(K, N, M, seed + 100 + j)[1] for j, M in enumerate(Ms)]
    states = [warm_state(N, M, seed + 200 + j, state_bf16) for j, M in enumerate(Ms)]
    return X, Ds, states


def run_multi(dev, X, Ds, states, step, hp=HP):
    dst = [[dev_state(a, dev) for a in s] for s in states]
    fg.forge_wgrad_adamw_multi(X.to(dev), [D.to(dev) for D in Ds], [s[0] for s in dst],
                               [s[1] for s in dst], [s[2] for s in dst], lr=hp.lr,
                               beta1=hp.beta1, beta2=hp.beta2, eps=hp.eps, wd=hp.wd, step=step)
    torch.cuda.synchronize()
    return [tuple(host_state(t) for t in s) for s in dst]


def run_single(dev, X, Ds, states, step, hp=HP):
    out = []
    Xd = X.to(dev)
    for D, s in zip(Ds, states):
        W, m, v = (dev_state(a, dev) for a in s)
        fg.forge_wgrad_adamw(Xd, D.to(dev), W, m, v, lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2,
                             eps=hp.eps, wd=hp.wd, step=step)
        torch.cuda.synchronize()
        out.append((host_state(W), host_state(m), host_state(v)))
    return out


@pytest.mark.parametrize("state_bf16", [False, True], ids=["f32state", "bf16state"])
@pytest.mark.parametrize("K", [200, 0, 1])
def test_multi_matches_oracle(cuda_device, K, state_bf16):
    N = 264
    X, Ds, states = case(K, N, MS, 31, state_bf16)
    got = run_multi(cuda_device, X, Ds, states, step=3)
    for D, (W, m, v), g in zip(Ds, states, got):
        G = oracle.wgrad(X, D)
        ref = adamw_ref(G, W, m, v, step=3, **vars(HP))
        check_adamw(g, ref, G, HP.lr, state_bf16)


@pytest.mark.parametrize("state_bf16", [False, True], ids=["f32state", "bf16state"])
def test_multi_bitwise_equals_single_calls(cuda_device, state_bf16):
    K, N = 300, 520
    X, Ds, states = case(K, N, MS, 32, state_bf16)
    multi = run_multi(cuda_device, X, Ds, states, step=5)
    single = run_single(cuda_device, X, Ds, states, step=5)
    for M, a, b in zip(MS, multi, single):
        if M > 128:
            for x, y in zip(a, b):
                assert np.array_equal(x, y), f"d_out {M}: multi and single calls differ"


def test_multi_eight_problems_and_one(cuda_device):
    K, N = 130, 136
    Ms = [8, 264, 12, 256, 520, 4, 136, 300]
    X, Ds, states = case(K, N, Ms, 33, False)
    got = run_multi(cuda_device, X, Ds, states, step=2)
    for D, (W, m, v), g in zip(Ds, states, got):
        G = oracle.wgrad(X, D)
        check_adamw(g, adamw_ref(G, W, m, v, step=2, **vars(HP)), G, HP.lr, False)
    one = run_multi(cuda_device, X, Ds[4:5], states[4:5], step=2)
    assert all(np.array_equal(x, y) for x, y in zip(one[0], got[4]))


def test_multi_run_to_run_bitwise(cuda_device):
    K, N = 257, 264
    X, Ds, states = case(K, N, MS, 34, False)
    a = run_multi(cuda_device, X, Ds, states, step=4)
    b = run_multi(cuda_device, X, Ds, states, step=4)
    for x, y in zip(a, b):
        assert all(np.array_equal(u, w) for u, w in zip(x, y))


def test_multi_with_staged_x(cuda_device):
    # d_in 262: X rows of 524 bytes, staged into 16-byte rows along with the
    # 260-byte dY rows of the 130-wide problem
    K, N = 150, 262
    Ms = [264, 130, 64]
    X, Ds, states = case(K, N, Ms, 35, False)
    got = run_multi(cuda_device, X, Ds, states, step=2)
    for D, (W, m, v), g in zip(Ds, states, got):
        G = oracle.wgrad(X, D)
        check_adamw(g, adamw_ref(G, W, m, v, step=2, **vars(HP)), G, HP.lr, False)


def test_multi_odd_widths(cuda_device):
    # d_in 263 (526-byte X rows) and d_out 301, 3 and 4097: every operand's
    # rows are a multiple of 2 bytes only, staged by the byte-granular copy
    K, N = 140, 263
    Ms = [301, 3, 4097, 264]
    X, Ds, states = case(K, N, Ms, 36, False)
    got = run_multi(cuda_device, X, Ds, states, step=2)
    for D, (W, m, v), g in zip(Ds, states, got):
        G = oracle.wgrad(X, D)
        check_adamw(g, adamw_ref(G, W, m, v, step=2, **vars(HP)), G, HP.lr, False)

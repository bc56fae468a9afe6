"""GPU parity at the workloads' full sizes, on sampled output rows.

Each test runs the fused call exactly as the benchmark does (same sizes, same
automatic kernel choice) and checks whole output rows of W and the state,
chosen to land in the first, last and interior tiles, element by element
against the fp64 oracle computed for those rows only.
"""
import numpy as np
import pytest
import torch

import oracle
import weight_grad_gemm_gb300 as fg
import workloads as wl
from parity_util import check_grad_from_m, check_state_bf16, check_state_f32, check_W, rms

pytestmark = pytest.mark.gpu


def sample_rows(N):
    rows = {0, 1, 127, 128, 255, 256, N // 2 - 1, N // 2, N - 257, N - 256, N - 2, N - 1}
    return sorted(r for r in rows if 0 <= r < N)


def host(t):
    return oracle.as_bits(t.cpu())


def state_host(t):
    t = t.cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def warm(N, M, dev, name, state_dtype=torch.float32, E=None):
    shape = (N, M) if E is None else (E, N, M)
    W = wl.randn(shape, wl.seed_of(name, "W"), device=dev, std=0.02)
    m = wl.randn(shape, wl.seed_of(name, "m"), device=dev, std=1e-3).to(state_dtype)
    v = (wl.randn(shape, wl.seed_of(name, "v"), device=dev, std=1e-3) ** 2).to(state_dtype)
    return W, m, v


def check_rows(W1, m1, v1, ref, G, lr, state_bf16, m0=None, beta1=None):
    # long contractions: the contract bounds, plus the gradient diagnostic
    if state_bf16:
        check_state_bf16(m1, ref["m_exact"], "m", diag=False)
        check_state_bf16(v1, ref["v_exact"], "v", diag=False)
    else:
        check_state_f32(m1, ref["m_exact"], "m", diag=False)
        check_state_f32(v1, ref["v_exact"], "v", diag=False)
        if m0 is not None and np.any(G):
            check_grad_from_m(m1, m0, G, beta1)
    check_W(W1, ref["W_exact"], G, lr, m_exact=ref["m_exact"])


def run_dense(wk, dev, state_dtype=torch.float32, step=4):
    """Steps 1 .. step-1 warm m, v from zero with the library on seeded inputs
    (the workloads' "warmed by prior steps" state); step `step` is checked
    against the oracle started from that state."""
    K, N, M = wk.K, wk.N, wk.M
    hp = wk.adam.f32()
    W = wl.randn((N, M), wl.seed_of(wk.name, "W"), device=dev, std=0.02)
    m = torch.zeros((N, M), dtype=state_dtype, device=dev)
    v = torch.zeros((N, M), dtype=state_dtype, device=dev)
    for t in range(1, step + 1):
        X = wl.activations(K, N, wl.seed_of(wk.name, "X", t), device=dev)
        D = wl.activations(K, M, wl.seed_of(wk.name, "dY", t), device=dev)
        if t < step:
            fg.forge_wgrad_adamw(X, D, W, m, v, lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2,
                                 eps=hp.eps, wd=hp.wd, step=t)
    rows = sample_rows(N)
    W0, m0, v0 = (state_host(t[rows]) for t in (W, m, v))
    fg.forge_wgrad_adamw(X, D, W, m, v, lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2, eps=hp.eps,
                         wd=hp.wd, step=step)
    torch.cuda.synchronize()
    assert fg.forge_get_device_status() == fg.FORGE_OK
    Xh, Dh = host(X), host(D)
    G = oracle.wgrad(Xh, Dh, rows=rows)
    ref = oracle.adamw(G, W0, m0, v0, step=step, **vars(hp))
    check_rows(state_host(W[rows]), state_host(m[rows]), state_host(v[rows]), ref, G, hp.lr,
               state_dtype == torch.bfloat16, m0=m0, beta1=hp.beta1)


def test_mlp_down_full_size(cuda_device):
    run_dense(wl.MLP_DOWN, cuda_device, step=4)


@pytest.mark.parametrize("state", ["f32", "bf16"])
@pytest.mark.parametrize("idx", [0, 1, 3], ids=["d_out4096", "d_out1024", "d_out4100"])
def test_attention_projections_full_size(cuda_device, idx, state):
    run_dense(wl.ATTN_PROJ[idx], cuda_device,
              torch.float32 if state == "f32" else torch.bfloat16, step=2)


@pytest.mark.parametrize("state", ["f32", "bf16"])
def test_attention_set_one_launch_full_size(cuda_device, state):
    """The four projections as the benchmark runs them: one multi-problem
    call over the shared X (K 16384, d_in 4096, d_out 4096/1024/1024/4100),
    step 1 warming m, v from zero, step 2 checked on sampled rows of every
    problem."""
    dev = cuda_device
    sd = torch.float32 if state == "f32" else torch.bfloat16
    wks = wl.ATTN_PROJ
    K, N = wks[0].K, wks[0].N
    hp = wks[0].adam.f32()
    Ws = [wl.randn((N, wk.M), wl.seed_of(wk.name, "W"), device=dev, std=0.02) for wk in wks]
    ms = [torch.zeros((N, wk.M), dtype=sd, device=dev) for wk in wks]
    vs = [torch.zeros((N, wk.M), dtype=sd, device=dev) for wk in wks]
    rows = sample_rows(N)
    for t in (1, 2):
        X = wl.activations(K, N, wl.seed_of("attn_set", "X", t), device=dev)
        Ds = [wl.activations(K, wk.M, wl.seed_of(wk.name, "dY", t), device=dev) for wk in wks]
        if t == 2:
            before = [tuple(state_host(a[rows]) for a in s3) for s3 in zip(Ws, ms, vs)]
        fg.forge_wgrad_adamw_multi(X, Ds, Ws, ms, vs, lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2,
                                   eps=hp.eps, wd=hp.wd, step=t)
    torch.cuda.synchronize()
    assert fg.forge_get_device_status() == fg.FORGE_OK
    Xh = host(X)
    for j, D in enumerate(Ds):
        W0, m0, v0 = before[j]
        G = oracle.wgrad(Xh, host(D), rows=rows)
        ref = oracle.adamw(G, W0, m0, v0, step=2, **vars(hp))
        check_rows(state_host(Ws[j][rows]), state_host(ms[j][rows]), state_host(vs[j][rows]),
                   ref, G, hp.lr, state == "bf16", m0=m0, beta1=hp.beta1)


@pytest.mark.parametrize("state", ["f32", "bf16"])
def test_moe_grouped_full_size(cuda_device, state):
    """8 experts of [14336, 4096]; step 2 of the routed workload, on which 4
    seeded experts receive no tokens (their m, v decay exactly by beta)."""
    wk = wl.MOE
    dev = cuda_device
    sdt = torch.float32 if state == "f32" else torch.bfloat16
    E, N, M = wk.experts, wk.N, wk.M
    step = 2
    zero = wl.moe_zero_experts(wl.seed_of(wk.name, "zero", step), E)
    counts = wl.zipf_top2_counts(wl.seed_of(wk.name, "route", step), tokens=16384, experts=E,
                                 zero_experts=zero)
    off = wl.offsets_from_counts(counts)
    T = int(off[-1])
    assert T == 32768 and all(counts[e] == 0 for e in zero)
    X = wl.activations(T, N, wl.seed_of(wk.name, "X", step), device=dev)
    D = wl.activations(T, M, wl.seed_of(wk.name, "dY", step), device=dev)
    hp = wk.adam.f32()
    # step 1 (all experts routed) warms the state from zero with the library
    W = wl.randn((E, N, M), wl.seed_of(wk.name, "W"), device=dev, std=0.02)
    m = torch.zeros((E, N, M), device=dev, dtype=sdt)
    v = torch.zeros((E, N, M), device=dev, dtype=sdt)
    c1 = wl.zipf_top2_counts(wl.seed_of(wk.name, "route", 1), tokens=16384, experts=E)
    off1 = torch.from_numpy(wl.offsets_from_counts(c1).astype(np.int32)).to(dev)
    fg.forge_grouped_wgrad_adamw(wl.activations(T, N, wl.seed_of(wk.name, "X", 1), device=dev),
                                 wl.activations(T, M, wl.seed_of(wk.name, "dY", 1), device=dev),
                                 W, m, v, off1, lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2,
                                 eps=hp.eps, wd=hp.wd, step=1)
    rows = sample_rows(N)[::2]
    W0, m0, v0 = (state_host(t[:, rows]) for t in (W, m, v))
    offd = torch.from_numpy(off.astype(np.int32)).to(dev)
    fg.forge_grouped_wgrad_adamw(X, D, W, m, v, offd, lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2,
                                 eps=hp.eps, wd=hp.wd, step=step)
    torch.cuda.synchronize()
    assert fg.forge_get_device_status() == fg.FORGE_OK
    Xh, Dh = host(X), host(D)
    W1, m1, v1 = (state_host(t[:, rows]) for t in (W, m, v))
    for e in range(E):
        G = oracle.wgrad(Xh, Dh, rows=rows, k_range=(int(off[e]), int(off[e + 1])))
        ref = oracle.adamw(G, W0[e], m0[e], v0[e], step=step, **vars(hp))
        check_rows(W1[e], m1[e], v1[e], ref, G, hp.lr, state == "bf16", m0=m0[e],
                   beta1=hp.beta1)
        if counts[e] == 0 and state == "f32":
            # g = 0: m' = RN(b1 m), v' = RN(b2 v) exactly, as the oracle rounds
            # them (with bf16 state the fp32 product is rounded again to bf16,
            # which the band check above covers)
            assert np.array_equal(m1[e], ref["m"]) and np.array_equal(v1[e], ref["v"])


@pytest.mark.parametrize("opt", ["adamw", "sgdm"])
def test_fp8_full_size(cuda_device, opt):
    wk = wl.FP8
    dev = cuda_device
    K, N, M = wk.K, wk.N, wk.M
    X, sx = wl.quantize_e4m3(wl.with_outliers((K, N), wl.seed_of(wk.name, "X"), device=dev))
    D, sy = wl.quantize_e4m3(wl.with_outliers((K, M), wl.seed_of(wk.name, "dY"), device=dev))
    sc = torch.tensor([sx, sy], dtype=torch.float32, device=dev)
    rows = sample_rows(N)[::2]
    Xh, Dh = host(X), host(D)
    if opt == "adamw":
        hp = wk.adam.f32()
        W, m, v = warm(N, M, dev, wk.name)
        m.zero_()
        v.zero_()  # the first AdamW step starts from zero moments
        W0, m0, v0 = (state_host(t[rows]) for t in (W, m, v))
        fg.forge_wgrad_adamw(X, D, W, m, v, lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2, eps=hp.eps,
                             wd=hp.wd, step=1, scales=sc)
        torch.cuda.synchronize()
        G = oracle.wgrad(Xh, Dh, rows=rows, scales=(sx, sy))
        ref = oracle.adamw(G, W0, m0, v0, step=1, **vars(hp))
        check_rows(state_host(W[rows]), state_host(m[rows]), state_host(v[rows]), ref, G, hp.lr,
                   False, m0=m0, beta1=hp.beta1)
    else:
        hp = wl.FP8_SGD.f32()
        W, buf, _ = warm(N, M, dev, wk.name)
        W0, b0 = state_host(W[rows]), state_host(buf[rows])
        fg.forge_wgrad_sgdm(X, D, W, buf, lr=hp.lr, momentum=hp.momentum, wd=hp.wd, scales=sc)
        torch.cuda.synchronize()
        G = oracle.wgrad(Xh, Dh, rows=rows, scales=(sx, sy))
        ref = oracle.sgdm(G, W0, b0, lr=hp.lr, momentum=hp.momentum, wd=hp.wd)
        check_state_f32(state_host(buf[rows]), ref["buf_exact"], "buf", diag=False)
        err = np.max(np.abs(state_host(W[rows]).astype(np.float64) - ref["W_exact"]))
        assert err <= 2e-3 * hp.lr * rms(ref["buf_exact"]) + 1e-7
    assert fg.forge_get_device_status() == fg.FORGE_OK

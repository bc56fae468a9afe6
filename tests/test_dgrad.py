"""GPU parity of the input gradient dX = dY W^T and of the ordered backward
step (dX from the weights before the update, then the fused update)."""
import numpy as np
import pytest
import torch

import oracle
import weight_grad_gemm_gb300 as fg
import workloads as wl

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01)


def bf16_ulp(x):
    """Spacing of bf16 values at |x| (8 significant bits)."""
    a = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def check_dx(got_bf16, exact):
    """Every element within one bf16 step of the exact value (the output
    rounding of an fp32 sum), plus 1e-5 rms for cancellation."""
    got = oracle.decode(oracle.as_bits(got_bf16.cpu()))
    exact = np.asarray(exact, np.float64)
    rms = float(np.sqrt(np.mean(exact ** 2))) if exact.size else 0.0
    err = np.abs(got - exact)
    bound = bf16_ulp(exact) + 1e-5 * rms
    bad = np.nonzero(err > bound)
    assert bad[0].size == 0, (bad[0][:5], got[bad][:5], exact[bad][:5])


@pytest.fixture(params=["single", "pair"])
def dgrad_form(request, monkeypatch):
    """Run on the one-CTA kernel and on CTA pairs."""
    monkeypatch.setenv("FORGE_DGRAD_KERNEL", request.param)
    return request.param


def inputs(K, N, M, seed, dev):
    D = wl.activations(K, M, wl.seed_of("dg-dY", seed, K, M), device=dev)
    Wb = wl.randn((N, M), wl.seed_of("dg-W", seed, N, M), device=dev, std=0.02).to(torch.bfloat16)
    return D, Wb


@pytest.mark.parametrize("K,N,M", [(200, 520, 296), (1, 8, 8), (129, 257, 64),
                                   (1000, 1032, 648), (300, 250, 4104), (64, 256, 128)])
def test_dgrad_matches_oracle(cuda_device, dgrad_form, K, N, M):
    D, Wb = inputs(K, N, M, 1, cuda_device)
    dX = torch.full((K, N), float("nan"), dtype=torch.bfloat16, device=cuda_device)
    fg.forge_dgrad(D, Wb, dX)
    torch.cuda.synchronize()
    assert fg.forge_get_device_status() == fg.FORGE_OK
    check_dx(dX, oracle.dgrad(oracle.as_bits(D.cpu()), oracle.as_bits(Wb.cpu())))


def test_dgrad_no_tokens(cuda_device):
    dev = cuda_device
    D, Wb = inputs(0, 64, 64, 2, dev)
    dX = torch.empty((0, 64), dtype=torch.bfloat16, device=dev)
    fg.forge_dgrad(D, Wb, dX)
    torch.cuda.synchronize()


# d_out (the contraction here) of any width: rows of 8200, 602, 6 and 8194
# bytes, which TMA cannot read, are staged into 16-byte rows first
@pytest.mark.parametrize("K,N,M", [(160, 264, 4100), (130, 136, 301), (70, 300, 3),
                                   (257, 520, 4097)])
def test_dgrad_any_row_width(cuda_device, dgrad_form, K, N, M):
    D, Wb = inputs(K, N, M, 3, cuda_device)
    dX = torch.full((K, N), float("nan"), dtype=torch.bfloat16, device=cuda_device)
    fg.forge_dgrad(D, Wb, dX)
    torch.cuda.synchronize()
    assert fg.forge_get_device_status() == fg.FORGE_OK
    check_dx(dX, oracle.dgrad(oracle.as_bits(D.cpu()), oracle.as_bits(Wb.cpu())))


def test_dgrad_offset_bases(cuda_device):
    """dY and Wb starting 2 bytes into their allocations (aligned rows)."""
    dev = cuda_device
    K, N, M = 150, 264, 392
    D, Wb = inputs(K, N, M, 4, dev)
    db = torch.empty(K * M + 1, dtype=torch.bfloat16, device=dev)
    wbb = torch.empty(N * M + 1, dtype=torch.bfloat16, device=dev)
    Do, Wo = db[1:].view(K, M), wbb[1:].view(N, M)
    Do.copy_(D)
    Wo.copy_(Wb)
    dX = torch.empty((K, N), dtype=torch.bfloat16, device=dev)
    fg.forge_dgrad(Do, Wo, dX)
    torch.cuda.synchronize()
    check_dx(dX, oracle.dgrad(oracle.as_bits(D.cpu()), oracle.as_bits(Wb.cpu())))


@pytest.mark.parametrize("given_copy", [True, False], ids=["Wb", "rounded"])
def test_backward_odd_width(cuda_device, given_copy):
    """The ordered step on d_out 301: dX from the staged (or freshly rounded,
    padded) weight copy, then the fused update, equal bit for bit to the two
    calls made separately."""
    dev = cuda_device
    K, N, M = 120, 264, 301
    X = wl.activations(K, N, wl.seed_of("bw-odd", "X"), device=dev)
    D = wl.activations(K, M, wl.seed_of("bw-odd", "dY"), device=dev)
    W = wl.randn((N, M), wl.seed_of("bw-odd", "W"), device=dev, std=0.02)
    m = torch.zeros_like(W)
    v = torch.zeros_like(W)
    Wb = W.to(torch.bfloat16)
    W2, m2, v2 = W.clone(), m.clone(), v.clone()
    dX = torch.empty((K, N), dtype=torch.bfloat16, device=dev)
    dX2 = torch.empty_like(dX)
    fg.forge_backward_adamw(X, D, W, m, v, dX, Wb=Wb if given_copy else None, step=1, **HP)
    fg.forge_dgrad(D, Wb, dX2)
    fg.forge_wgrad_adamw(X, D, W2, m2, v2, step=1, **HP)
    torch.cuda.synchronize()
    assert torch.equal(dX.view(torch.int16), dX2.view(torch.int16))
    for a, b in ((W, W2), (m, m2), (v, v2)):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    check_dx(dX, oracle.dgrad(oracle.as_bits(D.cpu()), oracle.as_bits(Wb.cpu())))


def test_dgrad_full_size_sampled_rows(cuda_device, dgrad_form):
    wk = wl.MLP_DOWN
    K, N, M = wk.K, wk.N, wk.M
    D, Wb = inputs(K, N, M, 4, cuda_device)
    dX = torch.empty((K, N), dtype=torch.bfloat16, device=cuda_device)
    fg.forge_dgrad(D, Wb, dX)
    torch.cuda.synchronize()
    rows = [0, 127, 128, 255, 256, K // 2, K - 1]
    exact = oracle.dgrad(oracle.as_bits(D.cpu()), oracle.as_bits(Wb.cpu()), rows=rows)
    check_dx(dX[rows], exact)


@pytest.mark.parametrize("given_copy", [True, False], ids=["Wb", "rounded"])
def test_backward_reads_weights_before_the_update(cuda_device, dgrad_form, given_copy):
    """forge_backward_adamw = forge_dgrad on the pre-update bf16 weights, then
    forge_wgrad_adamw: both halves bit for bit."""
    dev = cuda_device
    K, N, M = 384, 520, 296
    X = wl.activations(K, N, wl.seed_of("bw-X"), device=dev)
    D = wl.activations(K, M, wl.seed_of("bw-dY"), device=dev)
    W = wl.randn((N, M), wl.seed_of("bw-W"), device=dev, std=0.02)
    m = wl.randn((N, M), wl.seed_of("bw-m"), device=dev, std=1e-3)
    v = wl.randn((N, M), wl.seed_of("bw-v"), device=dev, std=1e-3) ** 2
    Wb = W.to(torch.bfloat16)  # nearest even, as the library rounds
    W1, m1, v1 = W.clone(), m.clone(), v.clone()
    dX1 = torch.empty((K, N), dtype=torch.bfloat16, device=dev)
    fg.forge_backward_adamw(X, D, W1, m1, v1, dX1, Wb=Wb if given_copy else None, step=3, **HP)
    W2, m2, v2 = W.clone(), m.clone(), v.clone()
    dX2 = torch.empty((K, N), dtype=torch.bfloat16, device=dev)
    fg.forge_dgrad(D, Wb, dX2)
    fg.forge_wgrad_adamw(X, D, W2, m2, v2, step=3, **HP)
    torch.cuda.synchronize()
    assert fg.forge_get_device_status() == fg.FORGE_OK
    assert torch.equal(dX1.view(torch.int16), dX2.view(torch.int16))
    for a, b in ((W1, W2), (m1, m2), (v1, v2)):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert not torch.equal(W1, W)  # the update did happen
    check_dx(dX1, oracle.dgrad(oracle.as_bits(D.cpu()), oracle.as_bits(Wb.cpu())))

"""GPU tests of forge_wgrad_adamw_noalloc, the entry point that stages
misaligned operands into the library's fixed per-device buffer instead of
allocating.  Its results must equal forge_wgrad_adamw's bit for bit, call
after call, and a call whose staging copy would not fit must be refused
before anything is written."""
import numpy as np
import pytest
import torch

import weight_grad_gemm_gb300 as fg
import workloads as wl

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01)


def state(N, M, seed, dev):
    W = wl.randn((N, M), wl.seed_of("na-W", seed), device=dev, std=0.02)
    m = wl.randn((N, M), wl.seed_of("na-m", seed), device=dev, std=1e-3)
    v = wl.randn((N, M), wl.seed_of("na-v", seed), device=dev, std=1e-3) ** 2
    return W, m, v


def bits(t):
    return t.view(torch.int32).cpu().numpy()


def test_no_alloc_matches_allocating_entry_call_after_call(cuda_device, monkeypatch):
    """Consecutive calls on two layers whose X rows (1044 bytes) and dY rows
    (8200, then 2004 bytes) both need staging: each call overwrites part of
    what the previous one left in the buffer with another layout, and layer
    a's second step starts from the state its first step wrote."""
    monkeypatch.delenv("FORGE_MISALIGNED", raising=False)
    dev = cuda_device
    layers = {"a": (522, 4100), "b": (522, 1002)}
    ref = {k: state(N, M, i, dev) for i, (k, (N, M)) in enumerate(layers.items())}
    got = {k: tuple(t.clone() for t in ref[k]) for k in layers}
    for step, name, K in ((1, "a", 300), (1, "b", 200), (2, "a", 300)):
        N, M = layers[name]
        X = wl.activations(K, N, wl.seed_of("na-X", name, step), device=dev)
        D = wl.activations(K, M, wl.seed_of("na-dY", name, step), device=dev)
        fg.forge_wgrad_adamw(X, D, *ref[name], step=step, **HP)
        fg.forge_wgrad_adamw_noalloc(X, D, *got[name], step=step, **HP)
        torch.cuda.synchronize()
        assert fg.forge_get_device_status() == fg.FORGE_OK
        for a, b in zip(ref[name], got[name]):
            assert np.array_equal(bits(a), bits(b))
        assert torch.isfinite(got[name][0]).all()


def test_no_alloc_aligned_operands_match(cuda_device):
    dev = cuda_device
    K, N, M = 256, 520, 264
    X = wl.activations(K, N, wl.seed_of("na-X", 9), device=dev)
    D = wl.activations(K, M, wl.seed_of("na-dY", 9), device=dev)
    W1, m1, v1 = state(N, M, 9, dev)
    W2, m2, v2 = W1.clone(), m1.clone(), v1.clone()
    fg.forge_wgrad_adamw(X, D, W1, m1, v1, step=3, **HP)
    fg.forge_wgrad_adamw_noalloc(X, D, W2, m2, v2, step=3, **HP)
    torch.cuda.synchronize()
    for a, b in ((W1, W2), (m1, m2), (v1, v2)):
        assert np.array_equal(bits(a), bits(b))


def test_no_alloc_refuses_staging_larger_than_its_buffer(cuda_device, monkeypatch):
    """33000 rows of 8200 bytes need 33000 x 8208 bytes > 256 MiB of staging."""
    monkeypatch.delenv("FORGE_MISALIGNED", raising=False)
    dev = cuda_device
    K, N, M = 33000, 8, 4100
    X = torch.zeros((K, N), dtype=torch.bfloat16, device=dev)
    D = torch.zeros((K, M), dtype=torch.bfloat16, device=dev)
    W, m, v = state(N, M, 3, dev)
    W0 = W.clone()
    with pytest.raises(fg.ForgeError) as e:
        fg.forge_wgrad_adamw_noalloc(X, D, W, m, v, step=1, **HP)
    assert e.value.status == fg.FORGE_ERR_SCRATCH_TOO_SMALL
    torch.cuda.synchronize()
    assert torch.equal(W, W0)
    # the allocating entry point takes the same call
    fg.forge_wgrad_adamw(X, D, W, m, v, step=1, **HP)
    torch.cuda.synchronize()
    assert fg.forge_get_device_status() == fg.FORGE_OK


# X rows of 1003 bf16 (2006 bytes) and dY rows of 1001 (2002 bytes) both
# stage into 2016-byte rows: 4032 bytes per token row.  Either operand alone
# fits the 256 MiB buffer at these row counts; only their sum decides.
BOTH_N, BOTH_M = 1003, 1001
ROWS_UNDER = (256 << 20) // 4032   # 66576 rows: 1024 bytes to spare
ROWS_OVER = ROWS_UNDER + 1


def test_no_alloc_refuses_when_both_staged_operands_together_overflow(cuda_device, monkeypatch):
    monkeypatch.delenv("FORGE_MISALIGNED", raising=False)
    dev = cuda_device
    K = ROWS_OVER
    X = torch.zeros((K, BOTH_N), dtype=torch.bfloat16, device=dev)
    D = torch.zeros((K, BOTH_M), dtype=torch.bfloat16, device=dev)
    W, m, v = state(BOTH_N, BOTH_M, 5, dev)
    W0, m0, v0 = W.clone(), m.clone(), v.clone()
    with pytest.raises(fg.ForgeError) as e:
        fg.forge_wgrad_adamw_noalloc(X, D, W, m, v, step=1, **HP)
    assert e.value.status == fg.FORGE_ERR_SCRATCH_TOO_SMALL
    torch.cuda.synchronize()
    for a, b in ((W, W0), (m, m0), (v, v0)):
        assert torch.equal(a, b)


def test_no_alloc_both_staged_operands_just_under_the_limit(cuda_device, monkeypatch):
    monkeypatch.delenv("FORGE_MISALIGNED", raising=False)
    dev = cuda_device
    K = ROWS_UNDER
    X = wl.activations(K, BOTH_N, wl.seed_of("na-X", "both"), device=dev)
    D = wl.activations(K, BOTH_M, wl.seed_of("na-dY", "both"), device=dev)
    W1, m1, v1 = state(BOTH_N, BOTH_M, 6, dev)
    W2, m2, v2 = W1.clone(), m1.clone(), v1.clone()
    fg.forge_wgrad_adamw(X, D, W1, m1, v1, step=2, **HP)
    fg.forge_wgrad_adamw_noalloc(X, D, W2, m2, v2, step=2, **HP)
    torch.cuda.synchronize()
    assert fg.forge_get_device_status() == fg.FORGE_OK
    for a, b in ((W1, W2), (m1, m2), (v1, v2)):
        assert np.array_equal(bits(a), bits(b))


def test_no_alloc_loader_mode_still_stages_odd_rows(cuda_device, monkeypatch):
    """With FORGE_MISALIGNED=loader, X rows of 1044 bytes go to the kernel's
    cp.async loader, while dY rows of 602 bytes (not a multiple of 4) cannot
    and are staged into the fixed buffer: both entry points agree bit for
    bit, call after call."""
    monkeypatch.setenv("FORGE_MISALIGNED", "loader")
    dev = cuda_device
    K, N, M = 300, 522, 301
    ref = state(N, M, 7, dev)
    got = tuple(t.clone() for t in ref)
    for step in (1, 2):
        X = wl.activations(K, N, wl.seed_of("na-ld-X", step), device=dev)
        D = wl.activations(K, M, wl.seed_of("na-ld-dY", step), device=dev)
        fg.forge_wgrad_adamw(X, D, *ref, step=step, **HP)
        fg.forge_wgrad_adamw_noalloc(X, D, *got, step=step, **HP)
        torch.cuda.synchronize()
        assert fg.forge_get_device_status() == fg.FORGE_OK
        for a, b in zip(ref, got):
            assert np.array_equal(bits(a), bits(b))

"""The fused calls inside a CUDA graph: captured once, replayed, they give
the same bits as the same calls made eagerly (launch configuration, tensor
maps and the staging copy's stream-ordered allocation all capture)."""
import pytest
import torch

import weight_grad_gemm_gb300 as fg
import workloads as wl

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01)


def state(N, M, dev, seed):
    W = wl.randn((N, M), wl.seed_of("g-W", seed), device=dev, std=0.02)
    m = wl.randn((N, M), wl.seed_of("g-m", seed), device=dev, std=1e-3)
    v = wl.randn((N, M), wl.seed_of("g-v", seed), device=dev, std=1e-3) ** 2
    return W, m, v


@pytest.mark.parametrize("M", [296, 4100], ids=["aligned", "staged"])
def test_fused_step_replays_from_a_graph(cuda_device, M):
    dev = cuda_device
    K, N = 320, 520
    X = wl.activations(K, N, wl.seed_of("g-X", M), device=dev)
    D = wl.activations(K, M, wl.seed_of("g-dY", M), device=dev)
    W, m, v = state(N, M, dev, M)
    We, me, ve = W.clone(), m.clone(), v.clone()
    for step in (1, 2):
        fg.forge_wgrad_adamw(X, D, We, me, ve, step=step, **HP)
    torch.cuda.synchronize()

    Wg, mg, vg = W.clone(), m.clone(), v.clone()
    fg.forge_wgrad_adamw(X, D, Wg.clone(), mg.clone(), vg.clone(), step=1, **HP)  # set-up outside
    torch.cuda.synchronize()
    steps = []
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for step in (1, 2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                fg.forge_wgrad_adamw(X, D, Wg, mg, vg, step=step, **HP)
            steps.append(g)
    torch.cuda.synchronize()
    # capture records without executing: the state is still the initial one
    assert torch.equal(Wg, W)
    for g in steps:
        g.replay()
    torch.cuda.synchronize()
    assert fg.forge_get_device_status() == fg.FORGE_OK
    for a, b in ((We, Wg), (me, mg), (ve, vg)):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_no_alloc_staged_step_replays_from_a_graph(cuda_device):
    """The no-allocation entry on its staging path (X rows of 1044 bytes, dY
    rows of 8200): a first call outside capture sets the device up, then the
    captured steps replay to the bits of the same calls made eagerly."""
    dev = cuda_device
    K, N, M = 4100, 522, 4100
    X = wl.activations(K, N, wl.seed_of("gn-X"), device=dev)
    D = wl.activations(K, M, wl.seed_of("gn-dY"), device=dev)
    W, m, v = state(N, M, dev, 7)
    We, me, ve = W.clone(), m.clone(), v.clone()
    for step in (1, 2):
        fg.forge_wgrad_adamw_noalloc(X, D, We, me, ve, step=step, **HP)
    torch.cuda.synchronize()
    Wg, mg, vg = W.clone(), m.clone(), v.clone()
    fg.forge_wgrad_adamw_noalloc(X, D, Wg.clone(), mg.clone(), vg.clone(), step=1, **HP)
    torch.cuda.synchronize()
    graphs = []
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for step in (1, 2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                fg.forge_wgrad_adamw_noalloc(X, D, Wg, mg, vg, step=step, **HP)
            graphs.append(g)
    torch.cuda.synchronize()
    assert torch.equal(Wg, W)
    for g in graphs:
        g.replay()
    torch.cuda.synchronize()
    assert fg.forge_get_device_status() == fg.FORGE_OK
    for a, b in ((We, Wg), (me, mg), (ve, vg)):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))

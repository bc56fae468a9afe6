"""The owner's optimizer step behind a reduce-scatter (data parallelism with
sharded optimizer state).

CPU (no GPU): the ownership partition gives every tile row exactly one
owner, and on 2 and 3 gloo ranks the reduce-scatter of the ranks' partial
gradients followed by each owner's AdamW on its shard reproduces, row for
row, the oracle's step over all tokens at once (the oracle stands in for the
kernels here; the collective is the same call the GPU ranks make on NCCL).

GPU: forge_owner_adamw / forge_owner_sgdm against the oracle, on a gradient
summed from two token shards (two ranks emulated on one GPU, one after the
other: nothing waits on anything), and bit for bit against the fused call
when fed the fused kernel's own dW.
"""
import multiprocessing as mp
import os
import socket

import numpy as np
import pytest

import oracle
from weight_grad_gemm_gb300 import owner

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01)


# ------------------------------------------------------------------ partition (CPU)

@pytest.mark.parametrize("N", [1, 255, 256, 257, 600, 4100, 14336])
@pytest.mark.parametrize("world", [1, 2, 3, 7, 8, 64])
def test_every_tile_row_has_exactly_one_owner(N, world):
    ranges = owner.owner_ranges(N, world)
    assert len(ranges) == world
    assert ranges[0][0] == 0 and ranges[-1][1] == N
    for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
        assert a1 == b0 and a0 <= a1  # contiguous, ordered, disjoint
    tiles = -(-N // owner.TILE_ROWS)
    counts = [0] * world
    for tn in range(tiles):
        counts[owner.tile_owner(tn, ranges)] += 1
    assert sum(counts) == tiles
    assert max(counts) - min(counts) <= 1  # balanced to one tile row
    for r0, r1 in ranges:  # ranges start on tile-row boundaries
        assert r0 % owner.TILE_ROWS == 0 or r0 == N
    with pytest.raises(ValueError):
        owner.tile_owner(tiles, ranges)


# ------------------------------------------------------------------ gloo ranks (CPU)

def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def gloo_case(K, N, M):
    """Seeded inputs and state for the multi-rank case (every rank builds the
    same ones)."""
    import workloads as wl
    X = oracle.as_bits(wl.activations(K, N, wl.seed_of("own-X", K, N)))
    D = oracle.as_bits(wl.activations(K, M, wl.seed_of("own-dY", K, M)))
    rng = np.random.default_rng(61)
    W = (rng.standard_normal((N, M)) * 0.02).astype(np.float32)
    m = (rng.standard_normal((N, M)) * 1e-3).astype(np.float32)
    v = (rng.random((N, M)) * 1e-5).astype(np.float32)
    return X, D, W, m, v


def rank_main(rank, world, port, K, N, M, cuts, out):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        X, D, W, m, v = gloo_case(K, N, M)
        ranges = owner.owner_ranges(N, world)
        # this rank's tokens: an uneven slice of the batch
        partial = oracle.wgrad(X, D, k_range=(cuts[rank], cuts[rank + 1]))
        shard = owner.reduce_scatter_rows(torch.from_numpy(partial), ranges).numpy()
        r0, r1 = ranges[rank]
        upd = oracle.adamw(shard, W[r0:r1], m[r0:r1], v[r0:r1], step=3, **HP)
        out.put((rank, r0, r1, shard, upd["W"], upd["m"], upd["v"]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,N", [(2, 600), (3, 600), (2, 512)])
def test_reduce_scatter_then_owner_step_matches_the_whole_batch(world, N):
    K, M = 90, 130
    cuts = [0, 37, 90] if world == 2 else [0, 20, 21, 90]  # one rank holds a single token
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=rank_main, args=(r, world, port, K, N, M, cuts, out))
             for r in range(world)]
    for p in procs:
        p.start()
    got = sorted((out.get(timeout=180) for _ in procs), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    X, D, W, m, v = gloo_case(K, N, M)
    G = oracle.wgrad(X, D)
    ref = oracle.adamw(G, W, m, v, step=3, **HP)
    covered = np.zeros(N, bool)
    for rank, r0, r1, shard, Ws, ms, vs in got:
        assert not covered[r0:r1].any()
        covered[r0:r1] = True
        # the sum of the partials equals the whole contraction up to fp64 rounding
        scale = np.abs(G[r0:r1]).max() if r1 > r0 else 1.0
        assert np.allclose(shard, G[r0:r1], rtol=0, atol=1e-12 * scale)
        # the owner's step on its shard is the whole-batch step on those rows;
        # stored fp32 state may differ where the fp64 sums round differently
        for a, b in ((Ws, ref["W"][r0:r1]), (ms, ref["m"][r0:r1]), (vs, ref["v"][r0:r1])):
            diff = np.abs(a.astype(np.float64) - b.astype(np.float64))
            assert (diff <= 2 * np.spacing(np.abs(b).astype(np.float32)).astype(np.float64)).all()
    assert covered.all()


# ------------------------------------------------------------------ the kernel (GPU)

def _dev_inputs(dev, K, N, M, seed, state_bf16):
    import torch
    from test_parity import bf16_inputs, dev_state, warm_state
    X, D = bf16_inputs(K, N, M, seed)
    W, m, v = warm_state(N, M, seed + 1, state_bf16)
    return X, D, W, m, v, [dev_state(a, dev) for a in (W, m, v)], torch


@pytest.mark.gpu
@pytest.mark.parametrize("state_bf16", [False, True], ids=["f32state", "bf16state"])
@pytest.mark.parametrize("K,N,M", [(200, 520, 296), (150, 263, 301), (64, 1, 3)])
def test_owner_adamw_on_summed_shards_matches_oracle(cuda_device, K, N, M, state_bf16):
    """Two ranks' token halves, reduced by a sum (the collective's job), each
    owner updating its row range: every row matches the oracle's step on the
    whole batch."""
    import weight_grad_gemm_gb300 as fg
    from test_parity import HP as PHP, adamw_ref, check_adamw, host_state
    dev = cuda_device
    X, D, W, m, v, (Wd, md, vd), torch = _dev_inputs(dev, K, N, M, 62, state_bf16)
    Xd, Dd = X.to(dev), D.to(dev)
    half = K // 2
    parts = []
    for a, b in ((0, half), (half, K)):
        g = torch.empty((N, M), device=dev)
        fg.forge_wgrad_only(Xd[a:b].contiguous(), Dd[a:b].contiguous(), g)
        parts.append(g)
    Gsum = parts[0] + parts[1]
    for r0, r1 in owner.owner_ranges(N, 2, unit=128):
        if r1 > r0:
            fg.forge_owner_adamw(Gsum[r0:r1], Wd[r0:r1], md[r0:r1], vd[r0:r1], lr=PHP.lr,
                                 beta1=PHP.beta1, beta2=PHP.beta2, eps=PHP.eps, wd=PHP.wd, step=4)
    torch.cuda.synchronize()
    G = oracle.wgrad(X, D)
    ref = adamw_ref(G, W, m, v, step=4, **vars(PHP))
    check_adamw((host_state(Wd), host_state(md), host_state(vd)), ref, G, PHP.lr, state_bf16)


@pytest.mark.gpu
@pytest.mark.parametrize("state_bf16", [False, True], ids=["f32state", "bf16state"])
@pytest.mark.parametrize("kind", ["bf16", "e4m3"])
def test_owner_step_on_the_fused_kernels_dw_is_bitwise_the_fused_call(cuda_device, kind,
                                                                      state_bf16):
    import torch

    import weight_grad_gemm_gb300 as fg
    from test_parity import (HP as PHP, bf16_inputs, dev_state, e4m3_inputs, scales_dev,
                             warm_state)
    dev = cuda_device
    K, N, M = 300, 520, 1032
    if kind == "bf16":
        X, D = bf16_inputs(K, N, M, 63)
        sc = None
    else:
        X, D, s = e4m3_inputs(K, N, M, 63)
        sc = scales_dev(s, dev)
    W, m, v = warm_state(N, M, 64, state_bf16)
    Xd, Dd = X.to(dev), D.to(dev)
    fused = [dev_state(a, dev) for a in (W, m, v)]
    fg.forge_wgrad_adamw(Xd, Dd, *fused, step=2, scales=sc, **vars(PHP))
    G = torch.empty((N, M), device=dev)
    fg.forge_wgrad_only(Xd, Dd, G, scales=sc)
    own = [dev_state(a, dev) for a in (W, m, v)]
    fg.forge_owner_adamw(G, *own, step=2, **vars(PHP))
    torch.cuda.synchronize()
    for a, b in zip(fused, own):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))


@pytest.mark.gpu
def test_owner_sgdm_bitwise_the_fused_call_and_edge_cases(cuda_device):
    import torch

    import weight_grad_gemm_gb300 as fg
    from test_parity import bf16_inputs, dev_state, warm_state
    dev = cuda_device
    K, N, M = 200, 264, 392
    X, D = bf16_inputs(K, N, M, 65)
    W, buf, _ = warm_state(N, M, 66)
    Xd, Dd = X.to(dev), D.to(dev)
    hp = dict(lr=1e-2, momentum=0.9, wd=0.05)
    fused = [dev_state(a, dev) for a in (W, buf)]
    fg.forge_wgrad_sgdm(Xd, Dd, *fused, **hp)
    G = torch.empty((N, M), device=dev)
    fg.forge_wgrad_only(Xd, Dd, G)
    own = [dev_state(a, dev) for a in (W, buf)]
    fg.forge_owner_sgdm(G, *own, **hp)
    # 999 elements: a gradient view one element past a 16-byte boundary takes
    # the scalar path, an aligned copy of it the vector path and a 3-element
    # tail; both must give the same bits
    Gs = G.reshape(-1)[1:1000]
    Ws, bs = own[0].reshape(-1)[1:1000].clone(), own[1].reshape(-1)[1:1000].clone()
    Wv, bv = Ws.clone(), bs.clone()
    fg.forge_owner_sgdm(Gs, Ws, bs, **hp)
    fg.forge_owner_sgdm(Gs.clone(), Wv, bv, **hp)
    torch.cuda.synchronize()
    for a, b in zip(fused, own):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert torch.equal(Ws.view(torch.int32), Wv.view(torch.int32))
    assert torch.equal(bs.view(torch.int32), bv.view(torch.int32))
    # n = 0 is a no-op; host memory is refused
    L = fg.lib()
    assert L.forge_owner_adamw(None, None, None, None, 0, fg.FORGE_F32, 1e-3, 0.9, 0.999, 1e-8,
                               0.0, 1, None) == fg.FORGE_OK
    host = np.zeros(16, np.float32)
    assert L.forge_owner_adamw(host.ctypes.data, own[0].data_ptr(), own[1].data_ptr(),
                               own[1].data_ptr(), 16, fg.FORGE_F32, 1e-3, 0.9, 0.999, 1e-8, 0.0,
                               1, None) == fg.FORGE_ERR_INVALID_ARG


@pytest.mark.gpu
def test_owner_step_full_size_mlp_shapes_bitwise(cuda_device):
    """The MLP down-projection shapes the owner workload benchmarks (K 8192,
    d_in 14336, d_out 4096, warm fp32 state): owner(dW) equals the fused step
    on every element, the shard split into two owners' row ranges."""
    import torch

    import weight_grad_gemm_gb300 as fg
    import workloads as wl
    dev = cuda_device
    wk = wl.MLP_DOWN
    K, N, M = wk.K, wk.N, wk.M
    X = wl.activations(K, N, wl.seed_of("own-full", "X"), device=dev)
    D = wl.activations(K, M, wl.seed_of("own-full", "dY"), device=dev)
    W = wl.randn((N, M), wl.seed_of("own-full", "W"), device=dev, std=0.02)
    m = wl.randn((N, M), wl.seed_of("own-full", "m"), device=dev, std=1e-3)
    v = wl.randn((N, M), wl.seed_of("own-full", "v"), device=dev, std=1e-3) ** 2
    hp = vars(wk.adam.f32())
    fused = [t.clone() for t in (W, m, v)]
    fg.forge_wgrad_adamw(X, D, *fused, step=4, **hp)
    G = torch.empty((N, M), device=dev)
    fg.forge_wgrad_only(X, D, G)
    own = [t.clone() for t in (W, m, v)]
    for r0, r1 in owner.owner_ranges(N, 2):
        fg.forge_owner_adamw(G[r0:r1], *(t[r0:r1] for t in own), step=4, **hp)
    torch.cuda.synchronize()
    assert fg.forge_get_device_status() == fg.FORGE_OK
    for a, b in zip(fused, own):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.gpu
@pytest.mark.parametrize("opt", ["adamw", "sgdm"])
def test_owner_step_through_nccl_one_rank(cuda_device, opt):
    """The user-facing step (partial dW, NCCL reduce-scatter, owner update)
    on a one-rank NCCL group: the collective is then a copy, and the step
    must equal the fused call bit for bit."""
    import torch
    import torch.distributed as dist

    import weight_grad_gemm_gb300 as fg
    from test_parity import bf16_inputs, dev_state, warm_state
    dev = cuda_device
    K, N, M = 200, 520, 392
    X, D = bf16_inputs(K, N, M, 66)
    W, m, v = warm_state(N, M, 67)
    Xd, Dd = X.to(dev), D.to(dev)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(free_port()))
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=dev)
    try:
        ranges = owner.owner_ranges(N, 1)
        fused = [dev_state(a, dev) for a in (W, m, v)]
        own = [dev_state(a, dev) for a in (W, m, v)]
        if opt == "adamw":
            hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01)
            fg.forge_wgrad_adamw(Xd, Dd, *fused, step=2, **hp)
            owner.owner_adamw_step(Xd, Dd, *own, ranges, step=2, **hp)
        else:
            hp = dict(lr=1e-2, momentum=0.9, wd=0.05)
            fg.forge_wgrad_sgdm(Xd, Dd, fused[0], fused[1], **hp)
            owner.owner_sgdm_step(Xd, Dd, own[0], own[1], ranges, **hp)
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    n = 3 if opt == "adamw" else 2
    for a, b in zip(fused[:n], own[:n]):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))

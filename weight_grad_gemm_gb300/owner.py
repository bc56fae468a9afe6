"""Owner partition behind a reduce-scatter: data parallelism with the
optimizer state sharded across ranks (ZeRO-2 style).

Each rank holds its own tokens, so its weight gradient is a partial sum.  The
ranks' partials are summed by a reduce-scatter that delivers every output
tile to exactly one owner, which alone applies the optimizer step (FORGE
assessment PR, tessera#565, "Math verified, not asserted", P3: the owner of a
tile is unambiguous under a reduce-scatter).  Ownership is by tile rows of
the fused kernel: the ceil(N / 256) d_in tile rows of W [N, M] are dealt out
as contiguous, balanced runs, so a rank's shard is one contiguous row range,
i.e. one flat range of the row-major weight, and a tile (tn, tm) belongs to
the owner of its row tn whatever tm is.

The step on rank r:
    1. partial dW over its own tokens, fp32 [N, M]       forge_wgrad_only
    2. reduce-scatter: rank r receives the sum of rows     torch.distributed
       ranges[r] over all ranks                            (NCCL on GPUs)
    3. AdamW (or SGD-momentum) on its shard of W, m, v     forge_owner_adamw
                                                           (forge_owner_sgdm)
This path materialises the partial gradients (the collective exchanges
them), so the zero-grad_W-bytes property of the fused single-GPU calls does
not apply to it.
"""
from __future__ import annotations

TILE_ROWS = 256  # d_in rows per output tile of the fused kernel


def owner_ranges(N: int, world: int, unit: int = TILE_ROWS) -> list[tuple[int, int]]:
    """Row ranges [(r0, r1)] of a [N, M] weight, one per rank: ceil(N / unit)
    tile rows in contiguous runs, the first (tiles % world) ranks taking one
    more.  Ranges are disjoint, ordered and cover [0, N); a rank gets an
    empty range when there are fewer tile rows than ranks."""
    if N < 1 or world < 1 or unit < 1:
        raise ValueError("N, world and unit must be positive")
    tiles = -(-N // unit)
    base, extra = divmod(tiles, world)
    out, t = [], 0
    for r in range(world):
        k = base + (1 if r < extra else 0)
        out.append((min(t * unit, N), min((t + k) * unit, N)))
        t += k
    return out


def tile_owner(tn: int, ranges: list[tuple[int, int]], unit: int = TILE_ROWS) -> int:
    """The rank that owns every tile of d_in tile row tn."""
    row = tn * unit
    for r, (r0, r1) in enumerate(ranges):
        if r0 <= row < r1:
            return r
    raise ValueError(f"tile row {tn} is outside the weight")


def reduce_scatter_rows(G, ranges, group=None):
    """Sum the ranks' partial gradients G [N, M] and return this rank's rows
    ranges[rank] of the sum ([r1 - r0, M], contiguous).  One reduce-scatter:
    over G itself when the ranges have equal lengths and cover it (every
    divisible case), else over a copy whose per-rank chunks are padded to the
    longest range."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    if len(ranges) != world:
        raise ValueError("one row range per rank expected")
    N, M = G.shape
    rows = max(r1 - r0 for r0, r1 in ranges)
    even = all(r1 - r0 == rows for r0, r1 in ranges) and rows * world == N
    if even:
        src = G.reshape(-1)
    else:
        buf = G.new_zeros((world, rows, M))
        for r, (r0, r1) in enumerate(ranges):
            buf[r, : r1 - r0] = G[r0:r1]
        src = buf.reshape(-1)
    out = torch.empty((rows, M), dtype=G.dtype, device=G.device)
    dist.reduce_scatter_tensor(out.reshape(-1), src, op=dist.ReduceOp.SUM, group=group)
    r0, r1 = ranges[rank]
    return out[: r1 - r0]


def owner_adamw_step(X, dY, W_shard, m_shard, v_shard, ranges, *, lr, beta1, beta2, eps, wd,
                     step, scales=None, grad=None, group=None):
    """One data-parallel step on this rank: the partial dW of its tokens
    (X [K_r, N], dY [K_r, M]), the reduce-scatter, and the owner's AdamW on
    its shard (W_shard, m_shard, v_shard: rows ranges[rank] of W, m, v).
    grad: an optional fp32 [N, M] buffer for the partial gradient.  All three
    run on the current stream, the one the collective orders itself after."""
    import torch
    import torch.distributed as dist

    import weight_grad_gemm_gb300 as fg
    N, M = X.shape[1], dY.shape[1]
    if grad is None:
        grad = torch.empty((N, M), dtype=torch.float32, device=X.device)
    fg.forge_wgrad_only(X, dY, grad, scales=scales)
    shard = reduce_scatter_rows(grad, ranges, group)
    r0, r1 = ranges[dist.get_rank(group)]
    if r1 > r0:
        fg.forge_owner_adamw(shard, W_shard, m_shard, v_shard, lr=lr, beta1=beta1, beta2=beta2,
                             eps=eps, wd=wd, step=step)


def owner_sgdm_step(X, dY, W_shard, mom_shard, ranges, *, lr, momentum, wd, scales=None,
                    grad=None, group=None):
    """owner_adamw_step with SGD-momentum: the partial dW of this rank's
    tokens, the reduce-scatter, and the owner's SGD-momentum step on its
    rows of W and the momentum buffer."""
    import torch
    import torch.distributed as dist

    import weight_grad_gemm_gb300 as fg
    N, M = X.shape[1], dY.shape[1]
    if grad is None:
        grad = torch.empty((N, M), dtype=torch.float32, device=X.device)
    fg.forge_wgrad_only(X, dY, grad, scales=scales)
    shard = reduce_scatter_rows(grad, ranges, group)
    r0, r1 = ranges[dist.get_rank(group)]
    if r1 > r0:
        fg.forge_owner_sgdm(shard, W_shard, mom_shard, lr=lr, momentum=momentum, wd=wd)

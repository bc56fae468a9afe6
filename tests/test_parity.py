"""GPU parity: the CUDA path against the fp64 oracle, element by element.

Sizes span several 128 x 256 output tiles with ragged edges in d_out (m),
d_in (n) and the token count (k), plus the degenerate cases (K = 0: pure
decay; K = 1; one partial tile).  Every call goes through the C ABI via the
Python binding.
"""
import numpy as np
import pytest
import torch

import oracle
import weight_grad_gemm_gb300 as fg
import workloads as wl
from parity_util import (check_dw, check_state_bf16, check_state_f32, check_W,
                         check_W_from_state, rms)

pytestmark = pytest.mark.gpu

HP = wl.AdamHP(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01).f32()

# (K tokens, N = d_in, M = d_out): several tiles, ragged m / n / k edges
SHAPES_BF16 = [
    (200, 520, 296),   # 3 n-tiles (last 8 wide), 3 m-tiles (last 40 wide), 4 k-blocks (last 8)
    (64, 256, 128),    # exactly one tile, one k-block
    (1, 8, 8),         # one token, one partial tile
    (17, 264, 136),
    (0, 264, 136),     # no tokens: g = 0
    (1000, 1032, 648),
]
SHAPES_E4M3 = [(300, 528, 304), (128, 256, 128), (1, 16, 16), (0, 272, 144)]


def bf16_inputs(K, N, M, seed=0, scale=None):
    X = wl.activations(K, N, wl.seed_of("X", seed, K, N), scale=scale)
    D = wl.activations(K, M, wl.seed_of("dY", seed, K, M), scale=scale)
    return X, D


def e4m3_inputs(K, N, M, seed):
    X, sx = wl.quantize_e4m3(wl.with_outliers((K, N), wl.seed_of("X8", seed, K, N)))
    D, sy = wl.quantize_e4m3(wl.with_outliers((K, M), wl.seed_of("dY8", seed, K, M)))
    return X, D, (sx, sy)


def warm_state(N, M, seed, state_bf16=False):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((N, M)) * 0.02).astype(np.float32)
    m = (rng.standard_normal((N, M)) * 1e-3).astype(np.float32)
    v = (rng.random((N, M)) * 1e-5).astype(np.float32)
    if state_bf16:
        m, v = oracle.round_bf16(m), oracle.round_bf16(v)
    return W, m, v


def dev_state(a, dev):
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(a).to(dev)


def host_state(t):
    t = t.cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def scales_dev(sc, dev):
    return torch.tensor(sc, dtype=torch.float32, device=dev)


@pytest.fixture(params=["stage", "loader"])
def misaligned_path(request, monkeypatch):
    """Operands TMA cannot address: staged into a padded copy, or fetched by
    the kernel's cp.async loader."""
    monkeypatch.setenv("FORGE_MISALIGNED", request.param)
    return request.param


@pytest.fixture(params=["single", "pair"])
def kernel_form(request, monkeypatch):
    """Run a dense test on the one-CTA kernel and on CTA pairs."""
    monkeypatch.setenv("FORGE_KERNEL", request.param)
    return request.param


# ------------------------------------------------------------------ dW only

@pytest.mark.parametrize("K,N,M", SHAPES_BF16)
def test_wgrad_only_bf16(cuda_device, kernel_form, K, N, M):
    X, D = bf16_inputs(K, N, M, 1)
    dW = torch.full((N, M), float("nan"), device=cuda_device)
    fg.forge_wgrad_only(X.to(cuda_device), D.to(cuda_device), dW)
    torch.cuda.synchronize()
    ref = oracle.wgrad(X, D)
    got = dW.cpu().numpy()
    assert np.isfinite(got).all()
    if K == 0:
        assert not got.any()
    else:
        check_dw(got, ref, "bf16")


@pytest.mark.parametrize("K,N,M", SHAPES_E4M3)
def test_wgrad_only_e4m3(cuda_device, kernel_form, K, N, M):
    X, D, sc = e4m3_inputs(K, N, M, 2)
    dW = torch.full((N, M), float("nan"), device=cuda_device)
    fg.forge_wgrad_only(X.to(cuda_device), D.to(cuda_device), dW, scales=scales_dev(sc, cuda_device))
    torch.cuda.synchronize()
    got = dW.cpu().numpy()
    assert np.isfinite(got).all()
    if K == 0:
        assert not got.any()
    else:
        check_dw(got, oracle.wgrad(X, D, scales=sc), "e4m3")


# ------------------------------------------------------------------ AdamW

def run_adamw(dev, X, D, W, m, v, step, hp=HP, scales=None):
    Wd, md, vd = dev_state(W, dev), dev_state(m, dev), dev_state(v, dev)
    fg.forge_wgrad_adamw(X.to(dev), D.to(dev), Wd, md, vd, lr=hp.lr, beta1=hp.beta1,
                         beta2=hp.beta2, eps=hp.eps, wd=hp.wd, step=step,
                         scales=None if scales is None else scales_dev(scales, dev))
    torch.cuda.synchronize()
    return host_state(Wd), host_state(md), host_state(vd)


def adamw_ref(G, W, m, v, step, **hp):
    """The oracle's AdamW step, with the inputs the all-elements W check needs."""
    ref = oracle.adamw(G, W, m, v, step=step, **hp)
    ref.update(W_old=W, hp=wl.AdamHP(**hp), step=step)
    return ref


def check_adamw(got, ref, G, lr, state_bf16):
    W, m, v = got
    if state_bf16:
        check_state_bf16(m, ref["m_exact"], "m")
        check_state_bf16(v, ref["v_exact"], "v")
    else:
        check_state_f32(m, ref["m_exact"], "m")
        check_state_f32(v, ref["v_exact"], "v")
    check_W(W, ref["W_exact"], G, lr, m_exact=ref["m_exact"])
    if "W_old" in ref:
        check_W_from_state(W, ref["W_old"], m, v, ref["hp"], ref["step"], state_bf16)


@pytest.mark.parametrize("state_bf16", [False, True], ids=["f32state", "bf16state"])
@pytest.mark.parametrize("K,N,M", SHAPES_BF16)
def test_adamw_bf16(cuda_device, kernel_form, K, N, M, state_bf16):
    X, D = bf16_inputs(K, N, M, 3)
    W, m, v = warm_state(N, M, 4, state_bf16)
    got = run_adamw(cuda_device, X, D, W, m, v, step=4)
    G = oracle.wgrad(X, D)
    ref = adamw_ref(G, W, m, v, step=4, **vars(HP))
    check_adamw(got, ref, G, HP.lr, state_bf16)


@pytest.mark.parametrize("state_bf16", [False, True], ids=["f32state", "bf16state"])
@pytest.mark.parametrize("K,N,M", SHAPES_E4M3)
def test_adamw_e4m3(cuda_device, kernel_form, K, N, M, state_bf16):
    X, D, sc = e4m3_inputs(K, N, M, 5)
    W, m, v = warm_state(N, M, 6, state_bf16)
    got = run_adamw(cuda_device, X, D, W, m, v, step=2, scales=sc)
    G = oracle.wgrad(X, D, scales=sc)
    ref = adamw_ref(G, W, m, v, step=2, **vars(HP))
    check_adamw(got, ref, G, HP.lr, state_bf16)


def test_adamw_first_step_from_zero_state(cuda_device, kernel_form):
    # step 1 from m = v = 0 (the linear-layer workload's start)
    K, N, M = 512, 256, 256
    X, D = bf16_inputs(K, N, M, 7, scale=0.05)
    rng = np.random.default_rng(8)
    W = (rng.standard_normal((N, M)) * 0.02).astype(np.float32)
    z = np.zeros((N, M), np.float32)
    got = run_adamw(cuda_device, X, D, W, z, z, step=1)
    G = oracle.wgrad(X, D)
    ref = adamw_ref(G, W, z, z, step=1, **vars(HP))
    check_adamw(got, ref, G, HP.lr, False)


def test_linear_workload_ten_steps_resynced(cuda_device, kernel_form):
    """The 10-step linear-layer workload; each step gated against the oracle
    started from the GPU's previous outputs."""
    wk = wl.LINEAR
    hp = wk.adam.f32()
    rng = np.random.default_rng(9)
    W = (rng.standard_normal((wk.N, wk.M)) * 0.02).astype(np.float32)
    m = np.zeros((wk.N, wk.M), np.float32)
    v = np.zeros((wk.N, wk.M), np.float32)
    for t in range(1, wk.steps + 1):
        X, D = bf16_inputs(wk.K, wk.N, wk.M, 100 + t, scale=0.05)
        got = run_adamw(cuda_device, X, D, W, m, v, step=t, hp=hp)
        G = oracle.wgrad(X, D)
        ref = adamw_ref(G, W, m, v, step=t, **vars(hp))
        check_adamw(got, ref, G, hp.lr, False)
        W, m, v = got


# ------------------------------------------------------------------ SGD momentum

@pytest.mark.parametrize("state_bf16", [False, True], ids=["f32state", "bf16state"])
@pytest.mark.parametrize("kind", ["bf16", "e4m3"])
@pytest.mark.parametrize("K,N,M", [(200, 528, 304), (0, 272, 144), (1, 16, 16)])
def test_sgdm(cuda_device, kernel_form, K, N, M, kind, state_bf16):
    if kind == "bf16":
        X, D = bf16_inputs(K, N, M, 10)
        sc = None
        G = oracle.wgrad(X, D)
    else:
        X, D, sc = e4m3_inputs(K, N, M, 11)
        G = oracle.wgrad(X, D, scales=sc)
    W, buf, _ = warm_state(N, M, 12, state_bf16)
    hp = wl.SgdHP(lr=1e-2, momentum=0.9, wd=0.05).f32()
    Wd, bd = dev_state(W, cuda_device), dev_state(buf, cuda_device)
    fg.forge_wgrad_sgdm(X.to(cuda_device), D.to(cuda_device), Wd, bd, lr=hp.lr,
                        momentum=hp.momentum, wd=hp.wd,
                        scales=None if sc is None else scales_dev(sc, cuda_device))
    torch.cuda.synchronize()
    ref = oracle.sgdm(G, W, buf, lr=hp.lr, momentum=hp.momentum, wd=hp.wd)
    if state_bf16:
        check_state_bf16(host_state(bd), ref["buf_exact"], "buf")
    else:
        check_state_f32(host_state(bd), ref["buf_exact"], "buf")
    # SGD moves W by lr * buf: compare W within 2e-3 * lr * rms(buf) + fp32 rounding of W
    err = np.max(np.abs(host_state(Wd).astype(np.float64) - ref["W_exact"]))
    assert err <= 2e-3 * hp.lr * rms(ref["buf_exact"]) + 2 * np.finfo(np.float32).eps * 0.1


# ------------------------------------------------------------------ grouped

def grouped_case(counts, N, M, seed, state_bf16=False, kind="bf16"):
    T = int(sum(counts))
    Tm = max(T, 1)
    if kind == "bf16":
        X, D = bf16_inputs(Tm, N, M, seed)
        sc = None
    else:
        X, D, sc = e4m3_inputs(Tm, N, M, seed)
    E = len(counts)
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((E, N, M)) * 0.02).astype(np.float32)
    m = (rng.standard_normal((E, N, M)) * 1e-3).astype(np.float32)
    v = (rng.random((E, N, M)) * 1e-5).astype(np.float32)
    if state_bf16:
        m, v = oracle.round_bf16(m), oracle.round_bf16(v)
    return X, D, wl.offsets_from_counts(counts), W, m, v, sc


def run_grouped(dev, X, D, off, W, m, v, step, hp=HP, scales=None):
    Wd, md, vd = dev_state(W, dev), dev_state(m, dev), dev_state(v, dev)
    offd = torch.from_numpy(np.asarray(off, np.int32)).to(dev)
    fg.forge_grouped_wgrad_adamw(X.to(dev), D.to(dev), Wd, md, vd, offd, lr=hp.lr,
                                 beta1=hp.beta1, beta2=hp.beta2, eps=hp.eps, wd=hp.wd, step=step,
                                 scales=None if scales is None else scales_dev(scales, dev))
    torch.cuda.synchronize()
    return host_state(Wd), host_state(md), host_state(vd)


def check_grouped(got, X, D, off, W, m, v, step, sc, state_bf16, hp=HP):
    ref = oracle.grouped_adamw(X, D, off, W, m, v, step=step, scales=sc or (1.0, 1.0),
                               **vars(hp))
    for e in range(len(off) - 1):
        G = oracle.wgrad(X, D, k_range=(int(off[e]), int(off[e + 1])), scales=sc or (1.0, 1.0))
        sub = {k: ref[k][e] for k in ("W_exact", "m_exact", "v_exact")}
        sub.update(W_old=W[e], hp=hp, step=step)
        check_adamw((got[0][e], got[1][e], got[2][e]), sub, G, hp.lr, state_bf16)


@pytest.fixture(params=["single", "pair"])
def grouped_form(request, monkeypatch):
    """Run a grouped test on the one-CTA kernel and on CTA pairs."""
    monkeypatch.setenv("FORGE_KERNEL", request.param)
    return request.param


@pytest.mark.parametrize("state_bf16", [False, True], ids=["f32state", "bf16state"])
def test_grouped_ragged_with_empty_experts(cuda_device, grouped_form, state_bf16):
    counts = [37, 0, 100, 64, 3, 0, 129]
    N, M = 264, 136
    X, D, off, W, m, v, sc = grouped_case(counts, N, M, 13, state_bf16)
    got = run_grouped(cuda_device, X, D, off, W, m, v, step=3)
    check_grouped(got, X, D, off, W, m, v, 3, sc, state_bf16)


def test_grouped_e4m3(cuda_device, grouped_form):
    counts = [200, 0, 57, 128]
    N, M = 272, 144
    X, D, off, W, m, v, sc = grouped_case(counts, N, M, 14, kind="e4m3")
    got = run_grouped(cuda_device, X, D, off, W, m, v, step=2, scales=sc)
    check_grouped(got, X, D, off, W, m, v, 2, sc, False)


@pytest.mark.parametrize("kind", ["bf16", "e4m3"])
def test_grouped_tails_on_k_step_boundaries(cuda_device, grouped_form, kind):
    """Experts whose last k-block ends on an MMA k-step (16 bf16 or 32 e4m3
    token rows) or one row past or short of one: whole k-steps, k-steps with
    rows of the next expert behind them, and blocks shorter than a k-step."""
    counts = [96, 16, 48, 80, 113, 1] if kind == "bf16" else [160, 32, 96, 64, 161, 31]
    N, M = 264, 392
    X, D, off, W, m, v, sc = grouped_case(counts, N, M, 17, kind=kind)
    got = run_grouped(cuda_device, X, D, off, W, m, v, step=2, scales=sc)
    check_grouped(got, X, D, off, W, m, v, 2, sc, False)


def test_grouped_all_experts_empty(cuda_device, grouped_form):
    counts = [0, 0, 0]
    N, M = 256, 128
    X, D, off, W, m, v, sc = grouped_case(counts, N, M, 15)
    got = run_grouped(cuda_device, X, D, off, W, m, v, step=5)
    ref = oracle.grouped_adamw(X, D, off, W, m, v, step=5, **vars(HP))
    for e in range(3):
        check_state_f32(got[1][e], ref["m_exact"][e])
        check_state_f32(got[2][e], ref["v_exact"][e])
        check_W(got[0][e], ref["W_exact"][e], np.zeros((N, M)), HP.lr, m_exact=ref["m_exact"][e])


def test_grouped_single_expert_equals_dense_bitwise(cuda_device, grouped_form):
    K, N, M = 300, 520, 296
    X, D, off, W, m, v, _ = grouped_case([K], N, M, 16)
    g = run_grouped(cuda_device, X, D, off, W, m, v, step=2)
    d = run_adamw(cuda_device, X, D, W[0], m[0], v[0], step=2)
    for a, b in zip(g, d):
        assert np.array_equal(a[0], b)


def test_grouped_many_experts(cuda_device, grouped_form):
    """257 experts, a third of them without tokens, ragged counts: the
    offset copy, validation and heavy-first ranking run over every expert."""
    rng = np.random.default_rng(24)
    counts = rng.integers(0, 40, size=257)
    counts[rng.random(257) < 0.33] = 0
    N, M = 136, 264
    X, D, off, W, m, v, sc = grouped_case(list(counts), N, M, 25)
    got = run_grouped(cuda_device, X, D, off, W, m, v, step=4)
    assert fg.forge_get_device_status() == fg.FORGE_OK
    check_grouped(got, X, D, off, W, m, v, 4, sc, False)


def test_grouped_rows_outside_every_expert(cuda_device, grouped_form):
    """offsets[0] > 0 and offsets[E] < T_max: the packed buffer's leading
    and trailing rows belong to no expert (here non-finite), and no expert's
    gradient reads them, not even in its first or last partial k-block."""
    counts = [30, 0, 70, 5]
    N, M = 264, 392
    lead, trail = 37, 23
    X, D, off, W, m, v, sc = grouped_case(counts, N, M, 28)
    T = int(off[-1])
    Xb = torch.full((lead + T + trail, N), float("nan"), dtype=torch.bfloat16)
    Db = torch.full((lead + T + trail, M), float("inf"), dtype=torch.bfloat16)
    Xb[lead:lead + T] = X[:T]
    Db[lead:lead + T] = D[:T]
    offb = np.asarray(off) + lead
    got = run_grouped(cuda_device, Xb, Db, offb, W, m, v, step=2)
    assert fg.forge_get_device_status() == fg.FORGE_OK
    for e in range(len(counts)):
        assert np.all(np.isfinite(got[0][e])) and np.all(np.isfinite(got[1][e]))
    check_grouped(got, X, D, off, W, m, v, 2, sc, False)


def test_grouped_max_experts(cuda_device, grouped_form):
    """1024 experts, the most one call takes: the expert table fills shared
    memory up to the next carve-out step; ragged counts of 0-5 tokens."""
    rng = np.random.default_rng(26)
    counts = rng.integers(0, 6, size=1024)
    N, M = 8, 136
    X, D, off, W, m, v, sc = grouped_case(list(counts), N, M, 27)
    got = run_grouped(cuda_device, X, D, off, W, m, v, step=3)
    assert fg.forge_get_device_status() == fg.FORGE_OK
    check_grouped(got, X, D, off, W, m, v, 3, sc, False)


def test_grouped_foreign_tokens_never_enter(cuda_device, grouped_form):
    """Expert e's gradient is the sum over its own tokens only: non-finite
    values in a neighbour's rows (which share the partial k-blocks at both
    ends of expert 1's segment) leave experts 0 and 2 exact."""
    counts = [40, 50, 30]
    N, M = 264, 264
    X, D, off, W, m, v, sc = grouped_case(counts, N, M, 23)
    X, D = X.clone(), D.clone()
    X[41, 5] = float("inf")
    X[60, :] = float("nan")
    D[45, 7] = float("-inf")
    got = run_grouped(cuda_device, X, D, off, W, m, v, step=2)
    ref = oracle.grouped_adamw(X, D, off, W, m, v, step=2, **vars(HP))
    for e in (0, 2):
        assert np.all(np.isfinite(got[0][e]))
        G = oracle.wgrad(X, D, k_range=(int(off[e]), int(off[e + 1])))
        sub = {k: ref[k][e] for k in ("W_exact", "m_exact", "v_exact")}
        check_adamw((got[0][e], got[1][e], got[2][e]), sub, G, HP.lr, False)


# ------------------------------------------------------------------ invariance (P1, no atomics)

def test_bitwise_run_to_run(cuda_device, kernel_form):
    K, N, M = 1000, 1032, 648
    X, D = bf16_inputs(K, N, M, 17)
    W, m, v = warm_state(N, M, 18)
    a = run_adamw(cuda_device, X, D, W, m, v, step=3)
    b = run_adamw(cuda_device, X, D, W, m, v, step=3)
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))


def relabel(order, counts, X, D, W, m, v):
    """The same experts under new labels: position j holds expert order[j],
    its token segment packed j-th and its W, m, v stacked j-th."""
    off = wl.offsets_from_counts(counts)
    Xp = torch.cat([X[off[e]:off[e + 1]] for e in order] + [X[off[-1]:]])
    Dp = torch.cat([D[off[e]:off[e + 1]] for e in order] + [D[off[-1]:]])
    offp = wl.offsets_from_counts([counts[e] for e in order])
    return Xp, Dp, offp, W[order], m[order], v[order]


# ties (133, 133 / 64, 64 / 0, 0) and empty experts, so that relabelling
# changes the heavy-first ranking (ties go by label) and the two-ended walk
ORDER_COUNTS = [70, 0, 133, 64, 9, 64, 0, 133]
ORDER_PERMS = [[7, 6, 5, 4, 3, 2, 1, 0], [3, 0, 6, 2, 7, 5, 1, 4]]


@pytest.mark.parametrize("state_bf16", [False, True], ids=["f32state", "bf16state"])
@pytest.mark.parametrize("perm", range(len(ORDER_PERMS)))
def test_grouped_bitwise_across_expert_order(cuda_device, grouped_form, state_bf16, perm):
    """P1's schedule independence on one multi-expert launch: relabelling the
    experts (segments packed in another order, state stacked to match) gives
    every expert the same W, m, v bit for bit."""
    counts = ORDER_COUNTS
    N, M = 520, 1032  # 3 x 5 pair tiles (3 x 9 one-CTA tiles) per expert
    X, D, off, W, m, v, _ = grouped_case(counts, N, M, 19, state_bf16)
    base = run_grouped(cuda_device, X, D, off, W, m, v, step=2)
    order = ORDER_PERMS[perm]
    Xp, Dp, offp, Wp, mp, vp = relabel(order, counts, X, D, W, m, v)
    got = run_grouped(cuda_device, Xp, Dp, offp, Wp, mp, vp, step=2)
    for j, e in enumerate(order):
        for a, b in zip(got, base):
            assert np.array_equal(a[j], b[e]), f"expert {e} differs under label {j}"


@pytest.mark.parametrize("band", ["1", "3", "8", "0"])
def test_grouped_bitwise_across_raster_bands(cuda_device, grouped_form, monkeypatch, band):
    """The tile walk's raster bands (1 d_out tile, 3, 8, whole rows) reorder
    the schedule, never a tile's own K order."""
    counts = ORDER_COUNTS
    N, M = 520, 1032
    X, D, off, W, m, v, _ = grouped_case(counts, N, M, 20)
    monkeypatch.setenv("FORGE_RASTER_BAND", "1")
    base = run_grouped(cuda_device, X, D, off, W, m, v, step=2)
    monkeypatch.setenv("FORGE_RASTER_BAND", band)
    got = run_grouped(cuda_device, X, D, off, W, m, v, step=2)
    for a, b in zip(got, base):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("band", ["3", "8", "0"])
def test_dense_bitwise_across_raster_bands(cuda_device, kernel_form, monkeypatch, band):
    K, N, M = 300, 1032, 2056  # 5 x 9 pair tiles (5 x 17 one-CTA tiles)
    X, D = bf16_inputs(K, N, M, 21)
    W, m, v = warm_state(N, M, 22)
    monkeypatch.setenv("FORGE_RASTER_BAND", "1")
    base = run_adamw(cuda_device, X, D, W, m, v, step=3)
    monkeypatch.setenv("FORGE_RASTER_BAND", band)
    got = run_adamw(cuda_device, X, D, W, m, v, step=3)
    for a, b in zip(got, base):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


# ------------------------------------------------------------------ failure detection

def test_bounded_wait_reports_timeout_and_context_survives(cuda_device):
    assert fg.forge_get_device_status() == fg.FORGE_OK
    fg.forge_selftest_wait_timeout(2000)  # 2 ms on a barrier nothing completes
    assert fg.forge_get_device_status() == fg.FORGE_ERR_TIMEOUT
    assert fg.forge_get_device_status() == fg.FORGE_OK  # read clears
    # the context is still usable
    X, D = bf16_inputs(64, 256, 128, 20)
    dW = torch.empty((256, 128), device=cuda_device)
    fg.forge_wgrad_only(X.to(cuda_device), D.to(cuda_device), dW)
    torch.cuda.synchronize()
    check_dw(dW.cpu().numpy(), oracle.wgrad(X, D))


def test_grouped_bad_offsets_flagged_on_device(cuda_device):
    X, D, off, W, m, v, _ = grouped_case([10, 20], 256, 128, 21)
    bad = np.array([0, 25, 20])  # decreasing
    W0 = W.copy()
    got = run_grouped(cuda_device, X, D, bad, W, m, v, step=1)
    assert fg.forge_get_device_status() == fg.FORGE_ERR_INVALID_ARG
    assert np.array_equal(got[0], W0)  # nothing written


# ------------------------------------------------------------------ rows TMA cannot address

# (K, N, M): row strides that are not multiples of 16 bytes are staged into a
# padded copy for TMA or fetched by the cp.async loader; d_out not a multiple
# of 4 also exercises the scalar epilogue
SHAPES_MISALIGNED_BF16 = [
    (300, 264, 4100),   # dY rows 8200 B -> 8-byte copies
    (130, 264, 302),    # dY rows 604 B -> 4-byte copies, scalar epilogue
    (200, 4100, 136),   # X rows 8200 B
    (77, 1002, 302),    # both operands, 4-byte copies
    (1, 6, 10),         # one token, tiny
]


@pytest.mark.parametrize("K,N,M", SHAPES_MISALIGNED_BF16)
def test_wgrad_only_misaligned_rows(cuda_device, misaligned_path, K, N, M):
    X, D = bf16_inputs(K, N, M, 40)
    dW = torch.full((N, M), float("nan"), device=cuda_device)
    fg.forge_wgrad_only(X.to(cuda_device), D.to(cuda_device), dW)
    torch.cuda.synchronize()
    check_dw(dW.cpu().numpy(), oracle.wgrad(X, D), "bf16")


@pytest.mark.parametrize("state_bf16", [False, True], ids=["f32state", "bf16state"])
@pytest.mark.parametrize("K,N,M", SHAPES_MISALIGNED_BF16)
def test_adamw_misaligned_rows(cuda_device, misaligned_path, K, N, M, state_bf16):
    X, D = bf16_inputs(K, N, M, 41)
    W, m, v = warm_state(N, M, 42, state_bf16)
    got = run_adamw(cuda_device, X, D, W, m, v, step=5)
    G = oracle.wgrad(X, D)
    ref = adamw_ref(G, W, m, v, step=5, **vars(HP))
    check_adamw(got, ref, G, HP.lr, state_bf16)


@pytest.mark.parametrize("K,N,M", [(256, 520, 1000), (100, 260, 4100)])
def test_e4m3_misaligned_rows(cuda_device, misaligned_path, K, N, M):
    X, D, sc = e4m3_inputs(K, N, M, 43)
    W, m, v = warm_state(N, M, 44)
    got = run_adamw(cuda_device, X, D, W, m, v, step=2, scales=sc)
    G = oracle.wgrad(X, D, scales=sc)
    ref = adamw_ref(G, W, m, v, step=2, **vars(HP))
    check_adamw(got, ref, G, HP.lr, False)


def test_offset_base_pointers(cuda_device, misaligned_path):
    # operands that start 8 bytes into an allocation: TMA needs 16-byte bases
    K, N, M = 96, 264, 136
    X, D = bf16_inputs(K, N, M, 45)
    xb = torch.empty(K * N + 4, dtype=torch.bfloat16, device=cuda_device)
    db = torch.empty(K * M + 4, dtype=torch.bfloat16, device=cuda_device)
    Xd = xb[4:].view(K, N)
    Dd = db[4:].view(K, M)
    Xd.copy_(X)
    Dd.copy_(D)
    dW = torch.empty((N, M), device=cuda_device)
    fg.forge_wgrad_only(Xd, Dd, dW)
    torch.cuda.synchronize()
    check_dw(dW.cpu().numpy(), oracle.wgrad(X, D))


def test_grouped_misaligned_rows(cuda_device, misaligned_path, grouped_form):
    counts = [37, 0, 100, 9]
    N, M = 264, 4100
    X, D, off, W, m, v, sc = grouped_case(counts, N, M, 46)
    got = run_grouped(cuda_device, X, D, off, W, m, v, step=2)
    check_grouped(got, X, D, off, W, m, v, 2, sc, False)


# Rows that are not a multiple of 4 bytes (odd bf16 widths, e4m3 widths not
# divisible by 4): always staged into 16-byte rows by the byte-granular copy,
# whichever loader the caller asks for; the epilogue takes its scalar path.
SHAPES_ODD_BF16 = [
    (150, 264, 1),      # d_out 1: one column
    (150, 264, 3),
    (130, 264, 301),    # 602-byte dY rows
    (100, 136, 4097),   # d_out 4097: one column past 16 pair tiles
    (120, 7, 136),      # d_in 7: 14-byte X rows
    (90, 4097, 136),    # d_in 4097
    (77, 7, 301),       # both operands odd
    (1, 3, 5),          # one token, tiny
]


@pytest.mark.parametrize("K,N,M", SHAPES_ODD_BF16)
def test_wgrad_only_odd_widths(cuda_device, misaligned_path, K, N, M):
    X, D = bf16_inputs(K, N, M, 47)
    dW = torch.full((N, M), float("nan"), device=cuda_device)
    fg.forge_wgrad_only(X.to(cuda_device), D.to(cuda_device), dW)
    torch.cuda.synchronize()
    check_dw(dW.cpu().numpy(), oracle.wgrad(X, D), "bf16")


@pytest.mark.parametrize("state_bf16", [False, True], ids=["f32state", "bf16state"])
@pytest.mark.parametrize("K,N,M", SHAPES_ODD_BF16)
def test_adamw_odd_widths(cuda_device, misaligned_path, K, N, M, state_bf16):
    X, D = bf16_inputs(K, N, M, 48)
    W, m, v = warm_state(N, M, 49, state_bf16)
    got = run_adamw(cuda_device, X, D, W, m, v, step=3)
    G = oracle.wgrad(X, D)
    ref = adamw_ref(G, W, m, v, step=3, **vars(HP))
    check_adamw(got, ref, G, HP.lr, state_bf16)


@pytest.mark.parametrize("K,N,M", [(130, 4097, 264), (100, 264, 4098), (96, 4099, 4099),
                                   (64, 5, 6)])
def test_e4m3_widths_not_divisible_by_four(cuda_device, misaligned_path, K, N, M):
    X, D, sc = e4m3_inputs(K, N, M, 50)
    W, m, v = warm_state(N, M, 51)
    got = run_adamw(cuda_device, X, D, W, m, v, step=2, scales=sc)
    G = oracle.wgrad(X, D, scales=sc)
    ref = adamw_ref(G, W, m, v, step=2, **vars(HP))
    check_adamw(got, ref, G, HP.lr, False)


@pytest.mark.parametrize("kind", ["bf16", "e4m3"])
def test_sgdm_odd_widths(cuda_device, kind):
    K, N, M = 140, 263, 301
    if kind == "bf16":
        X, D = bf16_inputs(K, N, M, 52)
        sc = None
        G = oracle.wgrad(X, D)
    else:
        X, D, sc = e4m3_inputs(K, N, M, 53)
        G = oracle.wgrad(X, D, scales=sc)
    W, buf, _ = warm_state(N, M, 54)
    hp = wl.SgdHP(lr=1e-2, momentum=0.9, wd=0.05).f32()
    Wd, bd = dev_state(W, cuda_device), dev_state(buf, cuda_device)
    fg.forge_wgrad_sgdm(X.to(cuda_device), D.to(cuda_device), Wd, bd, lr=hp.lr,
                        momentum=hp.momentum, wd=hp.wd,
                        scales=None if sc is None else scales_dev(sc, cuda_device))
    torch.cuda.synchronize()
    ref = oracle.sgdm(G, W, buf, lr=hp.lr, momentum=hp.momentum, wd=hp.wd)
    check_state_f32(host_state(bd), ref["buf_exact"], "buf")
    err = np.max(np.abs(host_state(Wd).astype(np.float64) - ref["W_exact"]))
    assert err <= 2e-3 * hp.lr * rms(ref["buf_exact"]) + 2 * np.finfo(np.float32).eps * 0.1


@pytest.mark.parametrize("kind,N,M", [("bf16", 263, 301), ("bf16", 7, 4097),
                                      ("e4m3", 261, 146)])
def test_grouped_odd_widths(cuda_device, grouped_form, kind, N, M):
    counts = [37, 0, 100, 9]
    X, D, off, W, m, v, sc = grouped_case(counts, N, M, 55, kind=kind)
    got = run_grouped(cuda_device, X, D, off, W, m, v, step=2, scales=sc)
    check_grouped(got, X, D, off, W, m, v, 2, sc, False)


def test_element_misaligned_base_is_rejected(cuda_device):
    """The one class of operand the library refuses: a bf16 base one byte
    off its element alignment (no kernel launches)."""
    K, N, M = 32, 264, 136
    raw = torch.zeros(K * N * 2 + 16, dtype=torch.uint8, device=cuda_device)
    D = torch.zeros((K, M), dtype=torch.bfloat16, device=cuda_device)
    dW = torch.zeros((N, M), device=cuda_device)
    st = fg.lib().forge_wgrad_only(raw.data_ptr() + 1, D.data_ptr(), dW.data_ptr(), M, N, K,
                                   fg.FORGE_BF16, None, None)
    assert st == fg.FORGE_ERR_MISALIGNED


def test_pointers_outside_device_memory_are_rejected(cuda_device):
    """Host memory (pageable or pinned) where device memory of the current
    device is required: refused before any launch, nothing written."""
    K, N, M = 64, 264, 136
    X = torch.zeros((K, N), dtype=torch.bfloat16, device=cuda_device)
    D = torch.zeros((K, M), dtype=torch.bfloat16, device=cuda_device)
    W = torch.zeros((N, M), device=cuda_device)
    m = torch.zeros((N, M), device=cuda_device)
    v = torch.zeros((N, M), device=cuda_device)
    host = np.zeros((N, M), np.float32)
    pinned = torch.zeros((N, M), pin_memory=True)
    L = fg.lib()

    def call(Wp, Xp=X.data_ptr()):
        return L.forge_wgrad_adamw(Xp, D.data_ptr(), Wp, m.data_ptr(), v.data_ptr(), M, N, K,
                                   fg.FORGE_BF16, fg.FORGE_F32, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1,
                                   None, None)

    assert call(host.ctypes.data) == fg.FORGE_ERR_INVALID_ARG
    assert call(pinned.data_ptr()) == fg.FORGE_ERR_INVALID_ARG
    xh = torch.zeros((K, N), dtype=torch.bfloat16, pin_memory=True)
    assert call(W.data_ptr(), xh.data_ptr()) == fg.FORGE_ERR_INVALID_ARG
    codes = torch.zeros(16, dtype=torch.uint8, device=cuda_device)
    assert L.forge_quantize_e4m3(X.data_ptr(), fg.FORGE_BF16, 16, codes.data_ptr(),
                                 pinned.data_ptr(), None) == fg.FORGE_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert not W.any() and not m.any()
    assert call(W.data_ptr()) == fg.FORGE_OK  # the same call on device memory runs
    torch.cuda.synchronize()

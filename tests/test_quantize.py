"""GPU parity of the e4m3 amax quantiser against the oracle: codes and the
scale must match bit for bit (the decision of each code is taken in fp32 on
both sides: the quotient x / s, then the nearest e4m3 value, ties to even),
and nothing outside codes and scale is written."""
import numpy as np
import pytest
import torch

import oracle
import weight_grad_gemm_gb300 as fg
import workloads as wl

pytestmark = pytest.mark.gpu


def gpu_quantize(x):
    codes = torch.empty(x.numel(), dtype=torch.uint8, device=x.device)
    scale = torch.full((1,), float("nan"), device=x.device)
    fg.forge_quantize_e4m3(x, codes, scale)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), float(scale.item())


def check(x):
    codes, s = gpu_quantize(x)
    want, ws = oracle.quantize_e4m3(x.detach().cpu().reshape(-1))
    assert s == ws
    bad = np.nonzero(codes != want)[0]
    assert bad.size == 0, (bad[:8], codes[bad[:8]], want[bad[:8]])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("shape", [(0,), (1,), (3,), (4,), (1001,), (257, 515), (4096, 520)])
def test_quantize_matches_oracle(cuda_device, dtype, shape):
    x = wl.with_outliers(shape, wl.seed_of("q", *shape), device=cuda_device).to(dtype)
    check(x)


def test_quantize_subnormal_codes_and_ties(cuda_device):
    # one large entry makes most quotients fall in e4m3's subnormal range; the
    # exact midpoints between codes (times s) test ties to even
    dev = cuda_device
    small = wl.randn((5000,), wl.seed_of("q-sub"), device=dev, std=1e-3)
    x = torch.cat([small, torch.tensor([448.0], device=dev)])  # s = 1
    check(x)
    vals = oracle.decode(np.arange(127, dtype=np.uint8))
    mids = torch.tensor((vals[:-1] + vals[1:]) / 2, dtype=torch.float32, device=dev)
    check(torch.cat([mids, -mids, torch.tensor([448.0], device=dev)]))


def test_quantize_degenerate_and_misaligned(cuda_device):
    dev = cuda_device
    codes, s = gpu_quantize(torch.zeros(33, device=dev))
    assert s == 1.0 and not codes.any()
    buf = wl.with_outliers((1 + 4003,), wl.seed_of("q-mis"), device=dev)
    check(buf[1:])  # 4 bytes past a 16-byte boundary: the scalar path
    b16 = buf.to(torch.bfloat16)
    check(b16[3:])


@pytest.mark.parametrize("n", [5, 7, 8, 9, 11, 12, 13, 2047, 2049, 70001])
@pytest.mark.parametrize("offset", [0, 1, 2, 3])
def test_quantize_codes_at_any_byte_offset(cuda_device, n, offset):
    """The first pass parks its partial maxima in a 4-byte aligned window of
    the codes buffer: codes that start 1-3 bytes past a word, and sizes
    around the single-block threshold, must come out exactly as the oracle's
    (the window is overwritten by the codes, never left behind)."""
    dev = cuda_device
    x = wl.with_outliers((n,), wl.seed_of("q-off", n, offset), device=dev)
    buf = torch.full((n + 8,), 0xAB, dtype=torch.uint8, device=dev)
    codes = buf[offset:offset + n]
    scale = torch.full((1,), float("nan"), device=dev)
    fg.forge_quantize_e4m3(x, codes, scale)
    torch.cuda.synchronize()
    want, ws = oracle.quantize_e4m3(x.cpu())
    assert float(scale.item()) == ws
    got = buf.cpu().numpy()
    assert np.array_equal(got[offset:offset + n], want)
    assert (got[:offset] == 0xAB).all() and (got[offset + n:] == 0xAB).all()


def test_quantize_full_size_and_feeds_the_fp8_call(cuda_device):
    """The fp8 workload's X [32768, 8192] and dY: codes and scales equal the
    oracle's over the whole tensors, and an e4m3 call takes them as they
    come (codes as X / dY, the two scales as its scales)."""
    from parity_util import check_dw
    wk = wl.FP8
    dev = cuda_device
    K, N, M = wk.K, wk.N, wk.M
    xf = wl.with_outliers((K, N), wl.seed_of(wk.name, "X"), device=dev)
    yf = wl.with_outliers((K, M), wl.seed_of(wk.name, "dY"), device=dev)
    qx = torch.empty((K, N), dtype=torch.float8_e4m3fn, device=dev)
    qy = torch.empty((K, M), dtype=torch.float8_e4m3fn, device=dev)
    sc = torch.empty(2, device=dev)
    fg.forge_quantize_e4m3(xf, qx, sc[0:1])
    fg.forge_quantize_e4m3(yf, qy, sc[1:2])
    torch.cuda.synchronize()
    cx, sx = oracle.quantize_e4m3(xf.cpu())
    assert float(sc[0]) == sx and np.array_equal(qx.view(torch.uint8).cpu().numpy(), cx)
    cy, sy = oracle.quantize_e4m3(yf.cpu())
    assert float(sc[1]) == sy and np.array_equal(qy.view(torch.uint8).cpu().numpy(), cy)
    n_cols = 256
    dW = torch.empty((n_cols, M), device=dev)
    fg.forge_wgrad_only(qx[:, :n_cols].contiguous(), qy, dW, scales=sc)
    torch.cuda.synchronize()
    rows = [0, 77, 255]
    G = oracle.wgrad(np.ascontiguousarray(cx[:, :n_cols]), cy, scales=(sx, sy), rows=rows)
    check_dw(dW[rows].cpu().numpy(), G, "e4m3")

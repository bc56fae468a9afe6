"""C-ABI contract tests that need no GPU.

The library must load on a machine without a GPU, export every function
that include/forge.h declares, and reject invalid arguments with the
documented status codes before making any CUDA call (the pages' fail-closed
pattern: a GPU evidence command exits red on a missing or wrong device).
"""
import ctypes
import os
import re

import pytest

import weight_grad_gemm_gb300 as fg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "forge.h")


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(fg.LIB_PATH):
        from weight_grad_gemm_gb300 import build
        build.build()
    return fg.lib()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"FORGE_API\s+[\w\s\*]+?\b(forge_\w+)\s*\(", text)


def test_header_declares_the_abi():
    names = declared_functions()
    assert set(names) == set(fg.EXPORTS)
    for n in ("forge_wgrad_adamw", "forge_wgrad_sgdm", "forge_wgrad_only",
              "forge_grouped_wgrad_adamw", "forge_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
    assert fg.forge_version() == 100


def test_status_strings(L):
    for code in range(-7, 1):
        s = fg.forge_status_string(code)
        assert isinstance(s, str) and s and s != "unknown status"
    assert fg.forge_status_string(-99) == "unknown status"


# A fake, never-dereferenced device address: every call below fails its host
# checks before any pointer is used.
FAKE = ctypes.c_void_p(0x10000)
HP = (1e-3, 0.9, 0.999, 1e-8, 0.01)


def adamw(L, X=FAKE, dY=FAKE, W=FAKE, m=FAKE, v=FAKE, M=64, N=64, K=64, it=fg.FORGE_BF16,
          st=fg.FORGE_F32, hp=HP, step=1, scales=None, fn="forge_wgrad_adamw"):
    return getattr(L, fn)(X, dY, W, m, v, M, N, K, it, st, *hp, step, scales, None)


@pytest.mark.parametrize("kw,code", [
    (dict(W=None), fg.FORGE_ERR_INVALID_ARG),
    (dict(m=None), fg.FORGE_ERR_INVALID_ARG),
    (dict(v=None), fg.FORGE_ERR_INVALID_ARG),
    (dict(X=None), fg.FORGE_ERR_INVALID_ARG),
    (dict(dY=None), fg.FORGE_ERR_INVALID_ARG),
    (dict(M=0), fg.FORGE_ERR_INVALID_ARG),
    (dict(N=-3), fg.FORGE_ERR_INVALID_ARG),
    (dict(K=-1), fg.FORGE_ERR_INVALID_ARG),
    (dict(M=1 << 31), fg.FORGE_ERR_INVALID_ARG),
    (dict(step=0), fg.FORGE_ERR_INVALID_ARG),
    (dict(it=fg.FORGE_F32), fg.FORGE_ERR_UNSUPPORTED_DTYPE),
    (dict(it=7), fg.FORGE_ERR_UNSUPPORTED_DTYPE),
    (dict(st=fg.FORGE_E4M3), fg.FORGE_ERR_UNSUPPORTED_DTYPE),
    (dict(it=fg.FORGE_E4M3), fg.FORGE_ERR_INVALID_ARG),           # e4m3 needs scales
    (dict(scales=FAKE), fg.FORGE_ERR_INVALID_ARG),               # bf16 takes no scales
    (dict(hp=(1e-3, 1.0, 0.999, 1e-8, 0.01)), fg.FORGE_ERR_INVALID_ARG),
    (dict(hp=(1e-3, 0.9, -0.1, 1e-8, 0.01)), fg.FORGE_ERR_INVALID_ARG),
    (dict(hp=(float("nan"), 0.9, 0.999, 1e-8, 0.01)), fg.FORGE_ERR_INVALID_ARG),
    (dict(hp=(1e-3, 0.9, 0.999, -1.0, 0.01)), fg.FORGE_ERR_INVALID_ARG),
    (dict(hp=(1e-3, 0.9, 0.999, 1e-8, float("inf"))), fg.FORGE_ERR_INVALID_ARG),
])
@pytest.mark.parametrize("fn", ["forge_wgrad_adamw", "forge_wgrad_adamw_noalloc"])
def test_adamw_rejects_invalid_arguments(L, kw, code, fn):
    assert adamw(L, fn=fn, **kw) == code


def test_sgdm_and_wgrad_only_reject_invalid_arguments(L):
    assert L.forge_wgrad_sgdm(FAKE, FAKE, None, FAKE, 8, 8, 8, 0, 2, 1e-2, 0.9, 0.0, None,
                              None) == fg.FORGE_ERR_INVALID_ARG
    assert L.forge_wgrad_sgdm(FAKE, FAKE, FAKE, FAKE, 8, 8, 8, 0, 2, 1e-2, -0.9, 0.0, None,
                              None) == fg.FORGE_ERR_INVALID_ARG
    assert L.forge_wgrad_sgdm(FAKE, FAKE, FAKE, FAKE, 8, 8, 8, 0, 1, 1e-2, 0.9, 0.0, None,
                              None) == fg.FORGE_ERR_UNSUPPORTED_DTYPE
    assert L.forge_wgrad_only(FAKE, FAKE, None, 8, 8, 8, 0, None, None) == fg.FORGE_ERR_INVALID_ARG
    assert L.forge_wgrad_only(FAKE, FAKE, FAKE, 8, 0, 8, 0, None, None) == fg.FORGE_ERR_INVALID_ARG
    assert L.forge_wgrad_only(FAKE, FAKE, FAKE, 8, 8, 8, 3, None, None) == \
        fg.FORGE_ERR_UNSUPPORTED_DTYPE


def test_grouped_rejects_invalid_arguments(L):
    def g(offs=FAKE, E=4, T=64, step=1):
        return L.forge_grouped_wgrad_adamw(FAKE, FAKE, FAKE, FAKE, FAKE, offs, E, T, 64, 64, 0, 2,
                                           *HP, step, None, None)
    assert g(offs=None) == fg.FORGE_ERR_INVALID_ARG
    assert g(E=0) == fg.FORGE_ERR_INVALID_ARG
    assert g(E=1025) == fg.FORGE_ERR_INVALID_ARG
    assert g(T=-1) == fg.FORGE_ERR_INVALID_ARG
    assert g(step=0) == fg.FORGE_ERR_INVALID_ARG


def multi(L, P=3, M=(64, 32, 72), dY=FAKE, W=FAKE, null_entry=None, N=64, K=64,
          it=fg.FORGE_BF16, st=fg.FORGE_F32, hp=HP, step=1, arrays=True):
    arr = ctypes.c_void_p * 8
    d = arr(*([dY] * 8))
    w, m, v = arr(*([W] * 8)), arr(*([FAKE] * 8)), arr(*([FAKE] * 8))
    if null_entry is not None:
        {"dY": d, "W": w, "m": m, "v": v}[null_entry][1] = None
    ms = (ctypes.c_int64 * 8)(*(list(M) + [64] * (8 - len(M))))
    return L.forge_wgrad_adamw_multi(FAKE, N, K, P, d if arrays else None, ms, w, m, v, it, st,
                                     *hp, step, None)


def test_multi_rejects_invalid_arguments(L):
    assert multi(L, P=0) == fg.FORGE_ERR_INVALID_ARG
    assert multi(L, P=9) == fg.FORGE_ERR_INVALID_ARG
    assert multi(L, arrays=False) == fg.FORGE_ERR_INVALID_ARG
    for which in ("dY", "W", "m", "v"):
        assert multi(L, null_entry=which) == fg.FORGE_ERR_INVALID_ARG
    assert multi(L, M=(64, 0, 72)) == fg.FORGE_ERR_INVALID_ARG
    assert multi(L, N=0) == fg.FORGE_ERR_INVALID_ARG
    assert multi(L, K=-1) == fg.FORGE_ERR_INVALID_ARG
    assert multi(L, step=0) == fg.FORGE_ERR_INVALID_ARG
    assert multi(L, hp=(1e-3, 0.9, 1.0, 1e-8, 0.01)) == fg.FORGE_ERR_INVALID_ARG
    assert multi(L, it=fg.FORGE_E4M3) == fg.FORGE_ERR_UNSUPPORTED_DTYPE
    assert multi(L, st=fg.FORGE_E4M3) == fg.FORGE_ERR_UNSUPPORTED_DTYPE


def test_quantize_rejects_invalid_arguments(L):
    def q(x=FAKE, dt=fg.FORGE_F32, n=64, codes=FAKE, scale=FAKE):
        return L.forge_quantize_e4m3(x, dt, n, codes, scale, None)
    assert q(n=-1) == fg.FORGE_ERR_INVALID_ARG
    assert q(scale=None) == fg.FORGE_ERR_INVALID_ARG
    assert q(x=None) == fg.FORGE_ERR_INVALID_ARG
    assert q(codes=None) == fg.FORGE_ERR_INVALID_ARG
    assert q(dt=fg.FORGE_E4M3) == fg.FORGE_ERR_UNSUPPORTED_DTYPE
    assert q(x=ctypes.c_void_p(0x10002)) == fg.FORGE_ERR_MISALIGNED
    assert q(scale=ctypes.c_void_p(0x10001)) == fg.FORGE_ERR_MISALIGNED


def test_dgrad_and_backward_reject_invalid_arguments(L):
    def d(dY=FAKE, Wb=FAKE, dX=FAKE, M=64, N=64, K=64, dt=fg.FORGE_BF16):
        return L.forge_dgrad(dY, Wb, dX, M, N, K, dt, None)
    assert d(Wb=None) == fg.FORGE_ERR_INVALID_ARG
    assert d(dX=None) == fg.FORGE_ERR_INVALID_ARG
    assert d(M=0) == fg.FORGE_ERR_INVALID_ARG
    assert d(K=-1) == fg.FORGE_ERR_INVALID_ARG
    assert d(dt=fg.FORGE_E4M3) == fg.FORGE_ERR_UNSUPPORTED_DTYPE
    assert d(Wb=ctypes.c_void_p(0x10001)) == fg.FORGE_ERR_MISALIGNED  # not bf16-aligned
    assert d(dY=ctypes.c_void_p(0x10003)) == fg.FORGE_ERR_MISALIGNED

    def b(W=FAKE, Wb=FAKE, hp=HP, step=1, dt=fg.FORGE_BF16, st=fg.FORGE_F32):
        return L.forge_backward_adamw(FAKE, FAKE, W, FAKE, FAKE, Wb, FAKE, 64, 64, 64, dt, st,
                                      *hp, step, None)
    assert b(W=None) == fg.FORGE_ERR_INVALID_ARG
    assert b(step=0) == fg.FORGE_ERR_INVALID_ARG
    assert b(hp=(1e-3, 1.5, 0.999, 1e-8, 0.0)) == fg.FORGE_ERR_INVALID_ARG
    assert b(dt=fg.FORGE_E4M3) == fg.FORGE_ERR_UNSUPPORTED_DTYPE
    assert b(st=fg.FORGE_E4M3) == fg.FORGE_ERR_UNSUPPORTED_DTYPE
    assert b(W=ctypes.c_void_p(0x10002)) == fg.FORGE_ERR_MISALIGNED


def test_owner_steps_reject_invalid_arguments(L):
    def o(G=FAKE, W=FAKE, m=FAKE, v=FAKE, n=64, st=fg.FORGE_F32, hp=HP, step=1):
        return L.forge_owner_adamw(G, W, m, v, n, st, *hp, step, None)
    assert o(n=-1) == fg.FORGE_ERR_INVALID_ARG
    assert o(G=None) == fg.FORGE_ERR_INVALID_ARG
    assert o(v=None) == fg.FORGE_ERR_INVALID_ARG
    assert o(step=0) == fg.FORGE_ERR_INVALID_ARG
    assert o(hp=(1e-3, 0.9, 1.0, 1e-8, 0.0)) == fg.FORGE_ERR_INVALID_ARG
    assert o(st=fg.FORGE_E4M3) == fg.FORGE_ERR_UNSUPPORTED_DTYPE

    def sg(G=FAKE, W=FAKE, mom=FAKE, n=64, st=fg.FORGE_F32, lr=1e-2, mu=0.9, wd=0.0):
        return L.forge_owner_sgdm(G, W, mom, n, st, lr, mu, wd, None)
    assert sg(mom=None) == fg.FORGE_ERR_INVALID_ARG
    assert sg(lr=-1.0) == fg.FORGE_ERR_INVALID_ARG
    assert sg(mu=float("nan")) == fg.FORGE_ERR_INVALID_ARG
    assert sg(st=fg.FORGE_BF16 + 7) == fg.FORGE_ERR_UNSUPPORTED_DTYPE


def test_selftest_rejects_bad_limit(L):
    assert L.forge_selftest_wait_timeout(0, None) == fg.FORGE_ERR_INVALID_ARG


def test_valid_call_without_gpu_fails_closed(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; the fake pointers must not reach a kernel")
    assert adamw(L) == fg.FORGE_ERR_UNSUPPORTED_DEVICE
    assert adamw(L, fn="forge_wgrad_adamw_noalloc") == fg.FORGE_ERR_UNSUPPORTED_DEVICE
    assert multi(L) == fg.FORGE_ERR_UNSUPPORTED_DEVICE
    assert L.forge_dgrad(FAKE, FAKE, FAKE, 64, 64, 64, fg.FORGE_BF16, None) == \
        fg.FORGE_ERR_UNSUPPORTED_DEVICE
    assert L.forge_dgrad(FAKE, FAKE, FAKE, 60, 64, 64, fg.FORGE_BF16, None) == \
        fg.FORGE_ERR_UNSUPPORTED_DEVICE  # 120-byte rows are accepted (staged)
    assert L.forge_owner_adamw(FAKE, FAKE, FAKE, FAKE, 64, fg.FORGE_F32, *HP, 1, None) == \
        fg.FORGE_ERR_UNSUPPORTED_DEVICE
    assert fg.forge_get_device_status() == fg.FORGE_ERR_UNSUPPORTED_DEVICE

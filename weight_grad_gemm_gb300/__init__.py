"""Python binding for libforge.so: the fused weight-gradient GEMM + optimizer.

Thin ctypes marshalling over the C ABI declared in ``include/forge.h``; the
functions carry the same names.  Tensors are torch CUDA tensors; sizes are
taken from their shapes, pointers from ``data_ptr()`` and the stream from the
current torch stream unless one is given.  Every step of the computation runs
in the library's CUDA kernels: there is no CPU or PyTorch fallback, and
importing a function fails loudly if ``libforge.so`` has not been built
(``python -m weight_grad_gemm_gb300.build``).

Layouts: X [K, N] (tokens x d_in), dY [K, M] (tokens x d_out), W / m / v /
dW [N, M] (d_in x d_out), all contiguous; grouped: W / m / v [E, N, M] and
int32 offsets [E+1] on the device.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libforge.so")

FORGE_OK = 0
FORGE_ERR_INVALID_ARG = -1
FORGE_ERR_UNSUPPORTED_DTYPE = -2
FORGE_ERR_UNSUPPORTED_DEVICE = -3
FORGE_ERR_MISALIGNED = -4
FORGE_ERR_CUDA = -5
FORGE_ERR_TIMEOUT = -6
FORGE_ERR_SCRATCH_TOO_SMALL = -7

FORGE_BF16 = 0
FORGE_E4M3 = 1
FORGE_F32 = 2

EXPORTS = ("forge_wgrad_adamw", "forge_wgrad_adamw_noalloc", "forge_wgrad_adamw_multi",
           "forge_wgrad_sgdm", "forge_wgrad_only",
           "forge_quantize_e4m3", "forge_dgrad", "forge_backward_adamw",
           "forge_grouped_wgrad_adamw", "forge_owner_adamw", "forge_owner_sgdm",
           "forge_status_string", "forge_get_device_status",
           "forge_selftest_wait_timeout", "forge_version")


class ForgeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {forge_status_string(status)} ({status})")


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libforge.so with argument types set (raw C calls)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built: run `python -m weight_grad_gemm_gb300.build`")
    L = ctypes.CDLL(LIB_PATH)
    P, I64, I32, F, I = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float,
                         ctypes.c_int)
    L.forge_wgrad_adamw.argtypes = [P, P, P, P, P, I64, I64, I64, I, I, F, F, F, F, F, I64, P, P]
    L.forge_wgrad_adamw_noalloc.argtypes = L.forge_wgrad_adamw.argtypes
    L.forge_wgrad_adamw_multi.argtypes = [P, I64, I64, I32, P, P, P, P, P, I, I, F, F, F, F, F,
                                          I64, P]
    L.forge_quantize_e4m3.argtypes = [P, I, I64, P, P, P]
    L.forge_dgrad.argtypes = [P, P, P, I64, I64, I64, I, P]
    L.forge_backward_adamw.argtypes = [P, P, P, P, P, P, P, I64, I64, I64, I, I, F, F, F, F, F,
                                       I64, P]
    L.forge_wgrad_sgdm.argtypes = [P, P, P, P, I64, I64, I64, I, I, F, F, F, P, P]
    L.forge_wgrad_only.argtypes = [P, P, P, I64, I64, I64, I, P, P]
    L.forge_grouped_wgrad_adamw.argtypes = [P, P, P, P, P, P, I32, I64, I64, I64, I, I, F, F, F,
                                            F, F, I64, P, P]
    L.forge_owner_adamw.argtypes = [P, P, P, P, I64, I, F, F, F, F, F, I64, P]
    L.forge_owner_sgdm.argtypes = [P, P, P, I64, I, F, F, F, P]
    for f in ("forge_wgrad_adamw", "forge_wgrad_adamw_noalloc", "forge_wgrad_adamw_multi",
              "forge_wgrad_sgdm",
              "forge_wgrad_only", "forge_quantize_e4m3", "forge_dgrad", "forge_backward_adamw",
              "forge_grouped_wgrad_adamw", "forge_owner_adamw", "forge_owner_sgdm",
              "forge_get_device_status",
              "forge_selftest_wait_timeout"):
        getattr(L, f).restype = I
    L.forge_status_string.argtypes = [I]
    L.forge_status_string.restype = ctypes.c_char_p
    L.forge_get_device_status.argtypes = []
    L.forge_selftest_wait_timeout.argtypes = [ctypes.c_uint32, P]
    L.forge_version.argtypes = []
    L.forge_version.restype = I32
    _lib = L
    return L


# ---- marshalling helpers ---------------------------------------------------

def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return FORGE_BF16
    if t.dtype == torch.float8_e4m3fn:
        return FORGE_E4M3
    if t.dtype == torch.float32:
        return FORGE_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream, like):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(like.device)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status: int, where: str):
    if status != FORGE_OK:
        raise ForgeError(status, where)


def _sizes(X, dY):
    if X.dim() != 2 or dY.dim() != 2 or X.shape[0] != dY.shape[0]:
        raise ValueError(f"X [K, N] and dY [K, M] expected, got {tuple(X.shape)}, {tuple(dY.shape)}")
    return dY.shape[1], X.shape[1], X.shape[0]  # M, N, K


def _scales_ptr(scales, X):
    if scales is None:
        return None
    import torch
    if scales.dtype != torch.float32 or scales.numel() != 2:
        raise ValueError("scales must be a float32 tensor [sX, sdY]")
    return _ptr(scales)


# ---- the C ABI, tensor form ------------------------------------------------

def _adamw_call(name, X, dY, W, m, v, lr, beta1, beta2, eps, wd, step, scales, stream):
    M, N, K = _sizes(X, dY)
    for t in (W, m, v):
        if tuple(t.shape) != (N, M):
            raise ValueError(f"W/m/v must be [N={N}, M={M}], got {tuple(t.shape)}")
    if m.dtype != v.dtype:
        raise TypeError("m and v must share a dtype")
    s = getattr(lib(), name)(_ptr(X), _ptr(dY), _ptr(W), _ptr(m), _ptr(v), M, N, K,
                             _dtype_code(X), _dtype_code(m), lr, beta1, beta2, eps, wd,
                             int(step), _scales_ptr(scales, X), _stream(stream, W))
    _check(s, name)


def forge_wgrad_adamw(X, dY, W, m, v, *, lr, beta1, beta2, eps, wd, step, scales=None,
                      stream=None):
    _adamw_call("forge_wgrad_adamw", X, dY, W, m, v, lr, beta1, beta2, eps, wd, step, scales,
                stream)


def forge_wgrad_adamw_noalloc(X, dY, W, m, v, *, lr, beta1, beta2, eps, wd, step, scales=None,
                              stream=None):
    """forge_wgrad_adamw staging misaligned operands into the library's fixed
    per-device buffer instead of allocating (see include/forge.h)."""
    _adamw_call("forge_wgrad_adamw_noalloc", X, dY, W, m, v, lr, beta1, beta2, eps, wd, step,
                scales, stream)


def forge_wgrad_adamw_multi(X, dYs, Ws, ms, vs, *, lr, beta1, beta2, eps, wd, step,
                            stream=None):
    """One launch of forge_wgrad_adamw for each (dY, W, m, v) of the lists, all
    with the same X (see include/forge.h)."""
    n = len(dYs)
    if not (len(Ws) == len(ms) == len(vs) == n):
        raise ValueError("dYs, Ws, ms, vs must have one entry per problem")
    sizes = [_sizes(X, d) for d in dYs]
    N, K = X.shape[1], X.shape[0]
    for (M, _, _), W, m, v in zip(sizes, Ws, ms, vs):
        for t in (W, m, v):
            if tuple(t.shape) != (N, M):
                raise ValueError(f"W/m/v must be [N={N}, M={M}], got {tuple(t.shape)}")
        if m.dtype != v.dtype or m.dtype != ms[0].dtype:
            raise TypeError("every m and v must share one dtype")
        if X.dtype != dYs[0].dtype:
            raise TypeError("X and every dY must share one dtype")
    arr = ctypes.c_void_p * max(n, 1)
    dptr = arr(*[_ptr(d).value for d in dYs])
    wptr = arr(*[_ptr(t).value for t in Ws])
    mptr = arr(*[_ptr(t).value for t in ms])
    vptr = arr(*[_ptr(t).value for t in vs])
    mlen = (ctypes.c_int64 * max(n, 1))(*[M for M, _, _ in sizes])
    s = lib().forge_wgrad_adamw_multi(_ptr(X), N, K, n, dptr, mlen, wptr, mptr, vptr,
                                      _dtype_code(X), _dtype_code(ms[0]), lr, beta1, beta2, eps,
                                      wd, int(step), _stream(stream, Ws[0]))
    _check(s, "forge_wgrad_adamw_multi")


def forge_wgrad_sgdm(X, dY, W, mom, *, lr, momentum, wd, scales=None, stream=None):
    M, N, K = _sizes(X, dY)
    for t in (W, mom):
        if tuple(t.shape) != (N, M):
            raise ValueError(f"W/mom must be [N={N}, M={M}], got {tuple(t.shape)}")
    s = lib().forge_wgrad_sgdm(_ptr(X), _ptr(dY), _ptr(W), _ptr(mom), M, N, K, _dtype_code(X),
                               _dtype_code(mom), lr, momentum, wd, _scales_ptr(scales, X),
                               _stream(stream, W))
    _check(s, "forge_wgrad_sgdm")


def forge_wgrad_only(X, dY, dW, *, scales=None, stream=None):
    M, N, K = _sizes(X, dY)
    if tuple(dW.shape) != (N, M):
        raise ValueError(f"dW must be [N={N}, M={M}], got {tuple(dW.shape)}")
    s = lib().forge_wgrad_only(_ptr(X), _ptr(dY), _ptr(dW), M, N, K, _dtype_code(X),
                               _scales_ptr(scales, X), _stream(stream, dW))
    _check(s, "forge_wgrad_only")


def forge_quantize_e4m3(x, codes, scale, *, stream=None):
    """codes (uint8 or float8_e4m3fn, x.numel() elements) and scale (float32
    [1]) from x (float32 or bfloat16): s = amax / 448, codes = nearest e4m3 of
    x / s."""
    import torch
    if codes.numel() != x.numel() or codes.element_size() != 1:
        raise ValueError("codes must hold one byte per element of x")
    if scale.dtype != torch.float32 or scale.numel() != 1:
        raise ValueError("scale must be a float32 tensor of one element")
    s = lib().forge_quantize_e4m3(_ptr(x), _dtype_code(x), x.numel(), _ptr(codes), _ptr(scale),
                                  _stream(stream, codes))
    _check(s, "forge_quantize_e4m3")


def forge_dgrad(dY, Wb, dX, *, stream=None):
    """dX [K, N] (bf16) = dY [K, M] (bf16) times Wb [N, M] (bf16) transposed."""
    K, M = dY.shape
    N = Wb.shape[0]
    if Wb.dim() != 2 or Wb.shape[1] != M or tuple(dX.shape) != (K, N):
        raise ValueError(f"dY [K, M], Wb [N, M], dX [K, N] expected, got {tuple(dY.shape)}, "
                         f"{tuple(Wb.shape)}, {tuple(dX.shape)}")
    s = lib().forge_dgrad(_ptr(dY), _ptr(Wb), _ptr(dX), M, N, K, _dtype_code(dY),
                          _stream(stream, dX))
    _check(s, "forge_dgrad")


def forge_backward_adamw(X, dY, W, m, v, dX, *, lr, beta1, beta2, eps, wd, step, Wb=None,
                         stream=None):
    """dX = dY Wb^T, then the fused dW + AdamW on W, m, v, in that order on one
    stream.  Wb: the bf16 copy of W the forward used, or None to have W
    rounded to bf16 first."""
    M, N, K = _sizes(X, dY)
    for t in (W, m, v):
        if tuple(t.shape) != (N, M):
            raise ValueError(f"W/m/v must be [N={N}, M={M}], got {tuple(t.shape)}")
    if tuple(dX.shape) != (K, N) or (Wb is not None and tuple(Wb.shape) != (N, M)):
        raise ValueError("dX must be [K, N] and Wb [N, M]")
    if m.dtype != v.dtype:
        raise TypeError("m and v must share a dtype")
    s = lib().forge_backward_adamw(_ptr(X), _ptr(dY), _ptr(W), _ptr(m), _ptr(v), _ptr(Wb),
                                   _ptr(dX), M, N, K, _dtype_code(X), _dtype_code(m), lr, beta1,
                                   beta2, eps, wd, int(step), _stream(stream, W))
    _check(s, "forge_backward_adamw")


def forge_grouped_wgrad_adamw(X, dY, W, m, v, offsets, *, lr, beta1, beta2, eps, wd, step,
                              scales=None, stream=None):
    import torch
    M, N, T = _sizes(X, dY)
    E = offsets.numel() - 1
    if offsets.dtype != torch.int32 or E < 1:
        raise ValueError("offsets must be int32 [E+1] with E >= 1")
    for t in (W, m, v):
        if tuple(t.shape) != (E, N, M):
            raise ValueError(f"W/m/v must be [E={E}, N={N}, M={M}], got {tuple(t.shape)}")
    s = lib().forge_grouped_wgrad_adamw(_ptr(X), _ptr(dY), _ptr(W), _ptr(m), _ptr(v),
                                        _ptr(offsets), E, T, M, N, _dtype_code(X),
                                        _dtype_code(m), lr, beta1, beta2, eps, wd, int(step),
                                        _scales_ptr(scales, X), _stream(stream, W))
    _check(s, "forge_grouped_wgrad_adamw")


def _same_numel(G, *ts):
    for t in ts:
        if t.numel() != G.numel():
            raise ValueError(f"gradient shard and state must have one element each, got "
                             f"{G.numel()} and {t.numel()}")


def forge_owner_adamw(G, W, m, v, *, lr, beta1, beta2, eps, wd, step, stream=None):
    """The owner's AdamW step on its shard: G (fp32, the reduce-scattered sum
    of the ranks' partial dW), W (fp32), m, v (fp32 or bf16), all of one
    shape, updated in place (see include/forge.h)."""
    import torch
    _same_numel(G, W, m, v)
    if G.dtype != torch.float32 or W.dtype != torch.float32 or m.dtype != v.dtype:
        raise TypeError("G and W must be float32, m and v one dtype")
    s = lib().forge_owner_adamw(_ptr(G), _ptr(W), _ptr(m), _ptr(v), G.numel(), _dtype_code(m),
                                lr, beta1, beta2, eps, wd, int(step), _stream(stream, W))
    _check(s, "forge_owner_adamw")


def forge_owner_sgdm(G, W, mom, *, lr, momentum, wd, stream=None):
    """The owner's SGD-momentum step on its shard (see forge_owner_adamw)."""
    import torch
    _same_numel(G, W, mom)
    if G.dtype != torch.float32 or W.dtype != torch.float32:
        raise TypeError("G and W must be float32")
    s = lib().forge_owner_sgdm(_ptr(G), _ptr(W), _ptr(mom), G.numel(), _dtype_code(mom), lr,
                               momentum, wd, _stream(stream, W))
    _check(s, "forge_owner_sgdm")


def forge_status_string(status: int) -> str:
    return lib().forge_status_string(int(status)).decode()


def forge_get_device_status() -> int:
    return int(lib().forge_get_device_status())


def forge_selftest_wait_timeout(timeout_us: int, stream=None):
    import torch
    st = stream if stream is not None else torch.cuda.current_stream()
    _check(lib().forge_selftest_wait_timeout(int(timeout_us), ctypes.c_void_p(st.cuda_stream)),
           "forge_selftest_wait_timeout")


def forge_version() -> int:
    return int(lib().forge_version())

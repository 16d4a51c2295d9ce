"""libna: GB300-native multi-dimensional neighborhood attention (NA), forward and backward.

A thin ctypes binding over the C ABI in include/na.h: every function takes torch tensors that
already live on the GPU, checks shapes, and passes raw device pointers, sizes and the current CUDA
stream to the library.  All arithmetic runs in the library's CUDA kernels (tcgen05 tensor-core
kernels for bf16, CUDA-core FMA kernels for fp32); there is no fallback of any kind, and a missing
library raises.

Tensors are contiguous [B, L_1, .., L_n, heads, D] (n = 1..3); lse/delta are fp32 [B, L.., heads].
The unfused operations (na_qk, na_softmax, na_av and their gradients) keep the attention weights
as [B, L.., heads, K], K = the product of the kernel sizes, window offsets first axis outermost.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

__all__ = [
    "NAError", "load", "na_fwd", "na_bwd", "na_bwd_delta", "na_bwd_dq", "na_bwd_dkdv",
    "na_bwd_workspace_size", "na_device_status", "na_strerror", "na_plan_info", "library_path",
    "na_qk", "na_av", "na_softmax", "na_softmax_bwd", "na_qk_bwd", "na_av_bwd", "na_rpb_grad",
    "na_rpb_grad_workspace_size", "na_mask_window", "na_debug_wait_hook",
]

NA_BF16, NA_FP32, NA_FP16 = 0, 1, 2
_STATUS = {0: "NA_OK", 1: "NA_ERR_INVALID_ARG", 2: "NA_ERR_UNSUPPORTED", 3: "NA_ERR_ALIGNMENT",
           4: "NA_ERR_CUDA", 5: "NA_ERR_TIMEOUT", 6: "NA_ERR_WORKSPACE"}

_lib = None


class NAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_STATUS.get(status, status)} ({na_strerror(status)})")


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load libna.so (built by neighborhood_attention_fwd_gb300.build.build()); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"libna.so not found at {path}: run neighborhood_attention_fwd_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    IP = ctypes.POINTER(ctypes.c_int)
    geo = [I, I, IP, I, I]                   # B, ndim, spatial, heads, D
    kd = [IP, IP, F]                         # kernel, dilation, scale
    geo_nd = [I, I, IP, I]                   # B, ndim, spatial, heads
    lib.na_fwd.argtypes = [P, P, P, P, P] + geo + kd + [I, P]
    lib.na_bwd.argtypes = [P, P, P, P, P, P, P, P, P] + geo + kd + [I, P, ctypes.c_size_t, P]
    lib.na_bwd_delta.argtypes = [P, P, P] + geo + [I, P]
    lib.na_bwd_dq.argtypes = [P, P, P, P, P, P, P] + geo + kd + [I, P]
    lib.na_bwd_dkdv.argtypes = [P, P, P, P, P, P, P, P] + geo + kd + [I, P]
    lib.na_bwd_workspace_size.argtypes = [I, I, IP, I]
    lib.na_bwd_workspace_size.restype = ctypes.c_size_t
    lib.na_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
    lib.na_debug_wait_hook.argtypes = [ctypes.c_ulonglong, I]
    lib.na_strerror.argtypes = [I]
    lib.na_strerror.restype = ctypes.c_char_p
    lib.na_plan_info.argtypes = [I, I, I, IP, I, I, IP, IP, ctypes.POINTER(ctypes.c_int64)]
    lib.na_qk.argtypes = [P, P, P, P] + geo + kd + [I, P]
    lib.na_rpb_grad.argtypes = [P, P] + geo_nd + [IP, IP, I, P, ctypes.c_size_t, P]
    lib.na_rpb_grad_workspace_size.argtypes = [I, I, IP, I, IP]
    lib.na_rpb_grad_workspace_size.restype = ctypes.c_size_t
    lib.na_mask_window.argtypes = [P, P] + geo_nd + [IP, IP, I, P]
    lib.na_av.argtypes = [P, P, P] + geo + [IP, IP, I, P]
    lib.na_softmax.argtypes = [P, P] + geo_nd + [IP, I, P]
    lib.na_softmax_bwd.argtypes = [P, P, P] + geo_nd + [IP, I, P]
    lib.na_qk_bwd.argtypes = [P, P, P, P, P] + geo + kd + [I, P]
    lib.na_av_bwd.argtypes = [P, P, P, P, P] + geo + [IP, IP, I, P]
    for f in ("na_fwd", "na_bwd", "na_bwd_delta", "na_bwd_dq", "na_bwd_dkdv", "na_device_status", "na_plan_info",
              "na_qk", "na_av", "na_softmax", "na_softmax_bwd", "na_qk_bwd", "na_av_bwd", "na_rpb_grad",
              "na_mask_window"):
        getattr(lib, f).restype = I
    _lib = lib
    return lib


def na_strerror(status: int) -> str:
    return load().na_strerror(int(status)).decode()


def _ints(vals):
    vals = [int(x) for x in vals]
    return (ctypes.c_int * len(vals))(*vals)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return NA_BF16
    if t.dtype == torch.float32:
        return NA_FP32
    if t.dtype == torch.float16:
        return NA_FP16
    raise TypeError(f"unsupported dtype {t.dtype}: use bfloat16, float16 or float32")


def _geometry(q: torch.Tensor):
    if q.dim() < 4 or q.dim() > 6:
        raise ValueError("expected [B, L_1..L_n, heads, D] with n in 1..3")
    B = q.shape[0]
    spatial = tuple(int(s) for s in q.shape[1:-2])
    return B, len(spatial), spatial, int(q.shape[-2]), int(q.shape[-1])


def _check(t: torch.Tensor, shape, dtype, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype:
        raise ValueError(f"{name}: expected {tuple(shape)} {dtype}, got {tuple(t.shape)} {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ok(status: int, what: str):
    if status != 0:
        raise NAError(status, what)


def _kd(ndim, kernel, dilation):
    kernel = (kernel,) * ndim if isinstance(kernel, int) else tuple(kernel)
    dilation = (1,) * ndim if dilation is None else ((dilation,) * ndim if isinstance(dilation, int) else tuple(dilation))
    if len(kernel) != ndim or len(dilation) != ndim:
        raise ValueError("kernel and dilation need one entry per spatial axis")
    return kernel, dilation


def na_fwd(q, k, v, o, lse, kernel, dilation=None, scale=None, stream=None):
    """O = NA(q, k, v) and the natural-log LSE, written into o and lse."""
    B, ndim, spatial, heads, D = _geometry(q)
    for name, t in (("k", k), ("v", v), ("o", o)):
        _check(t, q.shape, q.dtype, name)
    _check(q, q.shape, q.dtype, "q")
    _check(lse, q.shape[:-1], torch.float32, "lse")
    kernel, dilation = _kd(ndim, kernel, dilation)
    scale = D ** -0.5 if scale is None else float(scale)
    st = load().na_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                       B, ndim, _ints(spatial), heads, D, _ints(kernel), _ints(dilation), scale,
                       _dtype_code(q), _stream(stream))
    _ok(st, "na_fwd")


def na_bwd_workspace_size(B, spatial, heads) -> int:
    return int(load().na_bwd_workspace_size(int(B), len(spatial), _ints(spatial), int(heads)))


def na_bwd(q, k, v, o, dO, lse, dQ, dK, dV, kernel, dilation=None, scale=None, workspace=None, stream=None):
    """dQ, dK, dV of NA for upstream gradient dO (Delta prologue + dQ pass + dK/dV pass)."""
    B, ndim, spatial, heads, D = _geometry(q)
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dO", dO), ("dQ", dQ), ("dK", dK), ("dV", dV)):
        _check(t, q.shape, q.dtype, name)
    _check(lse, q.shape[:-1], torch.float32, "lse")
    kernel, dilation = _kd(ndim, kernel, dilation)
    scale = D ** -0.5 if scale is None else float(scale)
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.data_ptr(), workspace.numel() * workspace.element_size())
    st = load().na_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dO.data_ptr(), lse.data_ptr(),
                       dQ.data_ptr(), dK.data_ptr(), dV.data_ptr(), B, ndim, _ints(spatial), heads, D,
                       _ints(kernel), _ints(dilation), scale, _dtype_code(q), ws_ptr, ws_bytes, _stream(stream))
    _ok(st, "na_bwd")


def na_bwd_delta(o, dO, delta, stream=None):
    """delta = <dO, O> per row (fp32)."""
    B, ndim, spatial, heads, D = _geometry(o)
    _check(dO, o.shape, o.dtype, "dO")
    _check(delta, o.shape[:-1], torch.float32, "delta")
    st = load().na_bwd_delta(o.data_ptr(), dO.data_ptr(), delta.data_ptr(), B, ndim, _ints(spatial), heads, D,
                             _dtype_code(o), _stream(stream))
    _ok(st, "na_bwd_delta")


def na_bwd_dq(q, k, v, dO, lse, delta, dQ, kernel, dilation=None, scale=None, stream=None):
    B, ndim, spatial, heads, D = _geometry(q)
    for name, t in (("k", k), ("v", v), ("dO", dO), ("dQ", dQ)):
        _check(t, q.shape, q.dtype, name)
    _check(lse, q.shape[:-1], torch.float32, "lse")
    _check(delta, q.shape[:-1], torch.float32, "delta")
    kernel, dilation = _kd(ndim, kernel, dilation)
    scale = D ** -0.5 if scale is None else float(scale)
    st = load().na_bwd_dq(q.data_ptr(), k.data_ptr(), v.data_ptr(), dO.data_ptr(), lse.data_ptr(), delta.data_ptr(),
                          dQ.data_ptr(), B, ndim, _ints(spatial), heads, D, _ints(kernel), _ints(dilation), scale,
                          _dtype_code(q), _stream(stream))
    _ok(st, "na_bwd_dq")


def na_bwd_dkdv(q, k, v, dO, lse, delta, dK, dV, kernel, dilation=None, scale=None, stream=None):
    B, ndim, spatial, heads, D = _geometry(q)
    for name, t in (("k", k), ("v", v), ("dO", dO), ("dK", dK), ("dV", dV)):
        _check(t, q.shape, q.dtype, name)
    _check(lse, q.shape[:-1], torch.float32, "lse")
    _check(delta, q.shape[:-1], torch.float32, "delta")
    kernel, dilation = _kd(ndim, kernel, dilation)
    scale = D ** -0.5 if scale is None else float(scale)
    st = load().na_bwd_dkdv(q.data_ptr(), k.data_ptr(), v.data_ptr(), dO.data_ptr(), lse.data_ptr(),
                            delta.data_ptr(), dK.data_ptr(), dV.data_ptr(), B, ndim, _ints(spatial), heads, D,
                            _ints(kernel), _ints(dilation), scale, _dtype_code(q), _stream(stream))
    _ok(st, "na_bwd_dkdv")


def na_device_status(stream=None):
    """Synchronise the stream and return (status, raw status word); clears the word."""
    raw = ctypes.c_uint32(0)
    st = load().na_device_status(_stream(stream), ctypes.byref(raw))
    return int(st), int(raw.value)


def na_debug_wait_hook(limit_ns: int = 0, withhold: bool = False) -> None:
    """Test hook: the wait limit of later tensor-core launches (0: the 2 s default) and, with
    withhold, the first CTA's first halo chunk left unfilled so that a wait runs out."""
    _ok(load().na_debug_wait_hook(int(limit_ns), 1 if withhold else 0), "na_debug_wait_hook")


PLAN_FIELDS = ("T1", "T2", "T3", "H1", "H2", "H3", "G1", "G2", "G3", "NC", "chunks_max", "ctas", "mma_flops",
               "tmem_cols", "smem_bytes", "chunks_total")


def na_plan_info(which: int, B, spatial, heads, D, kernel, dilation=None) -> dict:
    """Tile plan of the bf16 kernel `which` (0 forward, 1 dQ, 2 dK/dV) for this problem."""
    ndim = len(spatial)
    kernel, dilation = _kd(ndim, kernel, dilation)
    out = (ctypes.c_int64 * 16)()
    st = load().na_plan_info(int(which), int(B), ndim, _ints(spatial), int(heads), int(D), _ints(kernel),
                             _ints(dilation), out)
    _ok(st, "na_plan_info")
    return dict(zip(PLAN_FIELDS, [int(x) for x in out]))


# ---------------------------------------------------------------------------------------------
# Unfused operations: logits, window softmax, weighted sum, and their gradients
# ---------------------------------------------------------------------------------------------

def _window_size(kernel) -> int:
    n = 1
    for x in kernel:
        n *= int(x)
    return n


def _attn_geometry(attn: torch.Tensor, kernel):
    """B, ndim, spatial, heads of an attention-weight tensor [B, L.., heads, K]."""
    if attn.dim() < 4 or attn.dim() > 6:
        raise ValueError("expected attention weights [B, L_1..L_n, heads, K] with n in 1..3")
    ndim = attn.dim() - 3
    kernel = (kernel,) * ndim if isinstance(kernel, int) else tuple(kernel)
    if len(kernel) != ndim:
        raise ValueError("kernel needs one entry per spatial axis")
    if int(attn.shape[-1]) != _window_size(kernel):
        raise ValueError(f"last axis of the attention weights must be {_window_size(kernel)}")
    return int(attn.shape[0]), ndim, tuple(int(s) for s in attn.shape[1:-2]), int(attn.shape[-2]), kernel


def _rpb_shape(heads, kernel):
    return (heads,) + tuple(2 * int(x) - 1 for x in kernel)


def na_qk(q, k, attn, kernel, dilation=None, scale=None, stream=None, rpb=None):
    """attn = scale * q . k over each query's window, plus the relative positional bias rpb (fp32
    [heads, 2k_0 - 1, ..]) when given."""
    B, ndim, spatial, heads, D = _geometry(q)
    _check(k, q.shape, q.dtype, "k")
    _check(q, q.shape, q.dtype, "q")
    kernel, dilation = _kd(ndim, kernel, dilation)
    _check(attn, tuple(q.shape[:-1]) + (_window_size(kernel),), q.dtype, "attn")
    if rpb is not None:
        _check(rpb, _rpb_shape(heads, kernel), torch.float32, "rpb")
    scale = D ** -0.5 if scale is None else float(scale)
    st = load().na_qk(q.data_ptr(), k.data_ptr(), None if rpb is None else rpb.data_ptr(), attn.data_ptr(), B,
                      ndim, _ints(spatial), heads, D, _ints(kernel), _ints(dilation), scale, _dtype_code(q),
                      _stream(stream))
    _ok(st, "na_qk")


def na_rpb_grad_workspace_size(B, spatial, heads, kernel) -> int:
    kernel = (kernel,) * len(spatial) if isinstance(kernel, int) else tuple(kernel)
    return int(load().na_rpb_grad_workspace_size(int(B), len(spatial), _ints(spatial), int(heads), _ints(kernel)))


def na_rpb_grad(dattn, drpb, kernel, dilation=None, workspace=None, stream=None):
    """drpb (fp32 [heads, 2k_0 - 1, ..]) = the bias table's gradient given the logits' gradient dattn."""
    B, ndim, spatial, heads, kernel = _attn_geometry(dattn, kernel)
    kernel, dilation = _kd(ndim, kernel, dilation)
    _check(dattn, dattn.shape, dattn.dtype, "dattn")
    _check(drpb, _rpb_shape(heads, kernel), torch.float32, "drpb")
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.data_ptr(), workspace.numel() * workspace.element_size())
    st = load().na_rpb_grad(dattn.data_ptr(), drpb.data_ptr(), B, ndim, _ints(spatial), heads, _ints(kernel),
                            _ints(dilation), _dtype_code(dattn), ws_ptr, ws_bytes, _stream(stream))
    _ok(st, "na_rpb_grad")


def na_av(attn, v, o, kernel, dilation=None, stream=None):
    """o = sum over each query's window of attn * v."""
    B, ndim, spatial, heads, D = _geometry(v)
    _check(v, v.shape, v.dtype, "v")
    _check(o, v.shape, v.dtype, "o")
    kernel, dilation = _kd(ndim, kernel, dilation)
    _check(attn, tuple(v.shape[:-1]) + (_window_size(kernel),), v.dtype, "attn")
    st = load().na_av(attn.data_ptr(), v.data_ptr(), o.data_ptr(), B, ndim, _ints(spatial), heads, D,
                      _ints(kernel), _ints(dilation), _dtype_code(v), _stream(stream))
    _ok(st, "na_av")


def na_softmax(x, y, kernel, stream=None):
    """y = softmax of x over each row's K window weights (y may be x)."""
    B, ndim, spatial, heads, kernel = _attn_geometry(x, kernel)
    _check(x, x.shape, x.dtype, "x")
    _check(y, x.shape, x.dtype, "y")
    st = load().na_softmax(x.data_ptr(), y.data_ptr(), B, ndim, _ints(spatial), heads, _ints(kernel),
                           _dtype_code(x), _stream(stream))
    _ok(st, "na_softmax")


def na_softmax_bwd(y, dy, dx, kernel, stream=None):
    """dx = y * (dy - sum_t y dy), the gradient of the window softmax given its output y."""
    B, ndim, spatial, heads, kernel = _attn_geometry(y, kernel)
    for name, t in (("y", y), ("dy", dy), ("dx", dx)):
        _check(t, y.shape, y.dtype, name)
    st = load().na_softmax_bwd(y.data_ptr(), dy.data_ptr(), dx.data_ptr(), B, ndim, _ints(spatial), heads,
                               _ints(kernel), _dtype_code(y), _stream(stream))
    _ok(st, "na_softmax_bwd")


def na_qk_bwd(dattn, q, k, dq, dk, kernel, dilation=None, scale=None, stream=None):
    """dq, dk of na_qk given the logits' gradient dattn."""
    B, ndim, spatial, heads, D = _geometry(q)
    for name, t in (("q", q), ("k", k), ("dq", dq), ("dk", dk)):
        _check(t, q.shape, q.dtype, name)
    kernel, dilation = _kd(ndim, kernel, dilation)
    _check(dattn, tuple(q.shape[:-1]) + (_window_size(kernel),), q.dtype, "dattn")
    scale = D ** -0.5 if scale is None else float(scale)
    st = load().na_qk_bwd(dattn.data_ptr(), q.data_ptr(), k.data_ptr(), dq.data_ptr(), dk.data_ptr(), B, ndim,
                          _ints(spatial), heads, D, _ints(kernel), _ints(dilation), scale, _dtype_code(q),
                          _stream(stream))
    _ok(st, "na_qk_bwd")


def na_av_bwd(dO, attn, v, dattn, dv, kernel, dilation=None, stream=None):
    """dattn, dv of na_av given the output's gradient dO."""
    B, ndim, spatial, heads, D = _geometry(v)
    for name, t in (("dO", dO), ("v", v), ("dv", dv)):
        _check(t, v.shape, v.dtype, name)
    kernel, dilation = _kd(ndim, kernel, dilation)
    K = _window_size(kernel)
    _check(attn, tuple(v.shape[:-1]) + (K,), v.dtype, "attn")
    _check(dattn, tuple(v.shape[:-1]) + (K,), v.dtype, "dattn")
    st = load().na_av_bwd(dO.data_ptr(), attn.data_ptr(), v.data_ptr(), dattn.data_ptr(), dv.data_ptr(), B, ndim,
                          _ints(spatial), heads, D, _ints(kernel), _ints(dilation), _dtype_code(v),
                          _stream(stream))
    _ok(st, "na_av_bwd")


def na_mask_window(attn, sizes, kernel, dilation=None, stream=None):
    """Set, in place, the logits outside each query's variable window to -inf.  sizes: one sequence or
    tensor per axis, sizes[a][x] = the kernel size (odd, <= kernel[a]) of the queries at position x."""
    B, ndim, spatial, heads, kernel = _attn_geometry(attn, kernel)
    kernel, dilation = _kd(ndim, kernel, dilation)
    _check(attn, attn.shape, attn.dtype, "attn")
    if len(sizes) != ndim:
        raise ValueError("sizes needs one entry per spatial axis")
    parts = [torch.as_tensor(sz, dtype=torch.int32, device="cpu").reshape(-1) for sz in sizes]
    for L, part in zip(spatial, parts):
        if part.numel() != L:
            raise ValueError("sizes[a] needs one entry per position along axis a")
    # a copy from pageable host memory has finished when .to() returns, so the sizes are in place
    # whichever stream the kernel runs on; the temporary must then outlive the launch on that stream
    flat = torch.cat(parts).contiguous().to(attn.device)
    st = load().na_mask_window(attn.data_ptr(), flat.data_ptr(), B, ndim, _ints(spatial), heads, _ints(kernel),
                               _ints(dilation), _dtype_code(attn), _stream(stream))
    _ok(st, "na_mask_window")
    if isinstance(stream, torch.cuda.Stream):
        flat.record_stream(stream)
    elif stream is not None:
        torch.cuda.ExternalStream(int(stream)).synchronize()

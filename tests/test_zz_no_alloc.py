"""na_bwd_noalloc: the backward entry point for callers that cannot allocate device memory.

Some callers cannot allocate while they run: for example, a host framework that owns all device
memory under a fixed budget, or a latency-critical loop that forbids allocations.  They cannot let
na_bwd allocate its Delta workspace.  na_bwd_noalloc keeps that scratch in a fixed device array
inside the library instead.  This file checks it through the C ABI against na_bwd (which receives a
caller-provided workspace here) on two calls in a row.  The second call has a different, smaller
shape, so stale scratch contents from the first call would show up as a mismatch.  The file is named
so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import neighborhood_attention_fwd_gb300 as na
from neighborhood_attention_fwd_gb300 import build as nabuild
from neighborhood_attention_fwd_gb300 import inputs as nain

NA_NOALLOC_MAX_ROWS = 8 * 1024 * 1024
NA_ERR_WORKSPACE = 6


def _lib():
    nabuild.build()
    lib = na.load()
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    IP = ctypes.POINTER(ctypes.c_int)
    lib.na_bwd_noalloc.argtypes = [P] * 9 + [I, I, IP, I, I, IP, IP, F, I, P]
    lib.na_bwd_noalloc.restype = I
    return lib


def _ints(v):
    return (ctypes.c_int * len(v))(*[int(x) for x in v])


def _call_noalloc(lib, w, t, o, lse, dq, dk, dv):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    dtype = 0 if w.dtype == "bf16" else 1
    return lib.na_bwd_noalloc(t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(), o.data_ptr(),
                              t["dO"].data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                              w.B, w.ndim, _ints(w.spatial), w.heads, w.D, _ints(w.kernel), _ints(w.dilation),
                              ctypes.c_float(w.scale), dtype, stream)


def _check(name, got, ref, tol):
    g, r = got.double().cpu().numpy(), ref.double().cpu().numpy()
    assert np.isfinite(g).all(), name
    bound = tol * max(np.abs(r).max(), 1e-30)
    assert np.abs(g - r).max() <= bound, f"{name}: {np.abs(g - r).max():.3e} > {bound:.3e}"


@pytest.mark.gpu
def test_noalloc_backward_matches_na_bwd_on_two_calls():
    lib = _lib()
    cases = [
        nain.small_workload("bf16", (48, 40), 4, 32, (7, 9), (1, 2), B=2, seed=21),
        nain.small_workload("bf16", (6, 14, 13), 2, 32, (3, 5, 5), (1, 1, 1), B=1, seed=22),
    ]
    for w in cases:
        t = {k: v.cuda() for k, v in nain.make_inputs(w, device="cpu").items()}
        o = torch.empty_like(t["q"])
        lse = torch.empty(t["q"].shape[:-1], dtype=torch.float32, device="cuda")
        na.na_fwd(t["q"], t["k"], t["v"], o, lse, w.kernel, w.dilation, w.scale)
        # the existing entry point, with a caller-provided workspace
        ws = torch.empty(na.na_bwd_workspace_size(w.B, w.spatial, w.heads), dtype=torch.uint8, device="cuda")
        ref = [torch.empty_like(t["q"]) for _ in range(3)]
        na.na_bwd(t["q"], t["k"], t["v"], o, t["dO"], lse, *ref, w.kernel, w.dilation, w.scale, workspace=ws)
        # the allocation-free entry point
        got = [torch.full_like(t["q"], float("nan")) for _ in range(3)]
        assert _call_noalloc(lib, w, t, o, lse, *got) == 0
        st, raw = na.na_device_status()
        assert st == 0, f"device status {st} ({raw:#x})"
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            _check(name, g, r, 2e-2)


def test_noalloc_rejects_problems_beyond_its_scratch():
    # 2048 x 2048 tokens x 8 heads = 33.5M rows > the 8M-row scratch: rejected before any CUDA call
    lib = _lib()
    fake = ctypes.c_void_p(256)
    w = nain.WORKLOADS["2d_bf16_2048x2048_k13_d2"]
    assert w.tokens * w.heads > NA_NOALLOC_MAX_ROWS
    st = lib.na_bwd_noalloc(*([fake] * 9), w.B, w.ndim, _ints(w.spatial), w.heads, w.D, _ints(w.kernel),
                            _ints(w.dilation), ctypes.c_float(w.scale), 0, None)
    assert st == NA_ERR_WORKSPACE

"""na_bwd_noalloc: the backward entry point for callers that cannot allocate device memory.

Some callers cannot allocate while they run: for example, a host framework that owns all device
memory under a fixed budget, or a latency-critical loop that forbids allocations.  They cannot let
na_bwd allocate its Delta workspace.  na_bwd_noalloc keeps that scratch in a fixed device array
inside the library instead.  This file checks it through the C ABI against na_bwd (which receives a
caller-provided workspace here), bit for bit, on two calls in a row per case, over cases of
different shapes and all three element types, so stale scratch contents from an earlier call would
show up as a mismatch.  The file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

import neighborhood_attention_fwd_gb300 as na
from neighborhood_attention_fwd_gb300 import build as nabuild
from neighborhood_attention_fwd_gb300 import inputs as nain

NA_NOALLOC_MAX_ROWS = 8 * 1024 * 1024
NA_ERR_WORKSPACE = 6
DTYPE_CODE = {"bf16": 0, "fp32": 1, "fp16": 2}   # na_dtype


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
    dtype = DTYPE_CODE[w.dtype]
    return lib.na_bwd_noalloc(t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(), o.data_ptr(),
                              t["dO"].data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                              w.B, w.ndim, _ints(w.spatial), w.heads, w.D, _ints(w.kernel), _ints(w.dilation),
                              ctypes.c_float(w.scale), dtype, stream)


CASES = [
    nain.small_workload("bf16", (48, 40), 4, 32, (7, 9), (1, 2), B=2, seed=21),
    nain.small_workload("bf16", (6, 14, 13), 2, 32, (3, 5, 5), (1, 1, 1), B=1, seed=22),
    nain.small_workload("fp16", (30, 33), 2, 16, (5, 7), (2, 1), B=1, seed=23),
    nain.small_workload("fp32", (20, 17), 2, 32, (5, 3), (1, 2), B=1, seed=24),
]


@pytest.mark.gpu
def test_noalloc_backward_matches_na_bwd_on_two_calls():
    """Each case calls the allocation-free entry point twice in a row (the scratch array keeps the
    previous call's contents, which the next call must not see); the cases follow one another with
    different shapes and element types.  Both entry points run the same deterministic kernels, so
    the outputs must be bitwise equal."""
    lib = _lib()
    for w in CASES:
        t = {k: v.cuda() for k, v in nain.make_inputs(w, device="cpu").items()}
        o = torch.empty_like(t["q"])
        lse = torch.empty(t["q"].shape[:-1], dtype=torch.float32, device="cuda")
        na.na_fwd(t["q"], t["k"], t["v"], o, lse, w.kernel, w.dilation, w.scale)
        # the existing entry point, with a caller-provided workspace
        ws = torch.empty(na.na_bwd_workspace_size(w.B, w.spatial, w.heads), dtype=torch.uint8, device="cuda")
        ref = [torch.empty_like(t["q"]) for _ in range(3)]
        na.na_bwd(t["q"], t["k"], t["v"], o, t["dO"], lse, *ref, w.kernel, w.dilation, w.scale, workspace=ws)
        for call in range(2):
            got = [torch.full_like(t["q"], float("nan")) for _ in range(3)]
            assert _call_noalloc(lib, w, t, o, lse, *got) == 0
            st, raw = na.na_device_status()
            assert st == 0, f"device status {st} ({raw:#x})"
            for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
                assert torch.equal(g, r), f"{w.dtype} {w.spatial} call {call}: {name} differs from na_bwd"


def test_noalloc_rejects_problems_beyond_its_scratch():
    # 2048 x 2048 tokens x 8 heads = 33.5M rows > the 8M-row scratch: rejected before any CUDA call
    lib = _lib()
    fake = ctypes.c_void_p(256)
    w = nain.WORKLOADS["2d_bf16_2048x2048_k13_d2"]
    assert w.tokens * w.heads > NA_NOALLOC_MAX_ROWS
    st = lib.na_bwd_noalloc(*([fake] * 9), w.B, w.ndim, _ints(w.spatial), w.heads, w.D, _ints(w.kernel),
                            _ints(w.dilation), ctypes.c_float(w.scale), 0, None)
    assert st == NA_ERR_WORKSPACE

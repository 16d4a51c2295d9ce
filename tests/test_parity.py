"""GPU parity: the CUDA library against the fp64 oracle, through the C ABI.

Small problems are compared element by element on every output; the full-size workloads (the
shapes the benchmark times, launched the same way) are compared on sampled rows that the oracle
computes one by one, plus finiteness of every output.
"""
import numpy as np
import pytest
import torch

from neighborhood_attention_fwd_gb300 import inputs as nain
from na_testlib import check_full, check_sampled, host, run_gpu

pytestmark = pytest.mark.gpu

SMALL = [
    # dtype, spatial, heads, D, kernel, dilation, B
    ("fp32", (16, 16), 2, 16, (5, 5), (1, 1), 1),          # the small fp32 workload
    ("fp32", (37,), 3, 32, (7,), (2,), 2),
    ("fp32", (9, 11, 10), 2, 16, (3, 5, 3), (2, 1, 3), 1),
    ("fp32", (12, 13), 1, 64, (5, 3), (1, 4), 1),
    ("fp32", (7, 9), 2, 128, (7, 9), (1, 1), 1),            # kernel == extent: full attention
    ("fp32", (10, 23), 3, 64, (3, 7), (2, 3), 1),           # key quads over unequal classes (dK/dV quads from k2 >= 7)
    ("fp32", (4, 6, 19), 2, 16, (3, 3, 9), (1, 2, 2), 2),   # quads of one class position past a class end
    ("fp32", (300,), 2, 32, (63,), (2,), 1),                # a 63-key window on the quad kernels
    ("bf16", (40, 37), 3, 32, (5, 7), (1, 1), 2),
    ("bf16", (33, 45), 2, 32, (9, 9), (1, 1), 1),
    ("bf16", (200,), 2, 32, (7,), (1,), 2),
    ("bf16", (300,), 1, 16, (13,), (3,), 1),
    ("bf16", (6, 20, 19), 2, 32, (3, 5, 5), (1, 1, 1), 1),
    ("bf16", (10, 18, 21), 1, 64, (5, 7, 7), (1, 1, 1), 1),
    ("bf16", (41, 38), 2, 32, (13, 13), (2, 2), 1),
    ("bf16", (23, 29), 2, 16, (3, 5), (3, 2), 2),           # classes of unequal length
    ("bf16", (17, 16), 1, 64, (17, 15), (1, 1), 1),         # kernel == extent along axis 1
    ("bf16", (8, 30, 30), 1, 32, (1, 9, 1), (1, 2, 1), 1),  # kernel 1 on some axes
    ("bf16", (5, 9, 33), 2, 32, (5, 9, 3), (1, 1, 8), 1),
    ("bf16", (16, 8), 1, 32, (1, 1), (1, 1), 1),            # k = 1: O = V, dQ = dK = 0
    ("bf16", (6, 5, 70), 1, 32, (3, 5, 1), (2, 1, 1), 3),   # short axes: windows touch both borders
    ("bf16", (8, 20, 20), 1, 32, (5, 7, 7), (1, 1, 1), 1),  # long tiles: the forward's three score buffers
    ("bf16", (1000,), 2, 32, (255,), (1,), 1),               # a 255-key window (10-16 chunks per tile)
    ("bf16", (96, 96), 8, 32, (7, 7), (1, 1), 1),            # 576 tiles: several tiles per persistent CTA
    ("fp16", (64, 64), 2, 32, (31, 31), (2, 2), 1),         # 31x31 windows, dilation 2 (three score buffers)
    ("bf16", (40, 40), 1, 64, (39, 39), (1, 1), 1),         # windows of 39x39 on a 40x40 grid
    # fp16 operands on the same tensor-core kernels
    ("fp16", (40, 37), 3, 32, (5, 7), (1, 1), 2),
    ("fp16", (300,), 1, 16, (13,), (3,), 1),
    ("fp16", (6, 20, 19), 2, 32, (3, 5, 5), (1, 1, 1), 1),
    ("fp16", (41, 38), 2, 64, (13, 13), (2, 2), 1),
    ("fp16", (9, 17, 19), 2, 16, (5, 7, 7), (1, 1, 1), 1),  # three score buffers, D = 16
    ("fp16", (16, 8), 1, 32, (1, 1), (1, 1), 1),            # k = 1
    # D = 128: two 64-channel halves per operand; one forward CTA per SM; single-buffered dK/dV
    ("bf16", (33, 30), 2, 128, (7, 5), (1, 2), 1),
    ("bf16", (6, 12, 13), 1, 128, (3, 5, 5), (1, 1, 1), 2),
    ("fp16", (33, 30), 2, 128, (7, 5), (1, 2), 1),
    ("fp16", (6, 12, 13), 1, 128, (3, 5, 5), (1, 1, 1), 2),
    ("bf16", (200,), 1, 128, (13,), (3,), 1),
]


def _ids(c):
    return f"{c[0]}-{'x'.join(map(str, c[1]))}-h{c[2]}-D{c[3]}-k{'x'.join(map(str, c[4]))}-d{'x'.join(map(str, c[5]))}-B{c[6]}"


@pytest.mark.parametrize("case", SMALL, ids=[_ids(c) for c in SMALL])
def test_small_full_parity(case, cuda_lib):
    dtype, spatial, heads, D, kernel, dilation, B = case
    w = nain.small_workload(dtype, spatial, heads, D, kernel, dilation, B=B, seed=11)
    t = nain.make_inputs(w, device="cpu")
    gpu = run_gpu(w, {k: v.cuda() for k, v in t.items()})
    check_full(w, gpu, host(t))


def test_split_backward_matches_fused_entry_point(cuda_lib):
    w = nain.small_workload("bf16", (30, 26), 2, 32, (7, 5), (1, 2), B=1, seed=3)
    t = {k: v.cuda() for k, v in nain.make_inputs(w, device="cpu").items()}
    a = run_gpu(w, t)
    b = run_gpu(w, t, split_bwd=True)
    for key in ("o", "lse", "dq", "dk", "dv"):
        assert torch.equal(a[key], b[key]), key


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_forward_rescales_on_a_wide_score_range(cuda_lib, dtype):
    """q and k scaled by 3: scores spread over tens of log2 units, so the forward's running max moves
    by more than its 2^8 threshold across chunks and between the two parts of a long run (2D 33x45
    with a 9x9 window has runs of five 16-column groups), and O, and P already written, are rescaled.
    Forward only: the rescales are the forward's."""
    w = nain.small_workload(dtype, (33, 45), 2, 32, (9, 9), (1, 1), B=1, seed=21)
    t = nain.make_inputs(w, device="cpu")
    for key in ("q", "k"):
        t[key] = (t[key].float() * 3.0).to(t[key].dtype)
    gpu = run_gpu(w, {k: v.cuda() for k, v in t.items()}, want_bwd=False)
    check_full(w, gpu, host(t), want_bwd=False)


def test_backward_is_deterministic(cuda_lib):
    w = nain.small_workload("bf16", (40, 40), 2, 32, (9, 9), (1, 1), B=1, seed=4)
    t = {k: v.cuda() for k, v in nain.make_inputs(w, device="cpu").items()}
    a = run_gpu(w, t)
    b = run_gpu(w, t)
    for key in ("o", "lse", "dq", "dk", "dv"):
        assert torch.equal(a[key], b[key]), key


def test_delta_matches_rowwise_dot(cuda_lib):
    import neighborhood_attention_fwd_gb300 as na

    for dtype in (torch.bfloat16, torch.float32):
        g = torch.Generator().manual_seed(5)
        o = torch.randn(2, 9, 7, 3, 32, generator=g).to(dtype)
        dO = torch.randn(2, 9, 7, 3, 32, generator=g).to(dtype)
        delta = torch.empty(2, 9, 7, 3, dtype=torch.float32, device="cuda")
        na.na_bwd_delta(o.cuda(), dO.cuda(), delta)
        ref = (o.double() * dO.double()).sum(-1)
        tol = 1e-5 if dtype == torch.float32 else 1e-4
        assert (delta.cpu().double() - ref).abs().max() <= tol * ref.abs().max()


FULL = [name for name in nain.WORKLOADS if nain.WORKLOADS[name].dtype == "bf16"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_parity(name, cuda_lib):
    w = nain.WORKLOADS[name]
    t = nain.make_inputs(w, device="cuda")
    gpu = run_gpu(w, t)
    h = host(t)
    check_sampled(w, gpu, h, n=256)


def test_full_size_fp16_headline_shape_sampled(cuda_lib):
    """The 2D 1024x1024 / 9x9 shape with fp16 tensors (the dtype of the page's fast numbers), launched as
    bench.py --dtype fp16 launches it, on sampled rows."""
    import dataclasses

    base = nain.WORKLOADS[nain.HEADLINE]
    w = dataclasses.replace(base, name=base.name.replace("bf16", "fp16"), dtype="fp16")
    t = nain.make_inputs(w, device="cuda")
    gpu = run_gpu(w, t)
    check_sampled(w, gpu, host(t), n=192)


def test_full_size_fp32_workload(cuda_lib):
    w = nain.WORKLOADS["2d_fp32_16x16_k5"]
    t = nain.make_inputs(w, device="cpu")
    gpu = run_gpu(w, {k: v.cuda() for k, v in t.items()})
    check_full(w, gpu, host(t))

"""The benchmark's FLOP/byte model against the only figures the pages print for this path."""
import json
import os

import pytest

import bench
from neighborhood_attention_fwd_gb300 import inputs as nain

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "arithmetic_intensity.json")))


@pytest.mark.parametrize("dim,name", [("2d", "2d_bf16_1024x1024_k9"), ("3d", "3d_bf16_16x256x256_k3x5x5")])
def test_arithmetic_intensity_matches_the_page(dim, name):
    w = nain.WORKLOADS[name]
    tol = GOLDEN["tolerance_abs"]
    v = GOLDEN["values"]
    assert abs(bench.arithmetic_intensity(w, fused=True, elem_bytes=4) - v[f"{dim}_fused"]) <= tol
    assert abs(bench.arithmetic_intensity(w, fused=False, elem_bytes=4) - v[f"{dim}_unfused"]) <= tol


def test_a40_threshold():
    v = GOLDEN["values"]
    assert abs(v["a40_peak_tflops"] * 1e12 / (v["a40_bandwidth_gbs"] * 1e9) - v["a40_threshold"]) <= GOLDEN["tolerance_abs"]


def test_useful_flops_and_bytes():
    w = nain.WORKLOADS["2d_bf16_1024x1024_k9"]
    f, b = bench.useful_flops(w)
    assert f == pytest.approx(4 * 1024 * 1024 * 81 * 32 * 8)
    assert b == pytest.approx(2.5 * f)
    kb = bench.kernel_bytes(w)
    assert kb["fwd"] == pytest.approx(1024 * 1024 * 8 * (4 * 64 + 4))


def test_unfused_call_work_model():
    """Per-call bytes and FLOPs of the unfused chain: the weights (R x K elements) cross HBM once per
    producer and once per consumer, and the products sum to the fused path's useful FLOPs."""
    w = nain.WORKLOADS["2d_bf16_1024x1024_k9"]
    work = bench.unfused_call_work(w)
    R = w.tokens * w.heads
    RK = R * w.keys_per_query * 2
    RD = R * w.D * 2
    assert work["softmax"] == (2 * RK, 0.0)
    assert work["qk"][0] == 2 * RD + RK and work["av"][0] == 2 * RD + RK
    f_fwd, f_bwd = bench.useful_flops(w)
    assert sum(work[c][1] for c in ("qk", "av")) == f_fwd
    assert sum(work[c][1] for c in ("av_bwd", "qk_bwd")) == 8.0 * R * w.keys_per_query * w.D
    # the fused backward's useful count adds the recomputed logits and probabilities (2 products)
    assert f_bwd == 10.0 * R * w.keys_per_query * w.D
    assert abs(bench.fp32_fma_tflops() - 80.55) < 0.01


def test_growing_window_sizes_and_masked_count():
    """The --varwin pattern grows from 1 to the full kernel along the first axis, and the masked-weight
    count matches a direct count over every row."""
    import numpy as np

    w = nain.small_workload("bf16", (10, 6), 2, 16, (5, 3), (1, 1), B=2)
    sizes = bench.growing_window_sizes(w)
    assert sizes[0] == [1, 1, 1, 1, 3, 3, 3, 5, 5, 5]
    assert sizes[1] == [3] * 6
    direct = sum((w.keys_per_query - k0 * 3) * 6 for k0 in sizes[0]) * w.B * w.heads
    assert bench.masked_weights(w, sizes) == direct
    head = nain.WORKLOADS[nain.HEADLINE]
    s = bench.growing_window_sizes(head)
    assert s[0][0] == 1 and s[0][-1] == 9 and all(np.diff(s[0]) >= 0)

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

"""Seeded synthetic inputs for neighborhood attention workloads.

This module only draws random numbers and describes workload shapes; it holds none of the
method's arithmetic, so the device library, the oracle, the tests and the benchmark can all use
it.  The workloads are the shapes of NATTEN issue #161 ("Backward pass is very slow towards much
tokens and large kernels": the user's benchmark script, B=1, 8 heads of dim 32, 2D 1024x1024 with
a 9x9 kernel and 3D 16x256x256 with a (3,5,5) kernel, loss = output.sum() so dO = 1), the
(8,128,128)/(5,7,7) model shape the user mentions later in the thread, a small fp32 case that the
oracle finishes in well under a second, and a large dilated 2D stress case.

Recipe: q, k, v and (when not ones) dO are drawn in that order, iid N(0, 1) in float32 from a
torch.Generator seeded with ``seed``, then rounded to bfloat16 (fp16) for bf16 (fp16) workloads.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str                 # "bf16", "fp16" or "fp32"
    B: int
    spatial: tuple
    heads: int
    D: int
    kernel: tuple
    dilation: tuple
    dO: str                    # "ones" or "randn"
    seed: int
    note: str = field(default="", compare=False)

    @property
    def ndim(self) -> int:
        return len(self.spatial)

    @property
    def shape(self) -> tuple:
        return (self.B, *self.spatial, self.heads, self.D)

    @property
    def scale(self) -> float:
        return float(self.D) ** -0.5

    @property
    def tokens(self) -> int:
        return int(self.B * np.prod(self.spatial))

    @property
    def keys_per_query(self) -> int:
        return int(np.prod(self.kernel))

    def torch_dtype(self):
        return {"bf16": torch.bfloat16, "fp16": torch.float16}.get(self.dtype, torch.float32)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("2d_fp32_16x16_k5", "fp32", 1, (16, 16), 2, 16, (5, 5), (1, 1), "randn", 1235,
                 "small fp32 case, every tile partial"),
        Workload("2d_bf16_1024x1024_k9", "bf16", 1, (1024, 1024), 8, 32, (9, 9), (1, 1), "ones", 1236,
                 "the issue's 2D benchmark shape"),
        Workload("3d_bf16_16x256x256_k3x5x5", "bf16", 1, (16, 256, 256), 8, 32, (3, 5, 5), (1, 1, 1),
                 "ones", 1237, "the issue's 3D benchmark shape"),
        Workload("3d_bf16_b2_8x128x128_k5x7x7", "bf16", 2, (8, 128, 128), 8, 32, (5, 7, 7), (1, 1, 1),
                 "randn", 1238, "the issue's (8,128,128)/(5,7,7) model shape"),
        Workload("2d_bf16_2048x2048_k13_d2", "bf16", 1, (2048, 2048), 8, 32, (13, 13), (2, 2), "randn",
                 1239, "large dilated 2D stress case"),
        Workload("2d_bf16_512x512_k9", "bf16", 1, (512, 512), 8, 32, (9, 9), (1, 1), "ones", 1240,
                 "profiling case: the 2D benchmark's kernels on a quarter of its tokens (inputs > L2)"),
    ]
}

# The workload the benchmark's headline line is quoted on.
HEADLINE = "2d_bf16_1024x1024_k9"


def make_inputs(w: Workload, device="cpu", seed: int | None = None):
    """Return dict(q, k, v, dO) as contiguous tensors of w.shape in w's dtype on `device`."""
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed if seed is None else seed)
    out = {}
    for name in ("q", "k", "v"):
        out[name] = torch.randn(w.shape, generator=gen, dtype=torch.float32, device=device).to(w.torch_dtype())
    if w.dO == "ones":
        out["dO"] = torch.ones(w.shape, dtype=w.torch_dtype(), device=device)
    else:
        out["dO"] = torch.randn(w.shape, generator=gen, dtype=torch.float32, device=device).to(w.torch_dtype())
    return out


def make_weights(w: Workload, kind: str = "randn", device="cpu", seed: int = 0):
    """A seeded tensor shaped like the unfused operations' attention weights [B, L.., heads, K] in
    w's dtype: iid N(0, 1) ("randn": logits, gradients) or U(0, 1) ("uniform": probability-like
    weights), drawn in float32 and rounded."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    shape = (w.B, *w.spatial, w.heads, w.keys_per_query)
    if kind == "uniform":
        x = torch.rand(shape, generator=gen, dtype=torch.float32, device=device)
    else:
        x = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
    return x.to(w.torch_dtype())


def make_rpb(w: Workload, device="cpu", seed: int = 0):
    """A seeded relative-positional-bias table, fp32 [heads, 2k_0 - 1, ..], iid N(0, 1)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    shape = (w.heads,) + tuple(2 * k - 1 for k in w.kernel)
    return torch.randn(shape, generator=gen, dtype=torch.float32, device=device)


def small_workload(dtype: str, spatial, heads, D, kernel, dilation, B=1, dO="randn", seed=7) -> Workload:
    """An ad-hoc workload (parity sweeps)."""
    return Workload(f"adhoc_{dtype}_{'x'.join(map(str, spatial))}", dtype, B, tuple(spatial), heads, D,
                    tuple(kernel), tuple(dilation), dO, seed)


def to_oracle_array(t: torch.Tensor) -> np.ndarray:
    """Host copy in the form the oracle reads: float32 values, bfloat16 bit patterns as uint16, or
    float16 values widened to float64 (exact: every float16 is a float64)."""
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float16:
        return t.numpy().astype(np.float64)
    if t.dtype == torch.float32:
        return t.numpy()
    raise TypeError(f"unsupported dtype {t.dtype}")

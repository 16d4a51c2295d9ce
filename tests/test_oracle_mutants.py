"""Mutation checks for the oracle's pins (CPU only).

Each case copies na_oracle.c, plants one plausible mistake in the copy (a wrong window start,
class length, scale, log base, sign or dropped term), compiles it into a temporary library and
runs the pins of test_oracle.py against it: at least one pin must fail.  The real oracle is not
touched.
"""
import os
import subprocess

import numpy as np
import pytest

import oracle
import test_oracle as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "na_oracle.c")

MUTANTS = {
    "window_start_off_by_one": ("int s = j - k / 2;", "int s = j - k / 2 + 1;"),
    "class_length_floor": ("int Lc = (L - c + d - 1) / d;", "int Lc = (L - c) / d;"),
    "no_border_shift": ("if (s > Lc - k) s = Lc - k;", ""),
    "lse_log2": ("*lse = m + log(l);", "*lse = m + log2(l);"),
    "dk_missing_scale": ("for (int e = 0; e < D; ++e) ok_[e] *= scale;", ""),
    "ds_sign": ("double ds = pij * (dp - st[si].delta);", "double ds = pij * (st[si].delta - dp);"),
    "dq_missing_delta": ("double ds = p * (dp - st[si].delta);", "double ds = p * dp;"),
    "dv_uses_ds": ("ov_[e] += pij * in_val(dO, oq + e, in_kind);", "ov_[e] += ds * in_val(dO, oq + e, in_kind);"),
    "dq_missing_scale": ("for (int c = 0; c < D; ++c) out[c] *= scale;", ""),
    "key_window_half_span": ("if (++off[a] <= g.k[a] - 1) break;\n                    off[a] = -(g.k[a] - 1);\n                }\n            }\n            for (int e",
                             "if (++off[a] <= g.k[a] / 2) break;\n                    off[a] = -(g.k[a] - 1);\n                }\n            }\n            for (int e"),
    "delta_uses_q": ("delta += in_val(dO, od + c, in_kind) * o[c];", "delta += in_val(q, od + c, in_kind) * o[c];"),
}


def build_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / f"lib_{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", str(lib), str(path), "-lm"],
                   check=True)
    return str(lib)


def pin_results():
    """Run a fast selection of the pins; return the names of those that fail."""
    failed = []
    checks = {
        "window": pins.test_window_is_nearest_k_in_class,
        "full_attention": lambda: pins.test_fwd_kernel_equal_extent_is_full_attention((3, 5, 5)),
    }
    for i, case in enumerate(pins.CASES):
        checks[f"dense_fwd_{i}"] = lambda c=case: pins.test_fwd_matches_dense_masked_attention(*c)
        checks[f"dense_bwd_{i}"] = lambda c=case: pins.test_bwd_matches_dense_autograd(*c)
    checks["fd"] = lambda: pins.test_bwd_matches_finite_differences((5, 6), (3, 3), (1, 2))
    for name, fn in checks.items():
        try:
            fn()
        except (AssertionError, ValueError):
            failed.append(name)
    return failed


def test_pins_pass_on_the_real_oracle():
    assert pin_results() == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(tmp_path, name):
    lib = build_mutant(tmp_path, name)
    with oracle.library(lib):
        failed = pin_results()
    assert failed, f"no pin caught the planted mistake {name}"

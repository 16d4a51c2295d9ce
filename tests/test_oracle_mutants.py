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


# ---------------------------------------------------------------------------------------------
# The unfused operations' oracle (oracle/unfused.py): mutants are compiled from edited source text
# into a fresh module object, and test_oracle_unfused.py's pins run against it.
# ---------------------------------------------------------------------------------------------

import types

import oracle.unfused as unfused
import test_oracle_unfused as unpins

UNFUSED_SRC = os.path.join(os.path.dirname(oracle.__file__), "unfused.py")

UNFUSED_MUTANTS = {
    "inverse_offset_order": ("offsets = (offsets[:, None] * self.kernel[a] + ti[None, :]).ravel()",
                             "offsets = (offsets[:, None] + ti[None, :] * (self.K // self.kernel[a] if a == 0 else 1)).ravel()"),
    "dk_missing_scale": ("dk = scale * _scatter", "dk = _scatter"),
    "softmax_bwd_sign": ("return y * (dy - (y * dy).sum(axis=-1, keepdims=True))",
                         "return y * (dy + (y * dy).sum(axis=-1, keepdims=True))"),
    "window_offsets_reversed": ("idx = idx + (tab[x[:, a]] * self.strides[a]).reshape(shape)",
                                "idx = idx + (tab[x[:, a]][:, ::-1] * self.strides[a]).reshape(shape)"),
    "dv_scatters_dO_with_dattn": ("dv = _scatter(af, gf, g, rows, B, N, heads)",
                                  "dv = _scatter(af, vf, g, rows, B, N, heads)"),
    "qk_missing_scale_on_rows": ("out = scale * np.einsum(\"rc,rtc->rt\"", "out = np.einsum(\"rc,rtc->rt\""),
    "rpb_relative_sign": ("rel = tab[x[:, a]] // d - (x[:, a] // d)[:, None] + (k - 1)",
                          "rel = (x[:, a] // d)[:, None] - tab[x[:, a]] // d + (k - 1)"),
    "rpb_axis_order": ("span = int(np.prod([2 * kk - 1 for kk in g.kernel[a + 1:]]))",
                       "span = int(np.prod([2 * kk - 1 for kk in g.kernel[:a]]))"),
    "varwin_full_kernel_start": ("first = np.array([first_neighbour(int(i), L, int(ka[i]), d) for i in range(L)])",
                                 "first = np.array([first_neighbour(int(i), L, int(g.kernel[a]), d) for i in range(L)])"),
    "varwin_span_off_by_one": ("hi = lo + d * (ka[x[:, a]][:, None] - 1)", "hi = lo + d * ka[x[:, a]][:, None]"),
    "rpb_grad_drops_batch": ("weights=_f64(wf[:, :, h, :]).sum(axis=0).ravel()", "weights=_f64(wf[0, :, h, :]).ravel()"),
}


def unfused_mutant(name):
    old, new = UNFUSED_MUTANTS[name]
    src = open(UNFUSED_SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mod = types.ModuleType(f"oracle._unfused_mutant_{name}")
    mod.__package__ = "oracle"
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), mod.__dict__)
    return mod


def unfused_pin_results(mod):
    failed = []
    checks = {"softmax_fd": unpins.test_softmax_bwd_matches_finite_differences,
              "inverse_lists": unpins.test_inverse_lists_cover_every_pair_once,
              "offset_order": lambda: unpins.test_offset_order_from_index_coded_keys((7, 9), (3, 5), (2, 1))}
    for i, case in enumerate(pins.CASES):
        checks[f"chain_fwd_{i}"] = lambda c=case: unpins.test_chain_forward_equals_fused_oracle(*c)
        checks[f"chain_bwd_{i}"] = lambda c=case: unpins.test_chain_backward_equals_fused_oracle(*c)
        checks[f"adjoint_{i}"] = lambda c=case: unpins.test_adjoint_identities(*c)
    for i in (2, 4, 6, 7):
        checks[f"rows_{i}"] = lambda c=pins.CASES[i]: unpins.test_sampled_rows_match_full(*c)
    for i in (0, 2, 4, 6):
        checks[f"rpb_dense_{i}"] = lambda c=pins.CASES[i]: unpins.test_rpb_chain_matches_dense_attention_with_bias(*c)
    for i, case in enumerate(pins.CASES):
        checks[f"rpb_adjoint_{i}"] = lambda c=case: unpins.test_rpb_grad_is_the_adjoint_of_the_bias(*c)
    checks["rpb_counts"] = unpins.test_rpb_grad_counts_pairs_per_relative_position
    for i, case in enumerate(unpins.VARWIN):
        checks[f"varwin_{i}"] = lambda c=case: unpins.test_variable_window_chain_matches_dense_attention(*c)
    checks["varwin_special"] = unpins.test_variable_window_special_cases
    checks["rpb_rows"] = unpins.test_rpb_sampled_rows_match_full
    saved = unpins.un
    unpins.un = mod
    try:
        for name, fn in checks.items():
            try:
                fn()
            except (AssertionError, ValueError, IndexError):
                failed.append(name)
    finally:
        unpins.un = saved
    return failed


def test_unfused_pins_pass_on_the_real_oracle():
    assert unfused_pin_results(unfused) == []


@pytest.mark.parametrize("name", sorted(UNFUSED_MUTANTS))
def test_unfused_pins_reject_mutant(name):
    assert unfused_pin_results(unfused_mutant(name)), f"no pin caught the planted mistake {name}"

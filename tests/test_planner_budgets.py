"""Host-side checks of the tile planner (CPU only) over random problems: every plan the library returns
fits the kernels' TMEM, shared-memory and register-run budgets, so a supported problem never reaches a
kernel with an impossible layout."""
import random

import pytest

import neighborhood_attention_fwd_gb300 as na
from neighborhood_attention_fwd_gb300 import build as nabuild


@pytest.fixture(scope="module")
def lib():
    nabuild.build()
    return na.load()


def random_problem(rng):
    ndim = rng.randint(1, 3)
    spatial, kernel, dilation = [], [], []
    for _ in range(ndim):
        d = rng.choice([1, 1, 1, 2, 3])
        k = rng.choice([1, 3, 5, 7, 9, 11, 13])
        L = rng.randint(k * d, k * d + (40 if ndim == 3 else 90))
        spatial.append(L)
        kernel.append(k)
        dilation.append(d)
    return tuple(spatial), tuple(kernel), tuple(dilation), rng.choice([16, 32, 64, 128])


def test_plans_fit_the_kernels_budgets(lib):
    rng = random.Random(2024)
    checked = 0
    for _ in range(150):
        spatial, kernel, dilation, D = random_problem(rng)
        for which in (0, 1, 2):
            try:
                p = na.na_plan_info(which, 1, spatial, 2, D, kernel, dilation)
            except na.NAError:
                continue  # outside what the tensor-core kernels support (documented in the header)
            checked += 1
            T = (p["T1"], p["T2"], p["T3"])
            G = (p["G1"], p["G2"], p["G3"])
            H = (p["H1"], p["H2"], p["H3"])
            NC = p["NC"]
            assert T[0] * T[1] * T[2] == 128 and all(t & (t - 1) == 0 for t in T)
            assert NC == G[0] * G[1] * G[2] and NC % 16 == 0 and NC >= 16
            # the window-bias operand: at most two 16-column groups per chunk and masked axis
            assert all(1 <= G[a] <= min(H[a], 32) for a in range(3))
            assert p["smem_bytes"] <= 227 * 1024
            if which == 0 and D <= 64:
                # two CTAs per SM: two score buffers (P written over them) and two accumulators in 256
                # TMEM columns, a softmax run of at most six groups, and two CTAs' shared memory
                assert p["tmem_cols"] == 256
                assert 2 * NC + 2 * D <= 256 and NC <= 96
                assert p["smem_bytes"] <= 113 * 1024
            elif which == 0:
                # D = 128: one CTA per SM with all 512 columns
                assert p["tmem_cols"] == 512 and 2 * NC + 2 * D <= 512 and NC <= 96
            elif which == 1:
                assert p["tmem_cols"] == 512 and 4 * NC + 2 * D <= 512  # S, dP (two each), dQ (two)
            elif D <= 64:
                assert p["tmem_cols"] == 512 and 4 * NC + 4 * D <= 512  # S, dP, dV and dK (two each)
            else:
                assert p["tmem_cols"] == 512 and 4 * NC + 2 * D <= 512  # dV and dK single-buffered at D = 128
            assert p["ctas"] >= 1 and p["chunks_max"] >= 1 and p["chunks_total"] >= p["ctas"] // 2
    assert checked > 200

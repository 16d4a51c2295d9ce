"""CPU model of the tensor-core kernels' tile geometry (host logic; no GPU).

The kernels decide, per CTA, which halo box to load and which chunks to process; the window-bias
product decides which (row, column) scores of a chunk stay live (one-hot local coordinates against
per-row window bits, per axis); and each softmax warp reads only the run of 16-column groups that
holds its rows' windows.  This test replays those decisions with the real tile plans
(na_plan_info) and checks, against the oracle's window function, that every (query, key) pair of
the neighbourhood is live in exactly one chunk and read by its warp, and that nothing else is
live; for dK/dV, that the inverse windows are exactly the queries whose windows hold each key.
"""
import itertools

import numpy as np
import pytest

import neighborhood_attention_fwd_gb300 as na
import oracle
from neighborhood_attention_fwd_gb300 import build as nabuild


@pytest.fixture(scope="module", autouse=True)
def lib():
    nabuild.build()
    na.load()


def win_start(j, Lc, k):
    return max(0, min(j - k // 2, Lc - k))


def inv_lo(j, k):
    return 0 if j < k else j - k // 2


def inv_hi(j, Lc, k):
    return Lc - 1 if j >= Lc - k else j + k // 2


def group_run(G, o, ulo, uhi):
    """The kernels' chunk_range: 16-column groups [glo, glo + n) covering a warp union."""
    lo = [max(ulo[a] - o[a], 0) for a in range(3)]
    hi = [min(uhi[a] - o[a], G[a]) for a in range(3)]
    if any(lo[a] >= hi[a] for a in range(3)):
        return 0, 0
    clo = (lo[0] * G[1] + lo[1]) * G[2] + lo[2]
    chi = ((hi[0] - 1) * G[1] + hi[1] - 1) * G[2] + hi[2]
    glo = clo >> 4
    return glo, ((chi + 15) >> 4) - glo


def replay(which, L, k, d, plan):
    """Yield (row_global_coords, key_or_query_global_coords) pairs the kernel keeps live."""
    T = (plan["T1"], plan["T2"], plan["T3"])
    H = (plan["H1"], plan["H2"], plan["H3"])
    G = (plan["G1"], plan["G2"], plan["G3"])
    NC = plan["NC"]
    assert NC == G[0] * G[1] * G[2] and NC % 16 == 0
    for a in range(3):
        if H[a] > 1:
            assert G[a] <= 32, "window-bias operand: at most two 16-column groups per axis"
    if which == 0:
        assert NC <= 96, "the forward's softmax takes runs of at most six groups"
    Lcm = [-(-L[a] // d[a]) for a in range(3)]
    ntile = [-(-Lcm[a] // T[a]) for a in range(3)]
    nchk = [-(-H[a] // G[a]) for a in range(3)]
    pairs = []
    for cls in itertools.product(*[range(x) for x in d]):
        Lc = [(L[a] - cls[a] + d[a] - 1) // d[a] for a in range(3)]
        for t in itertools.product(*[range(x) for x in ntile]):
            t0 = [t[a] * T[a] for a in range(3)]
            if any(t0[a] >= Lc[a] for a in range(3)):
                continue
            h0, nc = [0] * 3, [0] * 3
            for a in range(3):
                last = min(t0[a] + T[a], Lc[a]) - 1
                if which != 2:
                    lo, hi = win_start(t0[a], Lc[a], k[a]), win_start(last, Lc[a], k[a]) + k[a] - 1
                else:
                    lo, hi = inv_lo(t0[a], k[a]), inv_hi(last, Lc[a], k[a])
                h0[a] = min(lo, max(0, Lc[a] - H[a]))
                assert hi - h0[a] + 1 <= H[a], "halo box too small"
                nc[a] = min(nchk[a], (hi - h0[a] + G[a]) // G[a])
            rows = []
            for row in range(128):
                tq = (row // (T[2] * T[1]), (row // T[2]) % T[1], row % T[2])
                j = [t0[a] + tq[a] for a in range(3)]
                valid = all(j[a] < Lc[a] for a in range(3))
                lo, ln = [], []
                for a in range(3):
                    jc = min(j[a], Lc[a] - 1)
                    if which != 2:
                        lo.append(win_start(jc, Lc[a], k[a]) - h0[a])
                        ln.append(k[a])
                    else:
                        lo.append(inv_lo(jc, k[a]) - h0[a])
                        ln.append(inv_hi(jc, Lc[a], k[a]) - inv_lo(jc, k[a]) + 1)
                    if which != 0 and j[a] >= Lc[a]:
                        ln[a] = 0  # the row's bias part along this axis is all -2^100
                rows.append((valid, j, lo, ln))
            for w in range(4):
                lanes = rows[32 * w:32 * w + 32]
                live_rows = [r for r in lanes if all(x > 0 for x in r[3])]
                if live_rows:
                    ulo = [min(r[2][a] for r in live_rows) for a in range(3)]
                    uhi = [max(r[2][a] + r[3][a] for r in live_rows) for a in range(3)]
                else:
                    ulo, uhi = [1 << 30] * 3, [-(1 << 30)] * 3
                for ix in itertools.product(range(nc[0]), range(nc[1]), range(nc[2])):
                    o = [ix[a] * G[a] for a in range(3)]
                    glo, n = group_run(G, o, ulo, uhi)
                    assert 16 * (glo + n) <= NC, "group run outside the chunk"
                    for valid, j, lo, ln in lanes:
                        for col in range(NC):
                            loc = (col // (G[1] * G[2]), (col // G[2]) % G[1], col % G[2])
                            pos = [o[a] + loc[a] for a in range(3)]
                            # bias: 0 along every axis (masked axes: inside the row's range)
                            live = all(lo[a] <= pos[a] < lo[a] + ln[a] if H[a] > 1 else loc[a] == 0
                                       for a in range(3))
                            if not live or not valid:
                                continue  # a row past an axis end is computed but never stored
                            assert glo * 16 <= col < (glo + n) * 16, "a live score outside the warp's run"
                            other = [h0[a] + pos[a] for a in range(3)]
                            rg = tuple(cls[a] + d[a] * j[a] for a in range(3))
                            og = tuple(cls[a] + d[a] * other[a] for a in range(3))
                            pairs.append((rg, og))
    return pairs


def expected(which, L, k, d):
    exp = []
    for x in itertools.product(*[range(n) for n in L]):
        if which != 2:
            f = [oracle.first_neighbour(x[a], L[a], k[a], d[a]) for a in range(3)]
            for t in itertools.product(*[range(n) for n in k]):
                exp.append((tuple(x), tuple(f[a] + d[a] * t[a] for a in range(3))))
        else:
            # queries whose window holds key x: brute force over the axis
            per_axis = []
            for a in range(3):
                qs = [i for i in range(L[a])
                      if x[a] in {oracle.first_neighbour(i, L[a], k[a], d[a]) + d[a] * t for t in range(k[a])}]
                per_axis.append(qs)
            for qq in itertools.product(*per_axis):
                exp.append((tuple(x), tuple(qq)))
    return exp


CASES = [
    ((1, 16, 16), (1, 5, 5), (1, 1, 1)),
    ((1, 37, 29), (1, 9, 7), (1, 1, 1)),
    ((1, 1, 150), (1, 1, 13), (1, 1, 1)),
    ((1, 1, 100), (1, 1, 7), (1, 1, 3)),
    ((1, 23, 29), (1, 3, 5), (1, 3, 2)),
    ((1, 41, 38), (1, 13, 13), (1, 2, 2)),
    ((6, 20, 19), (3, 5, 5), (1, 1, 1)),
    ((10, 18, 21), (5, 7, 7), (1, 1, 1)),
    ((9, 11, 10), (3, 5, 3), (2, 1, 3)),
    ((5, 9, 33), (5, 9, 3), (1, 1, 8)),
]


@pytest.mark.parametrize("which", [0, 2])
@pytest.mark.parametrize("L,k,d", CASES)
def test_kernel_visits_exactly_the_neighbourhood(which, L, k, d):
    ndim = sum(1 for x in L if x > 1) or 1
    sp, kk, dd = L[3 - ndim:], k[3 - ndim:], d[3 - ndim:]
    for D in (16, 32, 64, 128):
        plan = na.na_plan_info(which, 1, sp, 1, D, kk, dd)
        got = replay(which, L, k, d, plan)
        exp = expected(which, L, k, d)
        assert len(got) == len(set(got)), "a pair is visited twice"
        assert sorted(got) == sorted(exp)

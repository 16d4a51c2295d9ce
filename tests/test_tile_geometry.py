"""CPU model of the tensor-core kernels' tile geometry (host logic; no GPU).

The kernels decide, per CTA, which halo box to load, which chunks to process, which halo rows and
8-column blocks each softmax warp visits (the union of its 32 rows' windows), and an 8-bit mask of
live keys per block.  This test replays those decisions with the real tile plans (na_plan_info) and
checks, against the oracle's window function, that every (query, key) pair of the neighbourhood is
visited exactly once and nothing else is, that every visited column lies inside the chunk, and
that dK/dV's inverse windows are exactly the queries whose windows hold each key.
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


def replay(which, L, k, d, plan):
    """Yield (row_global_coords, key_or_query_global_coords) pairs the kernel marks live."""
    T = (plan["T1"], plan["T2"], plan["T3"])
    H = (plan["H1"], plan["H2"], plan["H3"])
    G = (plan["G1"], plan["G2"], plan["G3"])
    NC = plan["NC"]
    Lcm = [-(-L[a] // d[a]) for a in range(3)]
    ntile = [-(-Lcm[a] // T[a]) for a in range(3)]
    nchk = [-(-H[0] // G[0]), -(-H[1] // G[1])]
    pairs = []
    for cls in itertools.product(*[range(x) for x in d]):
        Lc = [(L[a] - cls[a] + d[a] - 1) // d[a] for a in range(3)]
        for t in itertools.product(*[range(x) for x in ntile]):
            t0 = [t[a] * T[a] for a in range(3)]
            if any(t0[a] >= Lc[a] for a in range(3)):
                continue
            h0, need = [0] * 3, [0] * 3
            for a in range(3):
                last = min(t0[a] + T[a], Lc[a]) - 1
                if which != 2:
                    lo, hi = win_start(t0[a], Lc[a], k[a]), win_start(last, Lc[a], k[a]) + k[a] - 1
                else:
                    lo, hi = inv_lo(t0[a], k[a]), inv_hi(last, Lc[a], k[a])
                h0[a] = min(lo, max(0, Lc[a] - H[a]))
                need[a] = hi - h0[a] + 1
                assert need[a] <= H[a], "halo box too small"
            ncy = min(nchk[0], -(-need[0] // G[0]))
            ncz = min(nchk[1], -(-need[1] // G[1]))
            rows = []
            for row in range(128):
                tq = (row // (T[2] * T[1]), (row // T[2]) % T[1], row % T[2])
                j = [t0[a] + tq[a] for a in range(3)]
                valid = all(j[a] < Lc[a] for a in range(3))
                jc = [min(j[a], Lc[a] - 1) for a in range(3)]
                lo, ln = [], []
                for a in range(3):
                    if which != 2:
                        lo.append(win_start(jc[a], Lc[a], k[a]) - h0[a])
                        ln.append(k[a])
                    else:
                        lo.append(inv_lo(jc[a], k[a]) - h0[a])
                        ln.append(inv_hi(jc[a], Lc[a], k[a]) - inv_lo(jc[a], k[a]) + 1)
                if not valid and which != 0:
                    ln = [0, 0, 0]
                rows.append((valid, j, lo, ln))
            for w in range(4):
                lanes = rows[32 * w:32 * w + 32]
                live = [r for r in lanes if all(x > 0 for x in r[3])]
                if not live:
                    continue
                ulo = [min(r[2][a] for r in live) for a in range(3)]
                uhi = [max(r[2][a] + r[3][a] for r in live) for a in range(3)]
                blo, bhi = max(0, ulo[2]) >> 3, min(H[2], uhi[2] + 7) >> 3
                for ci in range(ncy * ncz):
                    y0, z0 = (ci // ncz) * G[0], (ci % ncz) * G[1]
                    ya, yb = max(ulo[0], y0), min(uhi[0], y0 + G[0])
                    za, zb = max(ulo[1], z0), min(uhi[1], z0 + G[1])
                    for y in range(ya, yb):
                        for z in range(za, zb):
                            seg = ((y - y0) * G[1] + (z - z0)) * H[2]
                            for bb in range(blo, bhi):
                                assert seg + bb * 8 + 8 <= NC, "TMEM/P column outside the chunk"
                                for valid, j, lo, ln in lanes:
                                    if not (0 <= y - lo[0] < ln[0] and 0 <= z - lo[1] < ln[1]):
                                        continue
                                    for e in range(8):
                                        x = 8 * bb + e
                                        if lo[2] <= x < lo[2] + ln[2]:
                                            assert valid or which == 0
                                            if not valid:
                                                continue
                                            other = [h0[0] + y, h0[1] + z, h0[2] + x]
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
    for D in (16, 32, 64):
        plan = na.na_plan_info(which, 1, sp, 1, D, kk, dd)
        got = replay(which, L, k, d, plan)
        exp = expected(which, L, k, d)
        assert len(got) == len(set(got)), "a pair is visited twice"
        assert sorted(got) == sorted(exp)

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


def range_bits(lo, hi, width=32):
    lo, hi = max(0, min(width, lo)), max(0, min(width, hi))
    return ((1 << hi) - 1) & ~((1 << lo) - 1) if hi > lo else 0


def segment_bits(G0, G1, y0, z0, ylo, yhi, zlo, zhi):
    zb = range_bits(zlo - z0, zhi - z0) & range_bits(0, G1)
    bits = 0
    for y in range(max(ylo, y0), min(yhi, y0 + G0)):
        bits |= zb << ((y - y0) * G1)
    return bits


def replay(which, L, k, d, plan):
    """Yield (row_global_coords, key_or_query_global_coords) pairs the kernel marks live."""
    T = (plan["T1"], plan["T2"], plan["T3"])
    H = (plan["H1"], plan["H2"], plan["H3"])
    G = (plan["G1"], plan["G2"], plan["G3"])
    NC = plan["NC"]
    NB = G[2] // 8
    assert G[2] % 8 == 0 and 1 <= NB <= 4
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
                for ci in range(nc[0] * nc[1] * nc[2]):
                    cx, r = ci % nc[2], ci // nc[2]
                    cz, cy = r % nc[1], r // nc[1]
                    y0, z0, x0 = cy * G[0], cz * G[1], cx * G[2]
                    useg = segment_bits(G[0], G[1], y0, z0, ulo[0], uhi[0], ulo[1], uhi[1])
                    xa, xb = ulo[2] - x0, uhi[2] - x0
                    ublk = range_bits(xa >> 3, (xb + 7) >> 3) & ((1 << NB) - 1) if xb > xa else 0
                    act = 0
                    for s_ in range(16):
                        if (useg >> s_) & 1:
                            act |= ublk << (s_ * NB)
                    for valid, j, lo, ln in lanes:
                        is_live = all(x > 0 for x in ln)
                        rowseg = segment_bits(G[0], G[1], y0, z0, lo[0], lo[0] + ln[0], lo[1], lo[1] + ln[1]) if is_live else 0
                        m8 = 0
                        for bb in range(NB):
                            m8 |= range_bits(lo[2] - x0 - 8 * bb, lo[2] + ln[2] - x0 - 8 * bb, 8) << (8 * bb)
                        for i in range(NC // 8):
                            if not (act >> i) & 1:
                                continue
                            assert 8 * i + 8 <= NC, "TMEM/P column outside the chunk"
                            seg, bb = i // NB, i % NB
                            if not (rowseg >> seg) & 1:
                                continue
                            byte = (m8 >> (8 * bb)) & 0xFF
                            y, z = y0 + seg // G[1], z0 + seg % G[1]
                            for e in range(8):
                                if (byte >> e) & 1:
                                    assert valid or which == 0
                                    if not valid:
                                        continue
                                    other = [h0[0] + y, h0[1] + z, h0[2] + x0 + 8 * bb + e]
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

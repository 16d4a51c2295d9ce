"""Pins for the fp64 oracle of the unfused operations (CPU only).

The unfused oracle (oracle/unfused.py) is checked against things other than itself: the chain
qk -> softmax -> av must reproduce the fused oracle's forward and the chained gradients its
backward (the fused oracle is pinned on its own in test_oracle.py); every linear operation and its
gradient must satisfy the adjoint identity <dy, A x> = <A^T dy, x>; the offset order of the weights
is read back from an index-coded key tensor and compared with the window re-derived as "the k
same-class positions nearest to i"; softmax_bwd is compared with central finite differences; and
the sampled-row routes (inverse lists) must agree with the full scatter.  The relative positional
bias is checked against dense attention whose bias is looked up from the two tokens' coordinates,
and its gradient against the adjoint identity (the logits are affine in the table) and against
closed-form pair counts.  A dropped scale, a transposed offset order, a wrong inverse list, a sign
error in the softmax gradient or a mirrored bias index fails one of them.
"""
import itertools

import numpy as np
import pytest

import oracle
import oracle.unfused as un
from test_oracle import CASES, nearest_k


def rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def case_tensors(spatial, B, heads, D, seed):
    shape = (B, *spatial, heads, D)
    return [rand(shape, seed + i) for i in range(4)]


@pytest.mark.parametrize("spatial,kernel,dilation,B,heads,D", CASES)
def test_chain_forward_equals_fused_oracle(spatial, kernel, dilation, B, heads, D):
    q, k, v, _ = case_tensors(spatial, B, heads, D, 11)
    scale = 0.37
    attn = un.qk(q, k, kernel, dilation, scale)
    o = un.av(un.softmax(attn), v, kernel, dilation)
    o_ref, _ = oracle.na_fwd(q, k, v, kernel, dilation, scale)
    assert np.abs(o - o_ref).max() <= 1e-12 * max(1.0, np.abs(o_ref).max())


@pytest.mark.parametrize("spatial,kernel,dilation,B,heads,D", CASES)
def test_chain_backward_equals_fused_oracle(spatial, kernel, dilation, B, heads, D):
    q, k, v, dO = case_tensors(spatial, B, heads, D, 21)
    scale = 0.41
    y = un.softmax(un.qk(q, k, kernel, dilation, scale))
    dy, dv = un.av_bwd(dO, y, v, kernel, dilation)
    dx = un.softmax_bwd(y, dy)
    dq, dk = un.qk_bwd(dx, q, k, kernel, dilation, scale)
    dq_ref, dk_ref, dv_ref = oracle.na_bwd(q, k, v, dO, kernel, dilation, scale)
    for got, ref in ((dq, dq_ref), (dk, dk_ref), (dv, dv_ref)):
        assert np.abs(got - ref).max() <= 1e-11 * max(1.0, np.abs(ref).max())


@pytest.mark.parametrize("spatial,kernel,dilation,B,heads,D", CASES)
def test_adjoint_identities(spatial, kernel, dilation, B, heads, D):
    q, k, v, dO = case_tensors(spatial, B, heads, D, 31)
    K = int(np.prod(kernel))
    wshape = (B, *spatial, heads, K)
    a = rand(wshape, 41)
    w = rand(wshape, 42)
    u = rand(q.shape, 43)
    scale = 0.29
    # logits: linear in q for fixed k, and in k for fixed q
    dq, dk = un.qk_bwd(w, q, k, kernel, dilation, scale)
    lhs_q = np.sum(w * un.qk(u, k, kernel, dilation, scale))
    lhs_k = np.sum(w * un.qk(q, u, kernel, dilation, scale))
    assert abs(lhs_q - np.sum(dq * u)) <= 1e-10 * max(1.0, abs(lhs_q))
    assert abs(lhs_k - np.sum(dk * u)) <= 1e-10 * max(1.0, abs(lhs_k))
    # weighted sum: linear in the weights for fixed v, and in v for fixed weights
    dattn, dv = un.av_bwd(dO, a, v, kernel, dilation)
    lhs_a = np.sum(dO * un.av(w, v, kernel, dilation))
    lhs_v = np.sum(dO * un.av(a, u, kernel, dilation))
    assert abs(lhs_a - np.sum(dattn * w)) <= 1e-10 * max(1.0, abs(lhs_a))
    assert abs(lhs_v - np.sum(dv * u)) <= 1e-10 * max(1.0, abs(lhs_v))


@pytest.mark.parametrize("spatial,kernel,dilation", [((13,), (5,), (2,)), ((7, 9), (3, 5), (2, 1)),
                                                     ((5, 6, 7), (3, 1, 5), (1, 3, 1))])
def test_offset_order_from_index_coded_keys(spatial, kernel, dilation):
    """attn[i, t] reads back which key offset t selects: key channel 0 holds the key's token index."""
    N = int(np.prod(spatial))
    q = np.zeros((1, *spatial, 1, 2))
    q[..., 0] = 1.0
    k = np.zeros_like(q)
    k[..., 0] = np.arange(N).reshape(spatial)[..., None]
    attn = un.qk(q, k, kernel, dilation, 1.0).reshape(N, -1)
    strides = [int(np.prod(spatial[a + 1:])) for a in range(len(spatial))]
    for tok, x in enumerate(itertools.product(*[range(L) for L in spatial])):
        per_axis = [nearest_k(x[a], spatial[a], kernel[a], dilation[a]) for a in range(len(spatial))]
        want = [sum(p * s for p, s in zip(nb, strides)) for nb in itertools.product(*per_axis)]
        assert attn[tok].tolist() == want, (x, attn[tok], want)


def test_softmax_bwd_matches_finite_differences():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 7))
    dy = rng.standard_normal((3, 7))
    dx = un.softmax_bwd(un.softmax(x), dy)
    h = 1e-6
    fd = np.zeros_like(x)
    for r in range(x.shape[0]):
        for t in range(x.shape[1]):
            e = np.zeros_like(x)
            e[r, t] = h
            fd[r, t] = np.sum(dy * (un.softmax(x + e) - un.softmax(x - e))) / (2 * h)
    assert np.abs(dx - fd).max() <= 1e-8


def test_softmax_rows_are_distributions_and_shift_invariant():
    x = rand((4, 5, 9), 6) * 30
    y = un.softmax(x)
    assert np.all(y > 0)
    assert np.abs(y.sum(-1) - 1).max() <= 1e-14
    assert np.abs(un.softmax(x + 123.0) - y).max() <= 1e-14


@pytest.mark.parametrize("spatial,kernel,dilation,B,heads,D", [CASES[2], CASES[4], CASES[6], CASES[7]])
def test_sampled_rows_match_full(spatial, kernel, dilation, B, heads, D):
    q, k, v, dO = case_tensors(spatial, B, heads, D, 51)
    K = int(np.prod(kernel))
    w = rand((B, *spatial, heads, K), 52)
    total = B * int(np.prod(spatial)) * heads
    rows = np.random.default_rng(53).choice(total, size=min(total, 17), replace=False)
    flat = lambda t: t.reshape(total, -1)[rows]
    scale = 0.5
    assert np.allclose(un.qk(q, k, kernel, dilation, scale, rows), flat(un.qk(q, k, kernel, dilation, scale)),
                       rtol=0, atol=1e-12)
    assert np.allclose(un.av(w, v, kernel, dilation, rows), flat(un.av(w, v, kernel, dilation)), rtol=0, atol=1e-12)
    assert np.allclose(un.softmax(w, rows), flat(un.softmax(w)), rtol=0, atol=1e-15)
    assert np.allclose(un.softmax_bwd(w, q[..., :1].repeat(K, -1), rows),
                       flat(un.softmax_bwd(w, q[..., :1].repeat(K, -1))), rtol=0, atol=1e-12)
    for got, full in zip(un.qk_bwd(w, q, k, kernel, dilation, scale, rows),
                         un.qk_bwd(w, q, k, kernel, dilation, scale)):
        assert np.allclose(got, flat(full), rtol=0, atol=1e-12)
    for got, full in zip(un.av_bwd(dO, w, v, kernel, dilation, rows), un.av_bwd(dO, w, v, kernel, dilation)):
        assert np.allclose(got, flat(full), rtol=0, atol=1e-12)


def test_inverse_lists_cover_every_pair_once():
    g = un.Geometry((9, 10), (3, 5), (2, 1))
    nb = g.neighbours(np.arange(g.N))
    pairs = set()
    for j in range(g.N):
        qs, ts = g.inverse(j)
        for qi, t in zip(qs.tolist(), ts.tolist()):
            assert nb[qi, t] == j
            pairs.add((qi, t))
    assert len(pairs) == g.N * g.K


# ---------------------------------------------------------------------------------------------
# Relative positional bias
# ---------------------------------------------------------------------------------------------

def dense_bias(spatial, kernel, dilation, table):
    """[heads, N, N] dense bias: for key j in query i's window (nearest-k-in-class characterisation),
    table[h, ((y_a - x_a) / d_a + k_a - 1)_a] from the two tokens' coordinates; -inf elsewhere."""
    coords = list(itertools.product(*[range(L) for L in spatial]))
    N = len(coords)
    heads = table.shape[0]
    out = np.full((heads, N, N), -np.inf)
    for i, x in enumerate(coords):
        per_axis = [nearest_k(x[a], spatial[a], kernel[a], dilation[a]) for a in range(len(spatial))]
        for y in itertools.product(*per_axis):
            j = coords.index(y)
            rel = tuple((y[a] - x[a]) // dilation[a] + kernel[a] - 1 for a in range(len(spatial)))
            out[:, i, j] = table[(slice(None),) + rel]
    return out


@pytest.mark.parametrize("spatial,kernel,dilation,B,heads,D", [CASES[0], CASES[2], CASES[4], CASES[6]])
def test_rpb_chain_matches_dense_attention_with_bias(spatial, kernel, dilation, B, heads, D):
    q, k, v, _ = case_tensors(spatial, B, heads, D, 61)
    table = rand((heads,) + tuple(2 * kk - 1 for kk in kernel), 62)
    scale = 0.33
    o = un.av(un.softmax(un.qk(q, k, kernel, dilation, scale, rpb=table)), v, kernel, dilation)
    N = int(np.prod(spatial))
    qf, kf, vf = (x.reshape(B, N, heads, D) for x in (q, k, v))
    s = scale * np.einsum("bihc,bjhc->bhij", qf, kf) + dense_bias(spatial, kernel, dilation, table)[None]
    p = np.exp(s - s.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    ref = np.einsum("bhij,bjhc->bihc", p, vf).reshape(o.shape)
    assert np.abs(o - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


@pytest.mark.parametrize("spatial,kernel,dilation,B,heads,D", CASES)
def test_rpb_grad_is_the_adjoint_of_the_bias(spatial, kernel, dilation, B, heads, D):
    """The logits are affine in the table: <dattn, qk(rpb) - qk(0)> = <rpb_grad(dattn), rpb>."""
    q, k, _, _ = case_tensors(spatial, B, heads, D, 71)
    K = int(np.prod(kernel))
    table = rand((heads,) + tuple(2 * kk - 1 for kk in kernel), 72)
    w = rand((B, *spatial, heads, K), 73)
    diff = un.qk(q, k, kernel, dilation, 0.5, rpb=table) - un.qk(q, k, kernel, dilation, 0.5)
    lhs = np.sum(w * diff)
    rhs = np.sum(un.rpb_grad(w, kernel, dilation) * table)
    assert abs(lhs - rhs) <= 1e-10 * max(1.0, abs(lhs))


def test_rpb_constant_per_head_leaves_probabilities_unchanged():
    spatial, kernel, dilation = (9, 10), (3, 5), (2, 1)
    q, k, _, _ = case_tensors(spatial, 1, 3, 4, 81)
    table = np.zeros((3, 5, 9)) + np.array([1.5, -2.0, 7.0])[:, None, None]
    a = un.softmax(un.qk(q, k, kernel, dilation, 0.7, rpb=table))
    b = un.softmax(un.qk(q, k, kernel, dilation, 0.7))
    assert np.abs(a - b).max() <= 1e-14


def test_rpb_sampled_rows_match_full():
    spatial, kernel, dilation = (5, 4, 7), (1, 3, 3), (2, 1, 2)
    q, k, _, _ = case_tensors(spatial, 2, 2, 4, 91)
    table = rand((2, 1, 5, 5), 92)
    total = 2 * int(np.prod(spatial)) * 2
    rows = np.random.default_rng(93).choice(total, size=19, replace=False)
    full = un.qk(q, k, kernel, dilation, 0.4, rpb=table).reshape(total, -1)[rows]
    assert np.allclose(un.qk(q, k, kernel, dilation, 0.4, rows, rpb=table), full, rtol=0, atol=1e-12)


def test_rpb_grad_counts_pairs_per_relative_position():
    """With dattn = 1 everywhere, drpb counts the (batch, query, offset) pairs at each relative
    position: summed over the table it is B * N * K per head, and in a 1D interior-only case each
    of the k centred offsets gets every query."""
    spatial, kernel, dilation = (9, 10), (3, 5), (2, 1)
    g = un.Geometry(spatial, kernel, dilation)
    ones = np.ones((2, *spatial, 3, g.K))
    d = un.rpb_grad(ones, kernel, dilation)
    assert np.allclose(d.reshape(3, -1).sum(-1), 2 * g.N * g.K)
    d1 = un.rpb_grad(np.ones((1, 5, 1, 5)), (5,), (1,))      # L = k: every query's window is the whole axis
    assert d1.reshape(-1).tolist() == [1, 2, 3, 4, 5, 4, 3, 2, 1]


# ---------------------------------------------------------------------------------------------
# Variable windows (kernel sizes that change along an axis)
# ---------------------------------------------------------------------------------------------

def dense_variable_mask(spatial, sizes, dilation):
    """[N, N] boolean: key j is kept for query i when, along every axis, j's coordinate is one of the
    k_a(i) same-class positions nearest to i's (the nearest-k characterisation with the query's own k)."""
    coords = list(itertools.product(*[range(L) for L in spatial]))
    index = {c: n for n, c in enumerate(coords)}
    N = len(coords)
    out = np.zeros((N, N), dtype=bool)
    for i, x in enumerate(coords):
        per_axis = [nearest_k(x[a], spatial[a], int(sizes[a][x[a]]), dilation[a]) for a in range(len(spatial))]
        for y in itertools.product(*per_axis):
            out[i, index[y]] = True
    return out


VARWIN = [
    # spatial, kernel, dilation, sizes per axis (None: the full kernel everywhere)
    ((11,), (5,), (1,), [[1, 1, 3, 3, 5, 5, 5, 3, 3, 1, 1]]),
    ((9, 10), (3, 5), (2, 1), [[1, 3, 1, 3, 3, 1, 3, 1, 3], None]),
    ((6, 5, 7), (5, 3, 3), (1, 1, 2), [[1, 1, 3, 3, 5, 5], None, [3, 1, 3, 1, 3, 1, 3]]),
]


def _sizes(spatial, kernel, sizes):
    return [np.full(L, k) if s is None else np.asarray(s) for L, k, s in zip(spatial, kernel, sizes)]


@pytest.mark.parametrize("spatial,kernel,dilation,sizes", VARWIN)
def test_variable_window_chain_matches_dense_attention(spatial, kernel, dilation, sizes):
    B, heads, D = 2, 2, 3
    q, k, v, _ = case_tensors(spatial, B, heads, D, 101)
    sz = _sizes(spatial, kernel, sizes)
    scale = 0.45
    logits = un.mask_window(un.qk(q, k, kernel, dilation, scale), sz, kernel, dilation)
    o = un.av(un.softmax(logits), v, kernel, dilation)
    N = int(np.prod(spatial))
    qf, kf, vf = (x.reshape(B, N, heads, D) for x in (q, k, v))
    s = scale * np.einsum("bihc,bjhc->bhij", qf, kf)
    s = np.where(dense_variable_mask(spatial, sz, dilation)[None, None], s, -np.inf)
    p = np.exp(s - s.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    ref = np.einsum("bhij,bjhc->bihc", p, vf).reshape(o.shape)
    assert np.abs(o - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


def test_variable_window_special_cases():
    spatial, kernel, dilation = (7, 8), (5, 3), (1, 2)
    q, k, v, _ = case_tensors(spatial, 1, 2, 4, 111)
    logits = un.qk(q, k, kernel, dilation, 0.5)
    full = un.mask_window(logits, _sizes(spatial, kernel, [None, None]), kernel, dilation)
    assert np.array_equal(full, logits)                        # the full kernel everywhere masks nothing
    ones = [np.ones(7, dtype=int), np.ones(8, dtype=int)]
    o = un.av(un.softmax(un.mask_window(logits, ones, kernel, dilation)), v, kernel, dilation)
    assert np.abs(o - v).max() <= 1e-14                         # kernel 1: each query sees only itself

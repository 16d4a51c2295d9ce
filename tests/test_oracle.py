"""Pins for the fp64 oracle (CPU only).

None of these checks reuses the oracle's own formulas: the window is re-derived as "the k
same-class positions nearest to i", dense attention is built from that mask with numpy, the
backward is checked against torch autograd of the dense formulation and against central finite
differences, and special cases are checked against their closed forms.  A mistake anywhere in
the oracle (window start, class length, clamp, scale, LSE base, a sign or an index in dS, a
missing term in dK or dV) fails at least one of them; test_oracle_mutants.py shows that.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------------------------------------
# Independent characterisation of the neighbourhood
# ---------------------------------------------------------------------------------------------

def nearest_k(i, L, k, d):
    """The k positions of i's residue class closest to i (no ties possible for odd k)."""
    cls = [p for p in range(L) if p % d == i % d]
    order = sorted(cls, key=lambda p: abs(p - i))
    sel = order[:k]
    if len(order) > k:
        assert abs(order[k] - i) > abs(order[k - 1] - i), "tie at the cut"
    return sorted(sel)


def dense_mask(spatial, kernel, dilation):
    """[N, N] boolean: mask[i, j] is True when token j is a neighbour of token i."""
    axes = []
    for L, k, d in zip(spatial, kernel, dilation):
        m = np.zeros((L, L), dtype=bool)
        for i in range(L):
            m[i, nearest_k(i, L, k, d)] = True
        axes.append(m)
    full = axes[0]
    for m in axes[1:]:
        full = np.einsum("ab,cd->acbd", full, m).reshape(full.shape[0] * m.shape[0], -1)
    return full


def dense_fwd(q, k, v, mask, scale):
    """Dense masked softmax attention, fp64.  q,k,v: [B, N, h, D]."""
    s = scale * np.einsum("bihc,bjhc->bhij", q, k)
    s = np.where(mask[None, None], s, -np.inf)
    m = s.max(-1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(-1, keepdims=True)
    p = e / l
    o = np.einsum("bhij,bjhc->bihc", p, v)
    lse = (m + np.log(l))[..., 0]                 # [B, h, N]
    return o, lse.transpose(0, 2, 1)


def rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


CASES = [
    # spatial, kernel, dilation, B, heads, D
    ((13,), (5,), (1,), 1, 2, 4),
    ((13,), (3,), (2,), 2, 1, 3),
    ((16,), (3,), (3,), 1, 2, 5),          # 16 = 5*3 + 1: classes of unequal length
    ((7, 8), (3, 5), (1, 1), 1, 2, 4),
    ((9, 10), (3, 3), (2, 3), 2, 1, 6),    # 10 not divisible by 3
    ((8, 8), (7, 1), (1, 4), 1, 1, 4),
    ((4, 6, 5), (3, 3, 5), (1, 2, 1), 1, 2, 3),
    ((5, 4, 7), (1, 3, 3), (2, 1, 2), 2, 1, 4),
]


# ---------------------------------------------------------------------------------------------
# Neighbourhood
# ---------------------------------------------------------------------------------------------

def test_window_is_nearest_k_in_class():
    for L in range(1, 40):
        for d in range(1, 5):
            for k in range(1, L // d + 1, 2):
                for i in range(L):
                    f = oracle.first_neighbour(i, L, k, d)
                    got = [f + d * t for t in range(k)]
                    assert got == nearest_k(i, L, k, d), (L, k, d, i)


def test_window_rejects_invalid():
    assert oracle.first_neighbour(0, 5, 2, 1) == -1       # even kernel
    assert oracle.first_neighbour(0, 5, 7, 1) == -1       # kernel longer than the axis
    assert oracle.first_neighbour(0, 9, 5, 2) == -1       # class of 4 positions < 5
    assert oracle.first_neighbour(5, 5, 3, 1) == -1       # index out of range


@pytest.mark.parametrize("spatial,kernel,dilation,B,heads,D", CASES)
def test_every_query_sees_k_keys_and_inverse_counts(spatial, kernel, dilation, B, heads, D):
    mask = dense_mask(spatial, kernel, dilation)
    K = int(np.prod(kernel))
    assert (mask.sum(1) == K).all()
    assert mask.sum() == mask.shape[0] * K


# ---------------------------------------------------------------------------------------------
# Forward
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("spatial,kernel,dilation,B,heads,D", CASES)
def test_fwd_matches_dense_masked_attention(spatial, kernel, dilation, B, heads, D):
    shape = (B, *spatial, heads, D)
    q, k, v = rand(shape, 1), rand(shape, 2), rand(shape, 3)
    scale = 0.37
    o, lse = oracle.na_fwd(q, k, v, kernel, dilation, scale)
    N = int(np.prod(spatial))
    mask = dense_mask(spatial, kernel, dilation)
    ro, rlse = dense_fwd(q.reshape(B, N, heads, D), k.reshape(B, N, heads, D),
                         v.reshape(B, N, heads, D), mask, scale)
    np.testing.assert_allclose(o.reshape(B, N, heads, D), ro, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse.reshape(B, N, heads), rlse, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("spatial", [(9,), (5, 7), (3, 5, 5)])
def test_fwd_kernel_equal_extent_is_full_attention(spatial):
    B, heads, D = 2, 2, 5
    shape = (B, *spatial, heads, D)
    q, k, v = rand(shape, 4), rand(shape, 5), rand(shape, 6)
    kernel = tuple(spatial)
    scale = D ** -0.5
    o, lse = oracle.na_fwd(q, k, v, kernel, (1,) * len(spatial), scale)
    N = int(np.prod(spatial))
    qq, kk, vv = (x.reshape(B, N, heads, D) for x in (q, k, v))
    s = scale * np.einsum("bihc,bjhc->bhij", qq, kk)
    p = np.exp(s - s.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    ref = np.einsum("bhij,bjhc->bihc", p, vv)
    np.testing.assert_allclose(o.reshape(B, N, heads, D), ref, rtol=1e-11, atol=1e-12)
    ref_lse = np.log(np.exp(s).sum(-1)).transpose(0, 2, 1)
    np.testing.assert_allclose(lse.reshape(B, N, heads), ref_lse, rtol=1e-11, atol=1e-12)


def test_fwd_kernel_one_is_identity():
    shape = (2, 6, 7, 3, 4)
    q, k, v = rand(shape, 7), rand(shape, 8), rand(shape, 9)
    o, lse = oracle.na_fwd(q, k, v, (1, 1), (1, 2), 0.5)
    np.testing.assert_array_equal(o, v)
    np.testing.assert_allclose(lse, 0.5 * (q * k).sum(-1), rtol=1e-13, atol=1e-13)


def test_fwd_constant_values_pass_through():
    shape = (1, 9, 8, 2, 3)
    q, k = rand(shape, 10), rand(shape, 11)
    v = np.broadcast_to(np.array([1.5, -2.0, 0.25]), shape).copy()
    o, _ = oracle.na_fwd(q, k, v, (5, 3), (1, 2), 1.0)
    np.testing.assert_allclose(o, v, rtol=1e-13, atol=1e-13)


def test_fwd_dilation_splits_into_residue_subproblems():
    spatial, kernel, dilation = (12, 10), (3, 3), (3, 2)
    shape = (1, *spatial, 2, 4)
    q, k, v = rand(shape, 12), rand(shape, 13), rand(shape, 14)
    o, lse = oracle.na_fwd(q, k, v, kernel, dilation, 0.3)
    for c1 in range(3):
        for c2 in range(2):
            sl = (slice(None), slice(c1, None, 3), slice(c2, None, 2))
            so, slse = oracle.na_fwd(q[sl], k[sl], v[sl], kernel, (1, 1), 0.3)
            np.testing.assert_allclose(o[sl], so, rtol=1e-13, atol=1e-13)
            np.testing.assert_allclose(lse[sl], slse, rtol=1e-13, atol=1e-13)


def test_fwd_interior_translation_equivariance():
    spatial, kernel = (20,), (5,)
    shape = (1, 20, 1, 3)
    q, k, v = rand(shape, 15), rand(shape, 16), rand(shape, 17)
    o, _ = oracle.na_fwd(q, k, v, kernel, (1,), 0.7)
    sh = lambda x: np.roll(x, 3, axis=1)
    o2, _ = oracle.na_fwd(sh(q), sh(k), sh(v), kernel, (1,), 0.7)
    # queries whose windows stay interior in both layouts
    np.testing.assert_allclose(o2[:, 2 + 3:17], o[:, 2:17 - 3], rtol=1e-13, atol=1e-13)


def test_fwd_rows_subset_matches_full():
    shape = (2, 7, 6, 3, 4)
    q, k, v = rand(shape, 18), rand(shape, 19), rand(shape, 20)
    o, lse = oracle.na_fwd(q, k, v, (3, 5), (2, 1), 0.4)
    rows = np.array([0, 5, 17, 100, 251, 2 * 42 * 3 - 1])
    so, slse = oracle.na_fwd(q, k, v, (3, 5), (2, 1), 0.4, rows=rows)
    np.testing.assert_array_equal(so, o.reshape(-1, 4)[rows])
    np.testing.assert_array_equal(slse, lse.reshape(-1)[rows])


def test_fwd_bf16_inputs_are_read_exactly():
    t = torch.randn(1, 6, 6, 2, 4, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    bits = t.view(torch.int16).numpy().view(np.uint16)
    f32 = t.float().numpy()
    a = oracle.na_fwd(bits, bits, bits, (3, 3), (1, 1), 0.5)
    b = oracle.na_fwd(f32, f32, f32, (3, 3), (1, 1), 0.5)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_fwd_rejects_invalid():
    x = np.zeros((1, 8, 1, 2), dtype=np.float32)
    with pytest.raises(ValueError):
        oracle.na_fwd(x, x, x, (4,), (1,), 1.0)          # even kernel
    with pytest.raises(ValueError):
        oracle.na_fwd(x, x, x, (5,), (2,), 1.0)          # class of 4 < 5


# ---------------------------------------------------------------------------------------------
# Backward
# ---------------------------------------------------------------------------------------------

def dense_torch_grads(q, k, v, dO, mask, scale):
    """Autograd of the dense masked formulation (torch float64, CPU)."""
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    s = scale * torch.einsum("bihc,bjhc->bhij", tq, tk)
    s = s.masked_fill(~torch.tensor(mask)[None, None], float("-inf"))
    p = torch.softmax(s, dim=-1)
    o = torch.einsum("bhij,bjhc->bihc", p, tv)
    o.backward(torch.tensor(dO, dtype=torch.float64))
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


@pytest.mark.parametrize("spatial,kernel,dilation,B,heads,D", CASES)
def test_bwd_matches_dense_autograd(spatial, kernel, dilation, B, heads, D):
    shape = (B, *spatial, heads, D)
    q, k, v, dO = rand(shape, 21), rand(shape, 22), rand(shape, 23), rand(shape, 24)
    scale = 0.45
    dq, dk, dv = oracle.na_bwd(q, k, v, dO, kernel, dilation, scale)
    N = int(np.prod(spatial))
    flat = lambda x: x.reshape(B, N, heads, D)
    rq, rk, rv = dense_torch_grads(flat(q), flat(k), flat(v), flat(dO), dense_mask(spatial, kernel, dilation), scale)
    np.testing.assert_allclose(flat(dq), rq, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(flat(dk), rk, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(flat(dv), rv, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("spatial,kernel,dilation", [((7,), (3,), (2,)), ((5, 6), (3, 3), (1, 2)),
                                                     ((3, 4, 4), (3, 1, 3), (1, 2, 1))])
def test_bwd_matches_finite_differences(spatial, kernel, dilation):
    B, heads, D = 1, 1, 3
    shape = (B, *spatial, heads, D)
    q, k, v = rand(shape, 25), rand(shape, 26), rand(shape, 27)
    G = rand(shape, 28)
    scale = 0.6
    dq, dk, dv = oracle.na_bwd(q, k, v, G, kernel, dilation, scale)

    def loss(qq, kk, vv):
        return float((oracle.na_fwd(qq, kk, vv, kernel, dilation, scale)[0] * G).sum())

    h = 1e-6
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        fd = np.zeros(shape)
        for idx in itertools.product(*[range(s) for s in shape]):
            args = [q.copy(), k.copy(), v.copy()]
            args[which][idx] += h
            lp = loss(*args)
            args[which][idx] -= 2 * h
            lm = loss(*args)
            fd[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-8)


def test_bwd_dv_column_sums_and_constant_keys():
    shape = (2, 9, 7, 2, 4)
    q, k, v, dO = rand(shape, 29), rand(shape, 30), rand(shape, 31), rand(shape, 32)
    dq, dk, dv = oracle.na_bwd(q, k, v, dO, (5, 3), (1, 2), 0.5)
    # rows of P sum to one, so the dV rows sum to the dO rows (per batch and head)
    np.testing.assert_allclose(dv.sum(axis=(1, 2)), dO.sum(axis=(1, 2)), rtol=1e-11, atol=1e-11)
    # dS rows sum to zero, so with every key equal dQ vanishes
    kc = np.broadcast_to(rand((1, 1, 1, 2, 4), 33), shape).copy()
    dq0, _, _ = oracle.na_bwd(q, kc, v, dO, (5, 3), (1, 2), 0.5)
    np.testing.assert_allclose(dq0, 0.0, atol=1e-12)


def test_bwd_sampled_rows_match_full():
    shape = (2, 8, 9, 3, 4)
    q, k, v, dO = rand(shape, 34), rand(shape, 35), rand(shape, 36), rand(shape, 37)
    args = ((3, 5), (2, 1), 0.3)
    dq, dk, dv = oracle.na_bwd(q, k, v, dO, *args)
    qrows = np.array([0, 7, 50, 211, 431])
    krows = np.array([1, 3, 99, 300, 431, 8])
    sdq, sdk, sdv = oracle.na_bwd(q, k, v, dO, *args, qrows=qrows, krows=krows)
    np.testing.assert_allclose(sdq, dq.reshape(-1, 4)[qrows], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(sdk, dk.reshape(-1, 4)[krows], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(sdv, dv.reshape(-1, 4)[krows], rtol=1e-13, atol=1e-14)

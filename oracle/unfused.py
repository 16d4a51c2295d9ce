"""Plain fp64 CPU oracle for the unfused neighborhood-attention operations.

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the benchmark's CPU baseline
may import this module; the library itself never does.  It shares no code with the CUDA library.

NATTEN issue #161 ("Backward pass is very slow towards much tokens and large kernels") runs the
unfused chain beside the fused operation: ``na2d_qk`` gives the attention logits of every query over
its window, a softmax over the window's weights follows, and ``na2d_av`` sums the values with those
weights (the user's benchmark script); the maintainer's profile of its backward lists the gradient
kernels for the logits' inputs (QGRAD, KGRAD), the weights (AGRAD) and the values (VGRAD).  This
module writes each of those operations out as its definition over the neighbour sets of the fused
oracle (``oracle.first_neighbour``):

* qk:           attn[i, t] = scale * q_i . k_{n(i, t)}
* softmax:      y[i, t] = exp(x[i, t]) / sum_u exp(x[i, u])  (max-shifted, which changes nothing)
* av:           o_i = sum_t attn[i, t] v_{n(i, t)}
* softmax_bwd:  dx[i, t] = y[i, t] (dy[i, t] - sum_u y[i, u] dy[i, u])
* qk_bwd:       dq_i = scale * sum_t dattn[i, t] k_{n(i, t)};  dk_j = scale * sum_{(i, t): n(i, t) = j} dattn[i, t] q_i
* av_bwd:       dattn[i, t] = dO_i . v_{n(i, t)};  dv_j = sum_{(i, t): n(i, t) = j} attn[i, t] dO_i

Relative positional bias (the maintainer's profile names the logits kernel QKRPB): an optional table
rpb[heads, 2 k_0 - 1, .., 2 k_{n-1} - 1] adds rpb[h, (c(n(i, t))_a - c(i)_a + k_a - 1)_a] to attn[i, t],
where c(.)_a is a position's class index along axis a (its index divided by the dilation).  Its
gradient is drpb[h, r] = sum over (batch, query, offset) with relative position r of dattn[i, t].

Variable windows (the user's request for kernel sizes that change along time, answered with "mask
the weights" of the unfused logits): per axis a and position x, a kernel size k_a(x) <= k_a.  Query i
keeps only the keys its own window of size k_a(i_a) (the same shifted-window rule, nested inside the
full window) holds along every axis; mask_window sets the other logits to -inf.

n(i, t) is the t-th key of query i's window: the window is the Cartesian product of the per-axis
windows, and t = (t_0 k_1 + t_1) k_2 + t_2 orders its offsets with the first axis outermost.  The
weight tensors are [B, L.., heads, K].

Sampled rows: with ``rows`` (flat indices (b * N + token) * heads + head) the gather operations
compute only those rows, and dk/dv on sampled key rows collect their queries from the per-axis
inverse lists (every query whose window along an axis holds the key's index there), while the full
tensors come from a scatter over every (query, offset) pair.  The two routes are independent ways
to the same sums and the tests compare them.

Parity pins (tests/test_oracle_unfused.py): the chain qk -> softmax -> av equals the fused oracle's
forward and the chained gradients equal its backward (the fused oracle is pinned on its own against
dense masked attention and finite differences); each linear operation passes the adjoint identity
<dy, A x> = <A^T dy, x> against its gradient; the offset order is checked against an index-coded
key tensor; softmax_bwd against central finite differences.
"""
from __future__ import annotations

import numpy as np

from . import first_neighbour


def axis_table(L: int, k: int, d: int) -> np.ndarray:
    """[L, k] spatial indices of each position's neighbours along one axis, in window order."""
    out = np.empty((L, k), dtype=np.int64)
    for i in range(L):
        f = first_neighbour(i, L, k, d)
        if f < 0:
            raise ValueError("invalid window for this axis")
        out[i] = f + d * np.arange(k)
    return out


class Geometry:
    """Per-axis neighbour tables of one problem; token indices are row-major over the spatial axes."""

    def __init__(self, spatial, kernel, dilation):
        self.spatial = tuple(int(s) for s in spatial)
        self.kernel = tuple(int(x) for x in kernel)
        self.dilation = tuple(int(x) for x in dilation)
        if not (len(self.spatial) == len(self.kernel) == len(self.dilation)):
            raise ValueError("spatial, kernel and dilation need the same length")
        self.tabs = [axis_table(L, k, d) for L, k, d in zip(self.spatial, self.kernel, self.dilation)]
        self.N = int(np.prod(self.spatial))
        self.K = int(np.prod(self.kernel))
        self.strides = [int(np.prod(self.spatial[a + 1:])) for a in range(len(self.spatial))]

    def coords(self, tok: np.ndarray) -> np.ndarray:
        """[n, ndim] spatial coordinates of token indices."""
        return np.stack(np.unravel_index(np.asarray(tok, dtype=np.int64), self.spatial), axis=-1)

    def neighbours(self, tok: np.ndarray) -> np.ndarray:
        """[n, K] token indices of the keys of each query token, offsets in window order."""
        x = self.coords(tok)
        n = x.shape[0]
        idx = np.zeros((n,) + (1,) * len(self.kernel), dtype=np.int64)
        for a, tab in enumerate(self.tabs):
            shape = [n] + [1] * len(self.kernel)
            shape[1 + a] = self.kernel[a]
            idx = idx + (tab[x[:, a]] * self.strides[a]).reshape(shape)
        return idx.reshape(n, self.K)

    def inverse(self, tok: int):
        """(query tokens, offsets) of every query whose window holds key token `tok`."""
        x = self.coords(np.array([tok]))[0]
        per_axis = []
        for a, tab in enumerate(self.tabs):
            qi, ti = np.nonzero(tab == x[a])
            per_axis.append((qi, ti))
        queries = np.zeros(1, dtype=np.int64)
        offsets = np.zeros(1, dtype=np.int64)
        for a, (qi, ti) in enumerate(per_axis):
            queries = (queries[:, None] + qi[None, :] * self.strides[a]).ravel()
            offsets = (offsets[:, None] * self.kernel[a] + ti[None, :]).ravel()
        return queries, offsets


def _split(x):
    """View [B, L.., heads, C] as [B, N, heads, C].  float32 inputs stay float32 here (exact for
    bf16 and fp16 values, and half the host memory at full size); every operand is widened to
    float64 by _f64 once gathered, before any arithmetic."""
    x = np.asarray(x)
    if x.dtype not in (np.float32, np.float64):
        raise TypeError(f"unsupported input dtype {x.dtype}: pass float32 or float64")
    return x.reshape(x.shape[0], -1, x.shape[-2], x.shape[-1])


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def _rows_of(rows, B, N, heads):
    r = np.asarray(rows, dtype=np.int64).ravel()
    return r // heads // N, (r // heads) % N, r % heads


def relative_index(g, tok):
    """[n, K] flat index into one head's bias table of every (query token, offset) pair: per axis the
    key's class index minus the query's, plus k - 1, flattened with the first axis outermost."""
    x = g.coords(tok)
    n = x.shape[0]
    idx = np.zeros((n,) + (1,) * len(g.kernel), dtype=np.int64)
    for a, tab in enumerate(g.tabs):
        d, k = g.dilation[a], g.kernel[a]
        rel = tab[x[:, a]] // d - (x[:, a] // d)[:, None] + (k - 1)       # [n, k_a]
        assert rel.min() >= 0 and rel.max() <= 2 * k - 2
        span = int(np.prod([2 * kk - 1 for kk in g.kernel[a + 1:]]))
        shape = [n] + [1] * len(g.kernel)
        shape[1 + a] = k
        idx = idx + (rel * span).reshape(shape)
    return idx.reshape(n, g.K)


def qk(q, k, kernel, dilation, scale, rows=None, rpb=None):
    """Attention logits: [B, L.., heads, K], or [len(rows), K] for sampled rows.  rpb (optional):
    [heads, 2 k_0 - 1, ..] bias table added to every logit at its relative position."""
    qf, kf = _split(q), _split(k)
    B, N, heads, _ = qf.shape
    g = Geometry(q.shape[1:-2], kernel, dilation)
    table = None if rpb is None else _f64(rpb).reshape(heads, -1)
    if rows is None:
        nb = g.neighbours(np.arange(N))                       # [N, K]
        out = scale * np.einsum("bnhc,bnthc->bnht", _f64(qf), _f64(kf[:, nb]))
        if table is not None:
            rel = relative_index(g, np.arange(N))             # [N, K]
            out = out + table[:, rel].transpose(1, 0, 2)[None]
        return out.reshape(tuple(q.shape[:-1]) + (g.K,))
    b, tok, h = _rows_of(rows, B, N, heads)
    nb = g.neighbours(tok)
    out = scale * np.einsum("rc,rtc->rt", _f64(qf[b, tok, h]), _f64(kf[b[:, None], nb, h[:, None]]))
    if table is not None:
        out = out + table[h[:, None], relative_index(g, tok)]
    return out


def rpb_grad(dattn, kernel, dilation):
    """Gradient of the bias table given the logits' gradient dattn [B, L.., heads, K]: a sum over
    batch, queries and offsets of dattn at each relative position, [heads, 2 k_0 - 1, ..]."""
    wf = _split(dattn)
    B, N, heads, K = wf.shape
    g = Geometry(dattn.shape[1:-2], kernel, dilation)
    rel = relative_index(g, np.arange(N))                     # [N, K]
    size = int(np.prod([2 * kk - 1 for kk in g.kernel]))
    out = np.zeros((heads, size), dtype=np.float64)
    for h in range(heads):
        out[h] = np.bincount(rel.ravel(), weights=_f64(wf[:, :, h, :]).sum(axis=0).ravel(), minlength=size)
    return out.reshape((heads,) + tuple(2 * kk - 1 for kk in g.kernel))


def av(attn, v, kernel, dilation, rows=None):
    """Weighted sums of the values: [B, L.., heads, D], or [len(rows), D]."""
    vf = _split(v)
    af = _split(attn)
    B, N, heads, D = vf.shape
    g = Geometry(v.shape[1:-2], kernel, dilation)
    if rows is None:
        nb = g.neighbours(np.arange(N))
        out = np.einsum("bnht,bnthc->bnhc", _f64(af), _f64(vf[:, nb]))
        return out.reshape(v.shape)
    b, tok, h = _rows_of(rows, B, N, heads)
    nb = g.neighbours(tok)
    return np.einsum("rt,rtc->rc", _f64(af[b, tok, h]), _f64(vf[b[:, None], nb, h[:, None]]))


def softmax(x, rows=None):
    """Softmax over the last axis (the window's K weights)."""
    x = np.asarray(x)
    if rows is not None:
        x = x.reshape(-1, x.shape[-1])[np.asarray(rows, dtype=np.int64).ravel()]
    x = _f64(x)
    e = np.exp(x - x.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def softmax_bwd(y, dy, rows=None):
    """Gradient of the window softmax given its output y and the output's gradient dy."""
    y, dy = np.asarray(y), np.asarray(dy)
    if rows is not None:
        r = np.asarray(rows, dtype=np.int64).ravel()
        y, dy = y.reshape(-1, y.shape[-1])[r], dy.reshape(-1, dy.shape[-1])[r]
    y, dy = _f64(y), _f64(dy)
    return y * (dy - (y * dy).sum(axis=-1, keepdims=True))


def _gather(w, src, g, rows, B, N, heads):
    """sum_t w[i, t] src_{n(i, t)} for every row (rows=None) or the sampled rows."""
    if rows is None:
        nb = g.neighbours(np.arange(N))
        return np.einsum("bnht,bnthc->bnhc", _f64(w), _f64(src[:, nb]))
    b, tok, h = _rows_of(rows, B, N, heads)
    nb = g.neighbours(tok)
    return np.einsum("rt,rtc->rc", _f64(w[b, tok, h]), _f64(src[b[:, None], nb, h[:, None]]))


def _scatter(w, src, g, rows, B, N, heads):
    """sum over (i, t) with n(i, t) = j of w[i, t] src_i, for every key j (rows=None: a scatter over
    all pairs) or the sampled key rows (their inverse lists)."""
    D = src.shape[-1]
    if rows is None:
        nb = g.neighbours(np.arange(N))                       # [N, K]
        out = np.zeros(src.shape, dtype=np.float64)
        for t in range(g.K):
            contrib = _f64(w[:, :, :, t, None]) * _f64(src)   # [B, N, heads, D]
            np.add.at(out, (slice(None), nb[:, t]), contrib)
        return out
    b, tok, h = _rows_of(rows, B, N, heads)
    out = np.zeros((b.size, D), dtype=np.float64)
    for r in range(b.size):
        qs, ts = g.inverse(int(tok[r]))
        out[r] = np.einsum("n,nc->c", _f64(w[b[r], qs, h[r], ts]), _f64(src[b[r], qs, h[r]]))
    return out


def qk_bwd(dattn, q, k, kernel, dilation, scale, rows=None):
    """(dq, dk) of qk given the logits' gradient dattn; full tensors, or rows of each."""
    qf, kf, wf = _split(q), _split(k), _split(dattn)
    B, N, heads, _ = qf.shape
    g = Geometry(q.shape[1:-2], kernel, dilation)
    dq = scale * _gather(wf, kf, g, rows, B, N, heads)
    dk = scale * _scatter(wf, qf, g, rows, B, N, heads)
    if rows is None:
        dq, dk = dq.reshape(q.shape), dk.reshape(q.shape)
    return dq, dk


def av_bwd(dO, attn, v, kernel, dilation, rows=None):
    """(dattn, dv) of av given the output's gradient dO; full tensors, or rows of each."""
    gf, vf, af = _split(dO), _split(v), _split(attn)
    B, N, heads, _ = vf.shape
    g = Geometry(v.shape[1:-2], kernel, dilation)
    if rows is None:
        nb = g.neighbours(np.arange(N))
        dattn = np.einsum("bnhc,bnthc->bnht", _f64(gf), _f64(vf[:, nb])).reshape(tuple(v.shape[:-1]) + (g.K,))
    else:
        b, tok, h = _rows_of(rows, B, N, heads)
        nb = g.neighbours(tok)
        dattn = np.einsum("rc,rtc->rt", _f64(gf[b, tok, h]), _f64(vf[b[:, None], nb, h[:, None]]))
    dv = _scatter(af, gf, g, rows, B, N, heads)
    if rows is None:
        dv = dv.reshape(v.shape)
    return dattn, dv


def mask_window(attn, sizes, kernel, dilation):
    """Logits with every offset outside the query's variable window set to -inf.  sizes: one integer
    array per axis, sizes[a][x] = the kernel size (odd, 1..kernel[a]) of queries at position x."""
    out = np.array(attn, dtype=np.float64, copy=True)
    B = out.shape[0]
    spatial = tuple(out.shape[1:-2])
    heads, K = out.shape[-2], out.shape[-1]
    g = Geometry(spatial, kernel, dilation)
    keys = g.coords(g.neighbours(np.arange(g.N)).ravel()).reshape(g.N, K, len(spatial))   # [N, K, ndim]
    x = g.coords(np.arange(g.N))                                                          # [N, ndim]
    keep = np.ones((g.N, K), dtype=bool)
    for a, (L, d) in enumerate(zip(spatial, g.dilation)):
        ka = np.asarray(sizes[a], dtype=np.int64)
        first = np.array([first_neighbour(int(i), L, int(ka[i]), d) for i in range(L)])      # own window start
        if (first < 0).any():
            raise ValueError("invalid variable kernel size")
        lo = first[x[:, a]][:, None]
        hi = lo + d * (ka[x[:, a]][:, None] - 1)
        keep &= (keys[:, :, a] >= lo) & (keys[:, :, a] <= hi)
    flat = out.reshape(B, g.N, heads, K)
    flat[np.broadcast_to(~keep[None, :, None, :], flat.shape)] = -np.inf
    return out

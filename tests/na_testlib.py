"""Helpers shared by the GPU parity tests: run the library, run the oracle, compare.

The comparison rule (per output tensor T): max|T_gpu - T_ref| <= tol * max|T_ref|, tol = 2e-2 for
bf16 and 1e-4 for fp32, evaluated in float64 on the host.  fp16 has 3 more mantissa bits than bf16;
its tolerance keeps the bf16 rule's ratio to the unit roundoff (2e-2 is about 5 * 2^-8, and 5 * 2^-11
is about 2.5e-3), rounded up to 5e-3 for the longer fp32 accumulations of the backward.
"""
import numpy as np
import torch

import oracle
from neighborhood_attention_fwd_gb300 import inputs as nain

TOL = {"bf16": 2e-2, "fp16": 5e-3, "fp32": 1e-4}


def run_gpu(w, t, want_bwd=True, split_bwd=False):
    """Forward (+ backward) of workload w on device tensors t = dict(q, k, v, dO)."""
    import neighborhood_attention_fwd_gb300 as na

    q, k, v, dO = t["q"], t["k"], t["v"], t["dO"]
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    na.na_fwd(q, k, v, o, lse, w.kernel, w.dilation, w.scale)
    out = {"o": o, "lse": lse}
    if want_bwd:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
        if split_bwd:
            delta = torch.empty_like(lse)
            na.na_bwd_delta(o, dO, delta)
            na.na_bwd_dq(q, k, v, dO, lse, delta, dq, w.kernel, w.dilation, w.scale)
            na.na_bwd_dkdv(q, k, v, dO, lse, delta, dk, dv, w.kernel, w.dilation, w.scale)
            out["delta"] = delta
        else:
            na.na_bwd(q, k, v, o, dO, lse, dq, dk, dv, w.kernel, w.dilation, w.scale)
        out.update(dq=dq, dk=dk, dv=dv)
    st, raw = na.na_device_status()
    assert st == 0, f"device status {st} raw {raw:#x}"
    return out


def host(t):
    return {k: nain.to_oracle_array(v) for k, v in t.items()}


def compare(name, got, ref, tol, scale_ref=None):
    """max|got - ref| <= tol * max|ref|.  A reference that is identically zero (e.g. dQ and dK when
    every kernel size is 1, where dS = P (dP - Delta) cancels exactly) makes that rule demand
    bit-exact cancellation in fp32; it is then measured against scale_ref (the sibling gradient)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    err = np.abs(got - ref).max() if ref.size else 0.0
    mref = np.abs(ref).max() if ref.size else 0.0
    if mref == 0.0 and scale_ref is not None:
        mref = float(np.abs(np.asarray(scale_ref)).max())
    bound = tol * max(mref, 1e-30)
    assert err <= bound, f"{name}: max abs err {err:.3e} > {bound:.3e} (tol {tol} x max|ref| {np.abs(ref).max():.3e})"
    return err / max(np.abs(ref).max(), 1e-30)


def compare_lse(got, ref, tol):
    """LSE under both rules: the relative one of the other outputs and an absolute bound of tol.
    The backward recomputes P = exp(S - LSE), so an LSE error of e scales a row's P by exp(-e),
    about 1 - e: an absolute bound of tol on LSE is the relative bound tol on P that the rule puts
    on O.  (The relative rule alone allows about 0.1 at LSE values near 5.)"""
    compare("LSE", got, ref, tol)
    err = float(np.abs(np.asarray(got, dtype=np.float64) - np.asarray(ref, dtype=np.float64)).max()) if ref.size else 0.0
    assert err <= tol, f"LSE: max abs err {err:.3e} > {tol} (absolute)"


def to64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def check_full(w, gpu, h, want_bwd=True):
    """Element-by-element comparison of every output against the full oracle."""
    tol = TOL[w.dtype]
    o, lse = oracle.na_fwd(h["q"], h["k"], h["v"], w.kernel, w.dilation, w.scale)
    rel = {"o": compare("O", to64(gpu["o"]), o, tol)}
    compare_lse(to64(gpu["lse"]), lse, tol)
    if want_bwd:
        dq, dk, dv = oracle.na_bwd(h["q"], h["k"], h["v"], h["dO"], w.kernel, w.dilation, w.scale)
        rel["dq"] = compare("dQ", to64(gpu["dq"]), dq, tol, scale_ref=dv)
        rel["dk"] = compare("dK", to64(gpu["dk"]), dk, tol, scale_ref=dv)
        rel["dv"] = compare("dV", to64(gpu["dv"]), dv, tol)
    return rel


def sample_rows(w, n, seed=0):
    """Row indices ((b*N + token)*heads + head): random rows plus every corner and edge midpoint."""
    rng = np.random.default_rng(seed)
    N = int(np.prod(w.spatial))
    total = w.B * N * w.heads
    rows = set(int(x) for x in rng.integers(0, total, size=n))
    axes = [sorted({0, 1, L // 2, L - 2, L - 1} & set(range(L))) for L in w.spatial]
    import itertools

    for b in {0, w.B - 1}:
        for coord in itertools.product(*axes):
            tok = 0
            for L, x in zip(w.spatial, coord):
                tok = tok * L + x
            for h in {0, w.heads - 1}:
                rows.add((b * N + tok) * w.heads + h)
    return np.array(sorted(rows), dtype=np.int64)


def check_sampled(w, gpu, h, n=256, want_bwd=True, seed=0):
    """Comparison on sampled rows that the oracle computes one by one (full-size workloads)."""
    tol = TOL[w.dtype]
    rows = sample_rows(w, n, seed)
    D = w.D
    idx = torch.as_tensor(rows, device=gpu["o"].device)
    pick = lambda t: to64(t.reshape(-1, D)[idx])          # gather on the device, then copy
    o, lse = oracle.na_fwd(h["q"], h["k"], h["v"], w.kernel, w.dilation, w.scale, rows=rows)
    rel = {"o": compare("O", pick(gpu["o"]), o, tol)}
    compare_lse(to64(gpu["lse"].reshape(-1)[idx]), lse, tol)
    if want_bwd:
        dq, dk, dv = oracle.na_bwd(h["q"], h["k"], h["v"], h["dO"], w.kernel, w.dilation, w.scale,
                                   qrows=rows, krows=rows)
        rel["dq"] = compare("dQ", pick(gpu["dq"]), dq, tol, scale_ref=dv)
        rel["dk"] = compare("dK", pick(gpu["dk"]), dk, tol, scale_ref=dv)
        rel["dv"] = compare("dV", pick(gpu["dv"]), dv, tol)
    for key in ("o", "dq", "dk", "dv"):
        if key in gpu:
            assert torch.isfinite(gpu[key]).all(), f"{key} has non-finite values"
    return rel

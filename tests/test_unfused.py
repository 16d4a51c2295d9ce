"""GPU parity of the unfused operations (logits, window softmax, weighted sum and their gradients)
against the fp64 oracle, through the C ABI.

Each operation is compared on its own, on seeded inputs of its own (the attention-weight inputs are
drawn by the input generator, never taken from another kernel's output), element by element at
small sizes.  The chains qk -> softmax -> av and their gradients are also compared with the fused
oracle's forward and backward, at small sizes in full and at the 2D benchmark shape on sampled rows.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle.unfused as un
from neighborhood_attention_fwd_gb300 import inputs as nain
from na_testlib import TOL, compare, host, sample_rows, to64

pytestmark = pytest.mark.gpu

CASES = [
    # dtype, spatial, heads, D, kernel, dilation, B
    ("fp32", (37,), 2, 16, (7,), (3,), 2),
    ("fp32", (6, 9, 10), 2, 128, (3, 3, 3), (2, 1, 1), 1),
    ("fp32", (16, 16), 2, 16, (5, 5), (1, 1), 1),
    ("bf16", (13, 18), 2, 32, (5, 7), (1, 2), 2),
    ("bf16", (6, 9, 10), 1, 64, (3, 5, 5), (1, 1, 2), 1),
    ("bf16", (20, 24), 3, 128, (9, 9), (1, 1), 1),
    ("bf16", (23, 29), 2, 16, (3, 5), (3, 2), 1),            # classes of unequal length
    ("fp16", (13, 18), 2, 32, (5, 7), (1, 2), 1),
    ("fp16", (5, 7, 9), 2, 16, (5, 7, 9), (1, 1, 1), 1),      # kernel == extent: full attention
    ("fp16", (16, 8), 1, 64, (1, 1), (1, 1), 1),              # k = 1
    # rows of 129-256 weights: the softmax in blocks of 8 rows, and a tail of 5 rows (861 rows)
    ("bf16", (7, 41), 3, 32, (5, 29), (1, 1), 1),
    ("fp16", (6, 8, 30), 2, 16, (3, 5, 11), (1, 1, 2), 1),
]

# Shapes whose weights rows (heads * K offsets) are a multiple of 16 bytes, the innermost kernel size at
# most 17 and D at most 64: the inverse-window gathers (dK of na_qk_bwd, dV of na_av_bwd) take their
# TMA-fed form, with source rows swizzled by 32, 64 or 128 bytes (D = 16, 32, 64).
CASES_TMA = [
    ("bf16", (13, 18), 8, 32, (5, 7), (1, 2), 2),
    ("fp16", (6, 9, 10), 8, 64, (3, 5, 5), (1, 1, 2), 1),
    ("bf16", (23, 29), 8, 16, (3, 5), (3, 2), 1),            # classes of unequal length
    ("bf16", (9, 70), 8, 32, (3, 17), (1, 1), 1),            # innermost kernel 17: a 32-query span
    ("fp16", (100,), 8, 16, (13,), (3,), 2),
    ("bf16", (5, 7, 9), 8, 64, (5, 7, 9), (1, 1, 1), 1),      # kernel == extent: full attention
    # several tensor-core logits strips (129 - k2 class positions each) along the innermost axis
    ("bf16", (4, 300), 8, 32, (3, 9), (1, 1), 1),
    ("fp16", (3, 261), 8, 16, (3, 7), (1, 2), 1),
]


def _ids(c):
    return f"{c[0]}-{'x'.join(map(str, c[1]))}-h{c[2]}-D{c[3]}-k{'x'.join(map(str, c[4]))}-d{'x'.join(map(str, c[5]))}-B{c[6]}"


def f32(t):
    """Host float32 copy (exact for fp32, bf16 and fp16 values) in the form the unfused oracle reads."""
    return t.detach().to("cpu", torch.float32).numpy()


def setup(case, seed=17):
    dtype, spatial, heads, D, kernel, dilation, B = case
    w = nain.small_workload(dtype, spatial, heads, D, kernel, dilation, B=B, seed=seed)
    t = nain.make_inputs(w, device="cpu")
    wt = {"logits": nain.make_weights(w, "randn", seed=seed + 1),
          "probs": nain.make_weights(w, "uniform", seed=seed + 2),
          "grad": nain.make_weights(w, "randn", seed=seed + 3)}
    return w, t, wt


def status_ok(na):
    st, raw = na.na_device_status()
    assert st == 0, f"device status {st} raw {raw:#x}"


@pytest.mark.parametrize("case", CASES + CASES_TMA, ids=[_ids(c) for c in CASES + CASES_TMA])
def test_each_operation_matches_the_oracle(case, cuda_lib):
    na = cuda_lib
    w, t, wt = setup(case)
    tol = TOL[w.dtype]
    dev = {k: v.cuda() for k, v in t.items()}
    wd = {k: v.cuda() for k, v in wt.items()}
    h = {k: f32(v) for k, v in t.items()}
    hw = {k: f32(v) for k, v in wt.items()}
    kern, dil, scale = w.kernel, w.dilation, w.scale

    attn = torch.empty_like(wd["logits"])
    na.na_qk(dev["q"], dev["k"], attn, kern, dil, scale)
    o = torch.empty_like(dev["q"])
    na.na_av(wd["probs"], dev["v"], o, kern, dil)
    y = torch.empty_like(wd["logits"])
    na.na_softmax(wd["logits"], y, kern)
    dx = torch.empty_like(wd["logits"])
    na.na_softmax_bwd(wd["probs"], wd["grad"], dx, kern)
    dq, dk = torch.empty_like(dev["q"]), torch.empty_like(dev["q"])
    na.na_qk_bwd(wd["grad"], dev["q"], dev["k"], dq, dk, kern, dil, scale)
    dattn, dv = torch.empty_like(wd["logits"]), torch.empty_like(dev["q"])
    na.na_av_bwd(dev["dO"], wd["probs"], dev["v"], dattn, dv, kern, dil)
    status_ok(na)

    compare("attn", to64(attn), un.qk(h["q"], h["k"], kern, dil, scale), tol)
    compare("o", to64(o), un.av(hw["probs"], h["v"], kern, dil), tol)
    compare("softmax", to64(y), un.softmax(hw["logits"]), tol)
    compare("softmax_bwd", to64(dx), un.softmax_bwd(hw["probs"], hw["grad"]), tol)
    rq, rk = un.qk_bwd(hw["grad"], h["q"], h["k"], kern, dil, scale)
    compare("dq", to64(dq), rq, tol)
    compare("dk", to64(dk), rk, tol)
    ra, rv = un.av_bwd(h["dO"], hw["probs"], h["v"], kern, dil)
    compare("dattn", to64(dattn), ra, tol)
    compare("dv", to64(dv), rv, tol)


def run_chain(na, w, dev):
    """qk -> softmax -> av, then the chained gradients, all on the device."""
    kern, dil, scale = w.kernel, w.dilation, w.scale
    q, k, v, dO = dev["q"], dev["k"], dev["v"], dev["dO"]
    K = w.keys_per_query
    attn = torch.empty(q.shape[:-1] + (K,), dtype=q.dtype, device=q.device)
    na.na_qk(q, k, attn, kern, dil, scale)
    na.na_softmax(attn, attn, kern)                          # in place
    o = torch.empty_like(q)
    na.na_av(attn, v, o, kern, dil)
    dattn, dv = torch.empty_like(attn), torch.empty_like(v)
    na.na_av_bwd(dO, attn, v, dattn, dv, kern, dil)
    na.na_softmax_bwd(attn, dattn, dattn, kern)              # in place over the incoming gradient
    dq, dk = torch.empty_like(q), torch.empty_like(k)
    na.na_qk_bwd(dattn, q, k, dq, dk, kern, dil, scale)
    status_ok(na)
    return {"o": o, "dq": dq, "dk": dk, "dv": dv}


@pytest.mark.parametrize("case", CASES, ids=[_ids(c) for c in CASES])
def test_chain_matches_the_fused_oracle(case, cuda_lib):
    w, t, _ = setup(case, seed=29)
    tol = TOL[w.dtype]
    got = run_chain(cuda_lib, w, {k: v.cuda() for k, v in t.items()})
    hh = host(t)
    o, _ = oracle.na_fwd(hh["q"], hh["k"], hh["v"], w.kernel, w.dilation, w.scale)
    dq, dk, dv = oracle.na_bwd(hh["q"], hh["k"], hh["v"], hh["dO"], w.kernel, w.dilation, w.scale)
    compare("O", to64(got["o"]), o, tol)
    compare("dQ", to64(got["dq"]), dq, tol, scale_ref=dv)
    compare("dK", to64(got["dk"]), dk, tol, scale_ref=dv)
    compare("dV", to64(got["dv"]), dv, tol)


def test_operations_are_deterministic(cuda_lib):
    na = cuda_lib
    w, t, _ = setup(("bf16", (30, 26), 2, 32, (7, 5), (1, 2), 1), seed=3)
    dev = {k: v.cuda() for k, v in t.items()}
    a = run_chain(na, w, dev)
    b = run_chain(na, w, dev)
    for key in a:
        assert torch.equal(a[key], b[key]), key


@pytest.mark.slow
def test_full_size_chain_sampled(cuda_lib):
    """The 2D benchmark shape (1024x1024, 8 heads of dim 32, 9x9, bf16): each operation on sampled rows
    against the unfused oracle, and the chain's outputs against the fused oracle."""
    na = cuda_lib
    w = nain.WORKLOADS["2d_bf16_1024x1024_k9"]
    t = nain.make_inputs(w, device="cuda")
    tol = TOL[w.dtype]
    got = run_chain(na, w, t)
    rows = sample_rows(w, 96, seed=5)
    idx = torch.as_tensor(rows, device="cuda")
    pick = lambda x: to64(x.reshape(-1, x.shape[-1])[idx])
    hh = host({k: v for k, v in t.items()})
    o, _ = oracle.na_fwd(hh["q"], hh["k"], hh["v"], w.kernel, w.dilation, w.scale, rows=rows)
    dq, dk, dv = oracle.na_bwd(hh["q"], hh["k"], hh["v"], hh["dO"], w.kernel, w.dilation, w.scale,
                               qrows=rows, krows=rows)
    compare("O", pick(got["o"]), o, tol)
    compare("dQ", pick(got["dq"]), dq, tol, scale_ref=dv)
    compare("dK", pick(got["dk"]), dk, tol, scale_ref=dv)
    compare("dV", pick(got["dv"]), dv, tol)
    for key, x in got.items():
        assert torch.isfinite(x).all(), key

    # each operation on its own, on seeded weights of the full shape
    h = {k: f32(v) for k, v in t.items()}
    probs = nain.make_weights(w, "uniform", device="cuda", seed=77)
    grad = nain.make_weights(w, "randn", device="cuda", seed=78)
    hp, hg = f32(probs), f32(grad)
    kern, dil, scale = w.kernel, w.dilation, w.scale
    attn = torch.empty_like(grad)
    rpb = nain.make_rpb(w, device="cuda", seed=79)
    na.na_qk(t["q"], t["k"], attn, kern, dil, scale, rpb=rpb)
    o2 = torch.empty_like(t["q"])
    na.na_av(probs, t["v"], o2, kern, dil)
    y = torch.empty_like(grad)
    na.na_softmax(grad, y, kern)
    dx = torch.empty_like(grad)
    na.na_softmax_bwd(probs, grad, dx, kern)
    dq2, dk2 = torch.empty_like(t["q"]), torch.empty_like(t["q"])
    na.na_qk_bwd(grad, t["q"], t["k"], dq2, dk2, kern, dil, scale)
    dattn, dv2 = torch.empty_like(grad), torch.empty_like(t["q"])
    na.na_av_bwd(t["dO"], probs, t["v"], dattn, dv2, kern, dil)
    status_ok(na)
    compare("attn", pick(attn), un.qk(h["q"], h["k"], kern, dil, scale, rows, rpb=f32(rpb)), tol)
    compare("o", pick(o2), un.av(hp, h["v"], kern, dil, rows), tol)
    compare("softmax", pick(y), un.softmax(hg, rows), tol)
    compare("softmax_bwd", pick(dx), un.softmax_bwd(hp, hg, rows), tol)
    rq, rk = un.qk_bwd(hg, h["q"], h["k"], kern, dil, scale, rows)
    compare("dq", pick(dq2), rq, tol)
    compare("dk", pick(dk2), rk, tol)
    ra, rv = un.av_bwd(h["dO"], hp, h["v"], kern, dil, rows)
    compare("dattn", pick(dattn), ra, tol)
    compare("dv", pick(dv2), rv, tol)


# ---------------------------------------------------------------------------------------------
# Relative positional bias
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("case", CASES, ids=[_ids(c) for c in CASES])
def test_rpb_logits_and_gradient_match_the_oracle(case, cuda_lib):
    na = cuda_lib
    w, t, wt = setup(case, seed=41)
    tol = TOL[w.dtype]
    dev = {k: v.cuda() for k, v in t.items()}
    rpb = nain.make_rpb(w, seed=42)
    attn = torch.empty_like(wt["logits"]).cuda()
    na.na_qk(dev["q"], dev["k"], attn, w.kernel, w.dilation, w.scale, rpb=rpb.cuda())
    drpb = torch.empty_like(rpb).cuda()
    na.na_rpb_grad(wt["grad"].cuda(), drpb, w.kernel, w.dilation)
    status_ok(na)
    h = {k: f32(v) for k, v in t.items()}
    compare("attn+rpb", to64(attn), un.qk(h["q"], h["k"], w.kernel, w.dilation, w.scale, rpb=f32(rpb)), tol)
    compare("drpb", to64(drpb), un.rpb_grad(f32(wt["grad"]), w.kernel, w.dilation), TOL["fp32"])


def test_rpb_grad_is_deterministic_and_takes_a_workspace(cuda_lib):
    na = cuda_lib
    w = nain.small_workload("bf16", (40, 37), 3, 32, (5, 7), (1, 2), B=2, seed=5)
    g = nain.make_weights(w, "randn", device="cuda", seed=6)
    a = torch.empty((3, 9, 13), dtype=torch.float32, device="cuda")
    b = torch.empty_like(a)
    na.na_rpb_grad(g, a, w.kernel, w.dilation)
    nbytes = na.na_rpb_grad_workspace_size(w.B, w.spatial, w.heads, w.kernel)
    ws = torch.empty(nbytes // 4, dtype=torch.float32, device="cuda")
    na.na_rpb_grad(g, b, w.kernel, w.dilation, workspace=ws)
    status_ok(na)
    assert torch.equal(a, b)


@pytest.mark.slow
def test_rpb_grad_full_size(cuda_lib):
    """The bias gradient over every query of the 512x512 shape (2M rows, 9x9) against the oracle."""
    na = cuda_lib
    w = nain.WORKLOADS["2d_bf16_512x512_k9"]
    g = nain.make_weights(w, "randn", device="cuda", seed=8)
    drpb = torch.empty((w.heads, 17, 17), dtype=torch.float32, device="cuda")
    na.na_rpb_grad(g, drpb, w.kernel, w.dilation)
    status_ok(na)
    compare("drpb", to64(drpb), un.rpb_grad(f32(g), w.kernel, w.dilation), TOL["fp32"])


# ---------------------------------------------------------------------------------------------
# Variable windows
# ---------------------------------------------------------------------------------------------

VARWIN = [
    # dtype, spatial, heads, D, kernel, dilation, B, sizes per axis (None: the full kernel)
    ("fp32", (11,), 2, 16, (5,), (1,), 2, [[1, 1, 3, 3, 5, 5, 5, 3, 3, 1, 1]]),
    ("bf16", (9, 10), 2, 32, (3, 5), (2, 1), 1, [[1, 3, 1, 3, 3, 1, 3, 1, 3], None]),
    ("fp16", (6, 5, 7), 1, 64, (5, 3, 3), (1, 1, 2), 1, [[1, 1, 3, 3, 5, 5], None, [3, 1, 3, 1, 3, 1, 3]]),
    # kernel sizes that grow along time, the shape the user asks about (8 frames, 5x7x7 windows)
    ("bf16", (8, 24, 20), 2, 32, (5, 7, 7), (1, 1, 1), 1, [[1, 1, 3, 3, 3, 5, 5, 5], None, None]),
]


def _varwin_ids(c):
    return f"{c[0]}-{'x'.join(map(str, c[1]))}-k{'x'.join(map(str, c[4]))}-d{'x'.join(map(str, c[5]))}"


def _full_sizes(spatial, kernel, sizes):
    return [np.full(L, k) if s is None else np.asarray(s) for L, k, s in zip(spatial, kernel, sizes)]


def compare_masked(name, got, ref, tol):
    """The -inf pattern must match exactly; the finite entries follow the tolerance rule."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    ninf_g, ninf_r = np.isneginf(got), np.isneginf(ref)
    assert np.array_equal(ninf_g, ninf_r), f"{name}: masked entries differ ({(ninf_g != ninf_r).sum()})"
    compare(name, got[~ninf_g], ref[~ninf_r], tol)


@pytest.mark.parametrize("case", VARWIN, ids=[_varwin_ids(c) for c in VARWIN])
def test_variable_window_chain_matches_the_oracle(case, cuda_lib):
    na = cuda_lib
    dtype, spatial, heads, D, kernel, dilation, B, sizes = case
    w = nain.small_workload(dtype, spatial, heads, D, kernel, dilation, B=B, seed=51)
    t = nain.make_inputs(w, device="cpu")
    tol = TOL[dtype]
    sz = _full_sizes(spatial, kernel, sizes)
    dev = {k: v.cuda() for k, v in t.items()}
    q, k, v, dO = dev["q"], dev["k"], dev["v"], dev["dO"]
    attn = torch.empty(q.shape[:-1] + (w.keys_per_query,), dtype=q.dtype, device="cuda")
    na.na_qk(q, k, attn, kernel, dilation, w.scale)
    na.na_mask_window(attn, sz, kernel, dilation)
    logits = attn.clone()
    na.na_softmax(attn, attn, kernel)
    o = torch.empty_like(q)
    na.na_av(attn, v, o, kernel, dilation)
    dattn, dv = torch.empty_like(attn), torch.empty_like(v)
    na.na_av_bwd(dO, attn, v, dattn, dv, kernel, dilation)
    na.na_softmax_bwd(attn, dattn, dattn, kernel)
    dq, dk = torch.empty_like(q), torch.empty_like(k)
    na.na_qk_bwd(dattn, q, k, dq, dk, kernel, dilation, w.scale)
    status_ok(na)

    h = {key: f32(val) for key, val in t.items()}
    ref_logits = un.mask_window(un.qk(h["q"], h["k"], kernel, dilation, w.scale), sz, kernel, dilation)
    compare_masked("masked logits", to64(logits), ref_logits, tol)
    y = un.softmax(ref_logits)
    compare("O", to64(o), un.av(y, h["v"], kernel, dilation), tol)
    ry, rv = un.av_bwd(h["dO"], y, h["v"], kernel, dilation)
    rq, rk = un.qk_bwd(un.softmax_bwd(y, ry), h["q"], h["k"], kernel, dilation, w.scale)
    compare("dQ", to64(dq), rq, tol, scale_ref=rv)
    compare("dK", to64(dk), rk, tol, scale_ref=rv)
    compare("dV", to64(dv), rv, tol)


def test_variable_window_mask_on_very_large_windows(cuda_lib):
    """A 1D window of 4999 offsets is beyond the mask kernel's offset table (it decodes per element):
    the mask on seeded logits matches the oracle's exactly, -inf pattern and kept values alike."""
    na = cuda_lib
    L, k = 5001, 4999
    w = nain.small_workload("bf16", (L,), 1, 16, (k,), (1,), B=1, seed=61)
    logits = nain.make_weights(w, "randn", seed=62)
    sizes = [[1 + 2 * ((i * 7) % 2500) for i in range(L)]]           # odd sizes 1..4999, scattered
    attn = logits.cuda()
    na.na_mask_window(attn, sizes, w.kernel, w.dilation)
    status_ok(na)
    ref = un.mask_window(f32(logits), [np.asarray(sizes[0])], w.kernel, w.dilation)
    got = to64(attn)
    assert np.array_equal(np.isneginf(got), np.isneginf(ref))
    keep = ~np.isneginf(ref)
    assert np.array_equal(got[keep], ref[keep])

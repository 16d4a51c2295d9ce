"""Bounded device-side waits: a wait that runs out is reported, and the next launch is clean.

The library's test hook lowers the wait limit of the tensor-core kernels to a few milliseconds and
makes the first CTA skip the copy of its first halo chunk, so the waits on that chunk never
complete (a flag that nothing sets, not a fault).  The kernels must record the wait site in the
status word, stop, let their issued copies land, free their tensor memory and return;
na_device_status then reports NA_ERR_TIMEOUT, and a launch after the hook is cleared must run
normally and match the oracle.
"""
import pytest
import torch

from neighborhood_attention_fwd_gb300 import inputs as nain
from na_testlib import check_full, host, run_gpu

NA_ERR_TIMEOUT = 5
# wait sites that can give up first when a halo chunk never arrives: the chunk itself, the scores
# computed from it (or a free score buffer), the P operand, the producer waiting to refill the slot
SITES = {2, 3, 4, 6}
# a short-tile shape and a long-tile one (its forward plan takes three score buffers)
SHAPES = {"short": ((40, 37), (5, 7), (1, 1)), "long": ((8, 20, 20), (5, 7, 7), (1, 1, 1))}


@pytest.mark.gpu
@pytest.mark.parametrize("phase", ["fwd", "bwd"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("shape", sorted(SHAPES))
def test_a_wait_that_runs_out_is_reported_and_the_next_launch_is_clean(cuda_lib, phase, dtype, shape):
    import neighborhood_attention_fwd_gb300 as na

    spatial, kernel, dilation = SHAPES[shape]
    w = nain.small_workload(dtype, spatial, 2, 32, kernel, dilation, B=1, seed=31)
    t = {k: v.cuda() for k, v in nain.make_inputs(w, device="cpu").items()}
    q, k, v, dO = t["q"], t["k"], t["v"], t["dO"]
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    na.na_fwd(q, k, v, o, lse, w.kernel, w.dilation, w.scale)   # the backward reads O and LSE
    assert na.na_device_status()[0] == 0
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    na.na_debug_wait_hook(2_000_000, True)
    try:
        if phase == "fwd":
            na.na_fwd(q, k, v, torch.empty_like(q), torch.empty_like(lse), w.kernel, w.dilation, w.scale)
        else:
            na.na_bwd(q, k, v, o, dO, lse, dq, dk, dv, w.kernel, w.dilation, w.scale)
        st, raw = na.na_device_status()
    finally:
        na.na_debug_wait_hook(0, False)
    assert st == NA_ERR_TIMEOUT, (st, hex(raw))
    assert raw & 0xF000 == 0x5000 and (raw & 0xFFF) in SITES, hex(raw)
    # the status word was cleared by the read, and the next launches run normally and correctly
    gpu = run_gpu(w, t)
    check_full(w, gpu, host(t))


def test_wait_hook_rejects_bad_arguments():
    import neighborhood_attention_fwd_gb300 as na
    from neighborhood_attention_fwd_gb300 import build as nabuild

    nabuild.build()
    lib = na.load()
    assert lib.na_debug_wait_hook(10, 0) == 1            # below 100 us
    assert lib.na_debug_wait_hook(20_000_000_000, 0) == 1  # above 10 s
    assert lib.na_debug_wait_hook(0, 2) == 1
    assert lib.na_debug_wait_hook(0, 0) == 0

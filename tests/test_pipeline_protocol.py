"""A CPU model of the tensor-core kernels' chunk handoff between softmax warps and the MMA issuers.

The kernels hand each chunk's P operand (dK/dV: P^T and dS^T) from the softmax warps to the issuers of the
update products through mbarriers with phase parity: an arrival counts toward whatever phase is current,
not toward the chunk the arriving warp means.  This model replays that protocol with random delays and
checks that an update product never starts before every warp has finished writing its chunk.  It pins the
dK/dV rule that a warp with nothing to write still waits for the products of chunk g - 2 before it
arrives: without the wait (the `shortcut` variant) an idle warp runs ahead and completes chunk g's phase
early, as seen on the GPU.  It also covers the forward, whose P is written over its scores in TMEM and
whose score and P V products come from two independent issuing lanes: a softmax warp that rescales the
output accumulator in TMEM must find the P V product of the chunk before already done.
"""
import random

import pytest


class Bar:
    """An mbarrier: `count` arrivals complete the current phase; a wait on parity p passes once the
    phase with that parity has completed (the parity of the number of completed phases differs from p)."""

    def __init__(self, count):
        self.count, self.pending, self.n = count, count, 0

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.n += 1
            self.pending = self.count

    def passed(self, parity):
        return (self.n & 1) != parity


def run_model(variant, chunks, idle, rng, n_warps=8, n_issuers=2, n_p=2, rescale_wait=True):
    """variant: 'backward' (the dK/dV protocol), 'shortcut' (idle warps arrive without the wait), or
    'forward' (P over the scores: the next score product waits for the P V product).  Returns the list
    of violations: an update of chunk g that started before a warp finished writing chunk g, or (forward)
    a rescale of the output accumulator while the P V product of the chunk before was still running."""
    if variant == "forward":
        n_issuers = 1  # one lane issues the forward's P V products, another its score products
    s_full = [Bar(1) for _ in range(2)]
    s_empty = [Bar(n_warps) for _ in range(2)]
    p_full = [Bar(n_warps) for _ in range(n_p)]
    p_empty = [Bar(n_issuers) for _ in range(n_p)]
    written = [-1] * n_warps  # last chunk each warp finished writing
    pv_done = [False] * chunks  # the update product of each chunk has completed
    violations = []

    def delay(lo, hi):
        return ("delay", rng.randint(lo, hi))

    def score_lane():
        for g in range(chunks):
            sb = g & 1
            if g >= 2:
                if variant == "forward":  # the buffer also holds P(g - 2): wait for its P V product
                    yield ("wait", p_empty[(g - 2) % n_p], ((g - 2) // n_p) & 1)
                else:
                    yield ("wait", s_empty[sb], ((g >> 1) - 1) & 1)
            yield delay(1, 6)
            s_full[sb].arrive()

    def softmax(w):
        for g in range(chunks):
            sb, pb = g & 1, g % n_p
            yield ("wait", s_full[sb], (g >> 1) & 1)
            yield delay(0, 2)  # read the run's scores
            if variant == "forward" and g >= 1 and rng.random() < 0.3:
                # the running max moved: rescale O, which the P V products of chunks g - 1, g - 2, ...
                # accumulate into, after the last of them is done
                if rescale_wait:
                    yield ("wait", p_empty[(g - 1) % n_p], ((g - 1) // n_p) & 1)
                if not pv_done[g - 1]:
                    violations.append(("rescale", g, w))
                yield delay(0, 2)
            if variant != "forward":
                s_empty[sb].arrive()  # released as soon as they are read
            if w in idle and variant != "forward":  # the forward zeroes an idle warp's P rows: a write
                if variant == "backward" and g >= n_p:
                    yield ("wait", p_empty[pb], ((g // n_p) - 1) & 1)
                p_full[pb].arrive()
                continue
            if variant != "forward" and g >= n_p:
                yield ("wait", p_empty[pb], ((g // n_p) - 1) & 1)
            yield delay(2, 12)  # compute and write P
            written[w] = g
            p_full[pb].arrive()

    def issuer(u):
        for g in range(chunks):
            pb = g % n_p
            yield ("wait", p_full[pb], (g // n_p) & 1)
            for w in range(n_warps):
                if w not in idle and written[w] < g:
                    violations.append((u, g, w))
            yield delay(1, 5)
            pv_done[g] = True
            p_empty[pb].arrive()

    agents = [score_lane()] + [softmax(w) for w in range(n_warps)]
    agents += [issuer(u) for u in range(n_issuers)]
    state = [None] * len(agents)  # current op of each agent
    live = set(range(len(agents)))
    stall = 0
    while live:
        progress = False
        order = list(live)
        rng.shuffle(order)
        for i in order:
            op = state[i]
            if op is not None and op[0] == "delay" and op[1] > 0:
                state[i] = ("delay", op[1] - 1)
                progress = True
                continue
            if op is not None and op[0] == "wait" and not op[1].passed(op[2]):
                continue
            try:
                state[i] = next(agents[i])
            except StopIteration:
                live.discard(i)
            progress = True
        stall = 0 if progress else stall + 1
        assert stall < 1000, f"{variant}: the protocol deadlocked"
    return violations


@pytest.mark.parametrize("variant", ["backward", "forward"])
def test_updates_never_start_before_the_operand_is_written(variant):
    rng = random.Random(7)
    for trial in range(300):
        idle = set(rng.sample(range(8), rng.randint(0, 6)))
        assert run_model(variant, 12, idle, rng) == [], (variant, trial, idle)


def test_the_shortcut_without_the_wait_lets_an_idle_warp_run_ahead():
    """The removed shortcut: idle warps arrive on P-full without waiting for chunk g - 2's products."""
    rng = random.Random(7)
    bad = 0
    for _ in range(300):
        idle = set(rng.sample(range(8), rng.randint(1, 6)))
        bad += bool(run_model("shortcut", 12, idle, rng))
    assert bad > 0


def test_three_p_buffers_keep_the_shortcut_safe():
    """dQ (three P buffers, two score buffers, one update issuer): an idle warp at chunk g + 3 needs the
    scores of g + 3, whose buffer was released by every warp's read of chunk g + 1, so every warp has
    already arrived for chunk g."""
    rng = random.Random(11)
    for _ in range(300):
        idle = set(rng.sample(range(8), rng.randint(1, 6)))
        assert run_model("shortcut", 12, idle, rng, n_issuers=1, n_p=3) == []


def test_a_rescale_without_the_wait_races_the_previous_update():
    """The forward's rescale of O without waiting for chunk g - 1's P V product: with the P V lane
    independent of the softmax warps, that product can still be running."""
    rng = random.Random(5)
    bad = 0
    for _ in range(300):
        idle = set(rng.sample(range(8), rng.randint(0, 6)))
        bad += any(v[0] == "rescale" for v in run_model("forward", 12, idle, rng, rescale_wait=False))
    assert bad > 0

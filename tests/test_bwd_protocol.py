"""Model check of the backward kernel's barrier protocol (race detection).

The gradient kernel (csrc/attn_bwd_kernel.cuh) runs, per CTA, one 128-key tile
against its query blocks with eight roles that synchronise only through
mbarriers: the TMA producer (K_j, V_j once, then a ring of Q_i + dO_i stages
with their row statistics), the MMA-issuing warp (S^T and dP^T two blocks
ahead, then dV, dK and dQ^T of the current block), two P/dS warpgroups, and four
dQ readout warps, the first of which also issues the TMA reduce of each staged
half of dQ_i and releases a half once the reduce issued after it has read its
data.

An mbarrier wait names its phase by parity alone, so the protocol must never
let a barrier run two phases ahead of a waiter, and it must never deadlock.
This test replays every wait and arrival of the eight roles, with the kernel's
arrival counts and ring depths, under many random interleavings, for blocks
counts from 1 to 13 and both ring depths (3 stages at d = 128, 4 at d = 64).
Asynchronous completions (TMA loads, MMA commits, the reduce's read of a half)
happen at once in the model, the most permissive timing.  Negative controls
plant two protocol mistakes the check must catch: an issuer that never
releases the second staging half, and a P barrier that expects one arrival more
than the P/dS warps make.

Like the kernel's own documentation, the model states the protocol; when the
kernel's waits or arrivals change, this model changes with it.
"""
import random

import pytest


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.done = name, count, count, 0

    def arrive(self, n=1):
        self.pending -= n
        assert self.pending >= 0, f"{self.name}: more arrivals than the count"
        if self.pending == 0:
            self.done += 1
            self.pending = self.count


def run(n_iter, stages, seed, release_second_half=True, pfull_count=8):
    rng = random.Random(seed)
    B = {}

    def mk(name, count=1):
        B[name] = Barrier(name, count)

    mk("KvFull")
    mk("KvDone")
    for s in range(stages):
        mk(("QFull", s))
        mk(("QEmpty", s))
    for b in (0, 1):
        mk(("SpFull", b))
        mk(("PFull", b), pfull_count)
        mk(("DsFull", b), 8)
        mk(("DsEmpty", b))
        mk(("DqFull", b))
        mk(("DqFree", b), 4)
    for h in (0, 1):
        mk(("StFull", h), 4)
        mk(("StEmpty", h))

    def wait(name, phase):
        return name, phase

    def producer():
        B["KvFull"].arrive()
        for it in range(n_iter):
            s = it % stages
            if it >= stages:
                yield wait(("QEmpty", s), it // stages - 1)
            B[("QFull", s)].arrive()  # Q_i, dO_i and the statistics

    def mma():
        yield wait("KvFull", 0)

        def issue_sdp(i):
            b = i & 1
            yield wait(("QFull", i % stages), i // stages)
            # S^T of block i into buffer b; dP^T over the columns where dQ^T(i - 2) was
            if i >= 2:
                yield wait(("DqFree", b), (i - 2) >> 1)
            B[("SpFull", b)].arrive()

        yield from issue_sdp(0)
        if n_iter > 1:
            yield from issue_sdp(1)
        for it in range(n_iter):
            b = it & 1
            yield wait(("PFull", b), it >> 1)   # dV += P^T dO_i
            yield wait(("DsFull", b), it >> 1)  # dK += dS^T Q_i, dQ^T = K^T dS^T
            B[("DqFull", b)].arrive()
            B[("DsEmpty", b)].arrive()
            B[("QEmpty", it % stages)].arrive()
            if it == n_iter - 1:
                B["KvDone"].arrive()
            if it + 2 < n_iter:
                yield from issue_sdp(it + 2)

    def pds(wg):
        for it in range(n_iter):
            b = it & 1
            yield wait(("SpFull", b), it >> 1)
            yield wait(("QFull", it % stages), it // stages)
            B[("PFull", b)].arrive(4)  # one arrival per warp of the warpgroup
            if it >= 2:
                yield wait(("DsEmpty", b), (it >> 1) - 1)
            B[("DsFull", b)].arrive(4)
        yield wait("KvDone", 0)

    def readout(warp):
        for it in range(n_iter):
            b = it & 1
            yield wait(("DqFull", b), it >> 1)
            B[("DqFree", b)].arrive()
            for h in (0, 1):
                if it >= 1:
                    yield wait(("StEmpty", h), it - 1)
                B[("StFull", h)].arrive()  # lane 0 of this warp, after its stores
                if warp == 8:  # the reduce issuer
                    yield wait(("StFull", h), it)
                    # reduce (it, h) issued; the one before it has read its half
                    if h == 1:
                        B[("StEmpty", 0)].arrive()
                    elif it > 0 and release_second_half:
                        B[("StEmpty", 1)].arrive()
        yield wait("KvDone", 0)

    roles = {"producer": producer(), "mma": mma(), "pds0": pds(0), "pds1": pds(1)}
    for w in (8, 9, 10, 11):
        roles[f"readout{w}"] = readout(w)
    waiting = {k: None for k in roles}
    alive = set(roles)
    while alive:
        runnable = []
        for k in sorted(alive):
            w = waiting[k]
            if w is None:
                runnable.append(k)
                continue
            done = B[w[0]].done
            if done >= w[1] + 2:
                return f"phase overrun: {k} waits {w[0]} phase {w[1]}, barrier already completed {done}"
            if done >= w[1] + 1:
                runnable.append(k)
        if not runnable:
            return f"deadlock: { {k: waiting[k] for k in sorted(alive)} }"
        k = rng.choice(runnable)
        waiting[k] = None
        try:
            waiting[k] = next(roles[k])
        except StopIteration:
            alive.discard(k)
    return None


@pytest.mark.parametrize("stages", [3, 4])
@pytest.mark.parametrize("n_iter", [1, 2, 3, 4, 5, 8, 13])
def test_protocol_has_no_overrun_and_no_deadlock(n_iter, stages):
    for seed in range(40):
        assert run(n_iter, stages, seed) is None


def test_checker_finds_an_issuer_that_never_releases_the_second_half():
    found = [run(4, 3, seed, release_second_half=False) for seed in range(5)]
    assert all(f and f.startswith("deadlock") for f in found)


def test_checker_finds_a_p_barrier_expecting_too_many_arrivals():
    found = [run(3, 3, seed, pfull_count=9) for seed in range(5)]
    assert all(f and f.startswith("deadlock") for f in found)

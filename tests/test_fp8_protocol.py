"""Model check of the FP8 forward kernel's barrier protocol (race detection).

The FP8 kernel (csrc/attn_fwd_fp8_kernel.cuh) has five roles: the TMA producer,
one MMA-issuing warp per query tile and one softmax warpgroup per query tile.
Causal launches with more units than SMs run a dynamic schedule: the producer
publishes each further unit through a two-slot ring (ItemFull, 1 arrival;
ItemEmpty, 10: both MMA warps and the eight softmax warps), which the model
includes.
They synchronise only through mbarriers, and an mbarrier wait names the phase
it waits for by its parity alone.  The waiter of phase k therefore sees phase
k + 2 as phase k.  The protocol must never let a barrier run two phases ahead
of a waiter, and must never deadlock.

This test replays every wait and arrival of the five roles, with the same counts
and the same work items as the kernel, under many random interleavings.  It
checks both properties over causal and non-causal schedules, several units per
CTA, an odd number of query tiles, and the K/V segments [jb, je) of split units
(alone and followed by whole units), where every item loads its own Q tiles and
its first product (jj == jb) starts O after the previous item's O was read out.  Where a role's arrival completes an
asynchronous operation (a TMA load, an MMA commit), the model completes it at
once; that is the most permissive timing for run-ahead.  A negative control
shows the check finds the race of a protocol with one P barrier per tile, which
lets the softmax finish P(k+1) before the MMA warp has waited for P(k).

Like the kernel's own documentation, the model states the protocol; when the
kernel's waits or arrivals change, this model changes with them.
"""
import random

import pytest

STAGES = 8  # the kernel's K/V ring depth


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.done = name, count, count, 0

    def arrive(self, n=1):
        self.pending -= n
        assert self.pending >= 0, f"{self.name}: more arrivals than the count"
        if self.pending == 0:
            self.done += 1
            self.pending = self.count


def unit_tiles(u, nq, BH, causal, heads_per_group):
    """(n0, n1): K/V tiles visited by the unit's two query tiles (the kernel's unit decoding)."""
    pairs = (nq + 1) // 2
    if causal:
        g, r = divmod(u, heads_per_group * pairs)
        heads_here = min(heads_per_group, BH - g * heads_per_group)
        pair = pairs - 1 - r // heads_here
    else:
        pair = u % pairs
    q0 = 2 * pair
    return [min(q0 + t + 1, nq) if causal else nq for t in (0, 1)]


def unit_items(units, nq, BH, causal, G):
    """Whole units as work items (jb, je, n0): tile 0 visits [jb, min(je, n0)), tile 1 [jb, je)."""
    out = []
    for u in units:
        n = unit_tiles(u, nq, BH, causal, G)
        out.append((0, n[1], n[0]))
    return out


def split_items(units, nq, BH, causal, G, nseg):
    """Every unit cut into nseg K/V segments of ceil(n1 / nseg) tiles (the kernel's decode_item)."""
    out = []
    for u in units:
        n = unit_tiles(u, nq, BH, causal, G)
        c = -(-n[1] // nseg)
        for sgi in range(nseg):
            jb = sgi * c
            out.append((jb, min(n[1], jb + c), n[0]))
    return out


def run(items, seed, per_buffer_p=True, dynamic=False):
    """Returns None, or a description of a deadlock or of a phase overrun."""
    rng = random.Random(seed)
    B = {}

    def mk(name, count=1):
        B[name] = Barrier(name, count)

    for s in range(STAGES):
        mk(("KvFull", s))
        mk(("KvEmpty", s), 2)
    for t in (0, 1):
        for n in ("QFull", "QEmpty", "SFull", "ODone", "OFull"):
            mk((n, t))
        mk(("SCons", t), 128)
        mk(("OEmpty", t), 128)
        mk(("ItemFull", t))           # dynamic schedule: the two ring slots
        mk(("ItemEmpty", t), 10)      # both MMA warps and the eight softmax warps
        for b in (0, 1):
            mk(("PFree", t, b))
            mk(("PHalf", t, b), 128)
            mk(("PFull", t, b), 128)

    def pbar(kind, t, k):  # barrier and phase index of P number k
        return ((kind, t, k & 1), k >> 1) if per_buffer_p else ((kind, t, 0), k)

    def wait(name, phase):
        return name, phase

    def take(r):  # reader side of the ring: entry r is the CTA's unit r + 1 (or the end)
        yield wait(("ItemFull", r % 2), r // 2)

    def producer():
        pos = 0
        for ul, (jb, je, _) in enumerate(items):
            for t in (0, 1):
                if ul:
                    yield wait(("QEmpty", t), ul - 1)
                B[("QFull", t)].arrive()
            for _ in range(2 * (je - jb)):  # K_j, V_j for every tile of the item
                st, use = pos % STAGES, pos // STAGES
                if use:
                    yield wait(("KvEmpty", st), use - 1)
                B[("KvFull", st)].arrive()
                pos += 1
            if dynamic:  # publish entry ul
                if ul >= 2:
                    yield wait(("ItemEmpty", ul % 2), ul // 2 - 1)
                B[("ItemFull", ul % 2)].arrive()

    def mma(t):
        s_cnt = p_cnt = kpos = 0
        for ul, (jb, n1, n0) in enumerate(items):
            nt = min(n1, n0) if t == 0 else n1  # this tile's K/V tiles are [jb, nt)
            yield wait(("QFull", t), ul)
            kp, vp = kpos, kpos + 1
            for j in range(jb, n1 + 1):
                if j < n1:
                    yield wait(("KvFull", kp % STAGES), kp // STAGES)
                    if j < nt:
                        if s_cnt:
                            yield wait(("SCons", t), s_cnt - 1)
                        B[("SFull", t)].arrive()
                        if j == nt - 1:
                            B[("QEmpty", t)].arrive()
                        s_cnt += 1
                    B[("KvEmpty", kp % STAGES)].arrive()
                    kp += 2
                if j == jb:
                    continue
                jj = j - 1
                yield wait(("KvFull", vp % STAGES), vp // STAGES)
                if jj < nt:
                    yield wait(*pbar("PHalf", t, p_cnt))
                    if jj == jb and ul:
                        yield wait(("OEmpty", t), ul - 1)
                    yield wait(*pbar("PFull", t, p_cnt))
                    B[("PFree", t, p_cnt & 1)].arrive()
                    B[("ODone", t)].arrive()
                    if jj == nt - 1:
                        B[("OFull", t)].arrive()
                    p_cnt += 1
                B[("KvEmpty", vp % STAGES)].arrive()
                vp += 2
            kpos = kp
            if dynamic:
                yield from take(ul)
                B[("ItemEmpty", ul % 2)].arrive(1)

    def softmax(t):
        s = 0
        for ul, (jb, je, n0) in enumerate(items):
            nt = min(je, n0) if t == 0 else je
            for j in range(jb, nt):
                yield wait(("SFull", t), s)
                if s >= 2:
                    yield wait(("PFree", t, s & 1), (s >> 1) - 1)
                B[("SCons", t)].arrive(128)
                if j > jb and rng.random() < 0.3:  # a row's maximum moved: rescale O
                    yield wait(("ODone", t), s - 1)
                B[pbar("PHalf", t, s)[0]].arrive(128)
                B[pbar("PFull", t, s)[0]].arrive(128)
                s += 1
            yield wait(("OFull", t), ul)
            B[("OEmpty", t)].arrive(128)
            if dynamic:
                yield from take(ul)
                B[("ItemEmpty", ul % 2)].arrive(4)

    roles = {"producer": producer(), "mma0": mma(0), "mma1": mma(1), "softmax0": softmax(0), "softmax1": softmax(1)}
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


CASES = [  # (query tiles per head, batch x heads, causal, grid, heads per group)
    (64, 8, True, 152, 8),
    (64, 8, False, 152, 8),
    (33, 3, True, 10, 3),
    (16, 4, False, 20, 4),
]


@pytest.mark.parametrize("dynamic", [False, True])
@pytest.mark.parametrize("nq,BH,causal,grid,G", CASES)
def test_protocol_has_no_overrun_and_no_deadlock(nq, BH, causal, grid, G, dynamic):
    units = BH * ((nq + 1) // 2)
    for block in range(0, min(grid, units), 5):
        mine = list(range(block, units, grid))[:3]
        for seed in range(12):
            assert run(unit_items(mine, nq, BH, causal, G), seed, dynamic=dynamic) is None


def test_dynamic_schedule_with_a_claimed_unit_order():
    """Units claimed out of stride order (as the counter hands them out), causal."""
    for mine in ([0, 7, 9, 30, 31], [3, 4, 5], [60, 2, 13]):
        for seed in range(20):
            assert run(unit_items(mine, 64, 8, True, 8), seed, dynamic=True) is None


SPLIT_CASES = [  # (query tiles per head, batch x heads, causal, heads per group, segments, the CTA's units)
    (64, 8, True, 8, 2, [0, 1, 2]),       # the heaviest causal units, two segments each
    (64, 8, True, 8, 4, [0, 8]),          # four segments (each still holds a tile of query tile 0)
    (32, 1, False, 1, 3, [13, 14, 15]),   # the last units of a non-causal launch, three segments
    (33, 3, True, 3, 2, [0, 3, 6]),       # odd query-tile count
]


@pytest.mark.parametrize("dynamic", [False, True])
@pytest.mark.parametrize("nq,BH,causal,G,nseg,mine", SPLIT_CASES)
def test_protocol_with_kv_segments(nq, BH, causal, G, nseg, mine, dynamic):
    """The split instantiation: items are K/V segments [jb, je) of units; every item loads
    its own Q tiles, and its first product starts O afresh (jj == jb)."""
    items = split_items(mine, nq, BH, causal, G, nseg)
    for jb, je, n0 in items:  # the split rule: every segment holds a tile of each query tile
        assert jb < min(je, n0)
    # segments, then whole units, as a CTA meets them when only some units are split
    mixed = items + unit_items([mine[-1] + 1], nq, BH, causal, G)
    for seed in range(15):
        assert run(items, seed, dynamic=dynamic) is None
        assert run(mixed, seed, dynamic=dynamic) is None


def test_checker_finds_the_single_p_barrier_race():
    units = list(range(0, 256, 152))
    found = [run(unit_items(units, 64, 8, True, 8), seed, per_buffer_p=False) for seed in range(12)]
    assert any(f and f.startswith("phase overrun") for f in found)

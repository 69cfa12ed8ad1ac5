"""Model check of the bf16 forward kernel's barrier protocol (race detection).

The kernel (csrc/attn_fwd_kernel.cuh) has four roles that synchronise only
through mbarriers: the TMA producer, the MMA-issuing warp and the two softmax
warpgroups.  An mbarrier wait names the phase it waits for by its parity
alone, so the waiter of phase k takes phase k + 2 for phase k: the protocol
must never let a barrier run two phases ahead of a waiter, and it must never
deadlock.

This test replays every wait and arrival of the four roles, with the kernel's
arrival counts, ring depth and issue order, under many random interleavings.
Where an arrival completes an asynchronous operation (a TMA load, an MMA
commit), the model completes it at once, the most permissive timing for
run-ahead.  It covers:
  - whole units and the split segments of the K/V split, for the heaviest units
    and for the last units (tile 0 visiting one K/V tile fewer than tile 1 in
    causal units, several items per CTA);
  - the static schedule and the dynamic one, in which the producer publishes
    each further item through a two-slot ring (ItemFull, 1 arrival; ItemEmpty,
    9 arrivals: the MMA warp and the eight softmax warps).
Negative controls show that the check finds the deadlock of an item ring whose
readers wait for the entry's index instead of its ring phase, and of one whose
ItemEmpty expects more arrivals than the readers make.  The model also shows
that the ItemEmpty wait is a second guarantee: without it the producer still
cannot run two entries ahead of a reader, because loading item r + 2 needs the
Q tiles that the MMA warp releases only after it has waited for the softmax
warps to finish item r.

Like the kernel's own documentation, the model states the protocol; when the
kernel's waits or arrivals change, this model changes with it.
"""
import random

import pytest

STAGES = 5      # K/V ring depth at d = 128 (8 at d = 64)
ITEM_RING = 2


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.done = name, count, count, 0

    def arrive(self, n=1):
        self.pending -= n
        assert self.pending >= 0, f"{self.name}: more arrivals than the count"
        if self.pending == 0:
            self.done += 1
            self.pending = self.count


def unit_tiles(q0, nkv, causal):
    return [min(q0 + t + 1, nkv) if causal else nkv for t in (0, 1)]


def items_of(units, nkv, causal, kv_split, split_units, split_first=0):
    """(jb, je, n0) of every work item, in item order (the kernel's decode_item)."""
    out = []
    for u, q0 in enumerate(units):
        n = unit_tiles(q0, nkv, causal)
        nseg = kv_split if split_first <= u < split_first + split_units else 1
        c = -(-n[1] // nseg)
        for s in range(nseg):
            jb = s * c
            out.append((jb, min(n[1], jb + c), n[0]))
    return out


def run(items, seed, dynamic, stages=STAGES, empty_count=9, producer_waits_empty=True, phase_by_index=False):
    """One CTA processing `items` in order.  None, or a deadlock / phase overrun."""
    rng = random.Random(seed)
    B = {}

    def mk(name, count=1):
        B[name] = Barrier(name, count)

    for s in range(stages):
        mk(("KvFull", s))
        mk(("KvEmpty", s))
    for t in (0, 1):
        for n in ("QFull", "QEmpty", "SFull", "OFull"):
            mk((n, t))
        mk(("PHalf", t), 128)
        mk(("PFull", t), 128)
        mk(("OEmpty", t), 128)
    for s in range(ITEM_RING):
        mk(("ItemFull", s))
        mk(("ItemEmpty", s), empty_count)

    def wait(name, phase):
        return name, phase

    def take(r):
        # consumer side of the ring: entry r is item r + 1 (None after the last)
        s = r % ITEM_RING
        yield wait(("ItemFull", s), r if phase_by_index else r // ITEM_RING)

    def producer():
        pos = 0
        for ul, (jb, je, _) in enumerate(items):
            for t in (0, 1):
                if ul:
                    yield wait(("QEmpty", t), ul - 1)
                B[("QFull", t)].arrive()
            for _ in range(2 * (je - jb)):  # K_j, V_j
                st, use = pos % stages, pos // stages
                if use:
                    yield wait(("KvEmpty", st), use - 1)
                B[("KvFull", st)].arrive()
                pos += 1
            if dynamic:  # publish entry ul (the next item, or the end)
                s = ul % ITEM_RING
                if ul >= ITEM_RING and producer_waits_empty:
                    yield wait(("ItemEmpty", s), ul // ITEM_RING - 1)
                B[("ItemFull", s)].arrive()

    def mma():
        kpos = 0
        pph = [0, 0]
        for ul, (jb, e1, n0) in enumerate(items):
            e0 = min(e1, n0)
            yield wait(("QFull", 0), ul)
            yield wait(("QFull", 1), ul)

            def pv(t, j, vp):
                if t == 0 or j >= e0:  # first use of V_j
                    yield wait(("KvFull", vp % stages), vp // stages)
                yield wait(("PHalf", t), pph[t])
                if j == jb and ul:
                    yield wait(("OEmpty", t), ul - 1)
                yield wait(("PFull", t), pph[t])
                pph[t] += 1
                if t == 1:
                    B[("KvEmpty", vp % stages)].arrive()  # V_j's last reader
                if j == (e0 if t == 0 else e1) - 1:
                    B[("OFull", t)].arrive()

            vpos = kpos + 1
            vprev = vpos
            for j in range(jb, e1):
                yield wait(("KvFull", kpos % stages), kpos // stages)
                if j < e0:
                    B[("SFull", 0)].arrive()
                    if j == e0 - 1:
                        B[("QEmpty", 0)].arrive()
                if j > jb:
                    yield from pv(1, j - 1, vprev)
                B[("SFull", 1)].arrive()
                B[("KvEmpty", kpos % stages)].arrive()  # K_j's last reader
                if j == e1 - 1:
                    B[("QEmpty", 1)].arrive()
                if j < e0:
                    yield from pv(0, j, vpos)
                vprev = vpos
                kpos += 2
                vpos += 2
            yield from pv(1, e1 - 1, vprev)
            if dynamic:
                yield from take(ul)
                B[("ItemEmpty", ul % ITEM_RING)].arrive(1)

    def softmax(t):
        s_cnt = 0
        for ul, (jb, je, n0) in enumerate(items):
            et = min(je, n0) if t == 0 else je
            for _ in range(jb, et):
                yield wait(("SFull", t), s_cnt)
                s_cnt += 1
                B[("PHalf", t)].arrive(128)  # the O rescale needs no wait: its PV completed before S_t
                B[("PFull", t)].arrive(128)
            yield wait(("OFull", t), ul)
            B[("OEmpty", t)].arrive(128)
            if dynamic:
                yield from take(ul)
                B[("ItemEmpty", ul % ITEM_RING)].arrive(4)  # lane 0 of each of the 4 warps

    roles = {"producer": producer(), "mma": mma(), "softmax0": softmax(0), "softmax1": softmax(1)}
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


def cta_items(nq, causal, kv_split, split_units, pick, split_first=0):
    """The items of one CTA: `pick` selects which item indices it takes, in order."""
    pairs = (nq + 1) // 2
    units = [2 * (pairs - 1 - r) if causal else 2 * r for r in range(pairs)]  # heaviest first when causal
    allitems = items_of(units, nq, causal, kv_split, split_units, split_first)
    return [allitems[i] for i in pick(len(allitems)) if i < len(allitems)]


CASES = [  # (query tiles, causal, kv_split, split units, CTA's item picks)
    (16, False, 1, 0, lambda n: range(0, n, 3)),                   # static stride, whole units
    (33, True, 1, 0, lambda n: range(1, n, 4)),                    # causal, odd tile count
    (32, True, 2, 6, lambda n: range(0, n, 5)),                    # split heaviest units into 2
    (30, True, 4, 3, lambda n: list(range(0, 12, 3)) + [13]),      # split into 4, then whole units
    (24, False, 3, 4, lambda n: range(2, n, 7)),                   # non-causal split into 3
    (40, True, 1, 0, lambda n: [0, 5, 6, 11, 12, 19]),             # a dynamic claim order
    (3, True, 1, 0, lambda n: range(n)),                           # one K/V tile per item at the end
]
TAIL_CASES = [  # the last units split (a partial last wave spread over all SMs)
    (40, False, 4, 5, lambda n: range(0, n, 3), 15),
    (33, False, 3, 2, lambda n: [0, 4] + list(range(15, n)), 15),
]


@pytest.mark.parametrize("dynamic", [False, True])
@pytest.mark.parametrize("nq,causal,kv_split,split_units,pick", CASES)
def test_protocol_has_no_overrun_and_no_deadlock(nq, causal, kv_split, split_units, pick, dynamic):
    items = cta_items(nq, causal, kv_split, split_units, pick)
    assert items
    for seed in range(25):
        assert run(items, seed, dynamic) is None
        assert run(items, seed, dynamic, stages=8) is None


@pytest.mark.parametrize("dynamic", [False, True])
@pytest.mark.parametrize("nq,causal,kv_split,split_units,pick,first", TAIL_CASES)
def test_protocol_with_the_last_units_split(nq, causal, kv_split, split_units, pick, first, dynamic):
    items = cta_items(nq, causal, kv_split, split_units, pick, first)
    assert items
    for seed in range(25):
        assert run(items, seed, dynamic) is None


def test_item_ring_cannot_run_ahead_even_without_its_empty_wait():
    """The Q and O barriers alone keep the producer within one entry of every reader."""
    for nq, causal, kv_split, split_units, pick in CASES:
        items = cta_items(nq, causal, kv_split, split_units, pick)
        for seed in range(15):
            assert run(items, seed, True, producer_waits_empty=False) is None


def test_checker_finds_readers_waiting_the_wrong_phase():
    """Readers that wait for phase r (the entry index) instead of r // 2 deadlock."""
    items = cta_items(16, True, 1, 0, lambda n: range(n))
    found = [run(items, seed, True, phase_by_index=True) for seed in range(5)]
    assert all(f and f.startswith("deadlock") for f in found)


def test_checker_finds_a_ring_that_expects_too_many_readers():
    """An ItemEmpty count above the 9 readers never completes: the producer deadlocks."""
    items = cta_items(16, True, 1, 0, lambda n: range(n))
    found = [run(items, seed, True, empty_count=10) for seed in range(5)]
    assert all(f and f.startswith("deadlock") for f in found)

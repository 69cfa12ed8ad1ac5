"""Host logic of the work split (attn_fwd_split_choice; no GPU needed).

attn_fwd_split picks, per launch, one of these schedules:
  - fewer units than SMs: the heaviest units are cut into segments of K/V tiles,
    either on the SMs the units leave idle (one wave, static), or, for causal
    launches, as many as pays under the dynamic schedule (CTAs claim the items,
    heaviest first);
  - more equal (non-causal) units than SMs: the units of the last, partial wave
    are cut into segments that spread over all SMs;
  - more causal units than SMs: no split, the dynamic schedule.
The segment that finishes a row last merges the row's segments in the kernel.
These tests pin the choices for the benchmark workloads, and check over a
sweep of shapes and SM counts that every choice is one the kernel can run: each
segment of each split unit holds at least one K/V tile of both query tiles
(the kernel's own segment arithmetic), a static split of an under-filled launch
stays one wave, and a split takes the dynamic schedule only for a causal launch
with fewer units than SMs.
"""
import ctypes

import pytest

import exact_long_sequence_gb300 as ela


@pytest.fixture(scope="module")
def lib():
    return ela.load_library()


def choice(lib, B, H, N, d, causal, sms=152):
    v = [ctypes.c_int() for _ in range(4)]
    st = lib.attn_fwd_split_choice(B, H, N, d, int(causal), sms, *[ctypes.byref(x) for x in v])
    assert st == ela.ATTN_OK
    return tuple(x.value for x in v)  # segs, first, units, dynamic


def plan(lib, B, H, N, d, causal, sms):
    p = ela.AttnPlan()
    assert lib.attn_plan(B, H, N, d, int(causal), sms, ctypes.byref(p)) == ela.ATTN_OK
    return p


def unit_tiles(u, BH, N, causal, G):
    """K/V tiles of the unit's two query tiles, in the kernel's unit order (decode_unit)."""
    nq = -(-N // 128)
    pairs = (nq + 1) // 2
    if causal:
        g, r = divmod(u, G * pairs)
        heads_here = min(G, BH - g * G)
        pair = pairs - 1 - r // heads_here
    else:
        pair = u % pairs
    q0 = 2 * pair
    return [min(q0 + t + 1, nq) if causal else nq for t in (0, 1)]


# (B, H, N, d, causal) -> (segments, first split unit, split units, dynamic) on 152 SMs
PINNED = {
    (1, 1, 256, 64, False): (1, 0, 0, 0),        # C1: one unit of two K/V tiles
    (1, 8, 4096, 64, True): (2, 0, 120, 1),      # C2: 120 of 128 units halved, 248 items claimed dynamically
                                                 # (45.9 -> 42.6 us against the static one-wave split)
    (1, 16, 16384, 128, False): (4, 912, 112, 0),  # C3: the last partial wave (1024 = 6 * 152 + 112)
    (1, 8, 65536, 128, True): (1, 0, 0, 1),      # C4: dynamic schedule
    (4, 32, 8192, 128, True): (1, 0, 0, 1),      # C5: dynamic schedule
    (1, 10, 4096, 128, False): (4, 152, 8, 0),   # 160 units: the 8 of the second wave
    (1, 2, 8192, 128, False): (2, 0, 64, 0),     # 64 equal units, all split in two
    (1, 19, 2048, 64, False): (1, 0, 0, 0),      # 152 units fill the SMs exactly
    (1, 8, 4096, 64, False): (1, 0, 0, 0),       # 128 equal units: 24 spare SMs cannot halve them all
    # the splits measured on a GB300 (GPU time per call, L2 flushed: unsplit -> split)
    (1, 1, 1024, 64, False): (3, 0, 4, 0),       # 19.1 -> 16.0 us
    (1, 1, 2048, 64, False): (4, 0, 8, 0),       # 27.3 -> 17.0 us
    (1, 1, 4096, 64, False): (4, 0, 16, 0),      # 47.7 -> 23.2 us
    (1, 1, 4096, 64, True): (3, 0, 13, 0),       # 47.8 -> 27.3 us
    (1, 1, 8192, 64, True): (4, 0, 26, 0),       # 86.7 -> 35.5 us
    # dynamic splits where the estimate beats the best static one by the margin
    (3, 1, 7000, 64, True): (3, 0, 72, 1),       # static 49.9 -> dynamic 46.1 us
    (1, 4, 6000, 128, True): (2, 0, 56, 0),      # the dynamic estimate is not enough better: static
}


@pytest.mark.parametrize("shape", sorted(PINNED))
def test_pinned_choices(lib, shape):
    assert choice(lib, *shape) == PINNED[shape]


def test_choices_are_runnable_over_a_sweep(lib):
    checked = splits = dyn_splits = 0
    for sms in (132, 148, 152, 160):
        for B, H in ((1, 1), (1, 3), (2, 5), (1, 8), (4, 16)):
            for N in (128, 300, 1000, 2048, 4096, 9000, 16384):
                for d in (64, 128):
                    for causal in (False, True):
                        segs, first, units, dyn = choice(lib, B, H, N, d, causal, sms)
                        p = plan(lib, B, H, N, d, causal, sms)
                        checked += 1
                        assert 1 <= segs <= 4
                        if segs == 1:
                            assert units == 0
                        else:
                            splits += 1
                            assert units >= 1 and first >= 0 and first + units <= p.num_units
                            if dyn:
                                dyn_splits += 1
                                assert causal and p.num_units < sms and first == 0
                            elif p.num_units < sms:
                                assert first == 0 and p.num_units + units * (segs - 1) <= sms  # one wave
                            else:
                                assert not causal and first == p.num_units - p.num_units % sms
                            for u in range(first, first + units):
                                n0, n1 = unit_tiles(u, B * H, N, causal, p.heads_per_group)
                                c = -(-n1 // segs)
                                for s in range(segs):
                                    jb, je = s * c, min(n1, s * c + c)
                                    assert jb < min(je, n0), (B, H, N, causal, sms, u, s)
                        if p.num_units > sms:
                            assert dyn == (1 if causal else 0)
                        else:
                            assert dyn == 0 or segs > 1
    assert checked == 4 * 5 * 7 * 2 * 2 and splits > 20 and dyn_splits > 5


def test_invalid_arguments(lib):
    v = [ctypes.c_int() for _ in range(4)]
    refs = [ctypes.byref(x) for x in v]
    assert lib.attn_fwd_split_choice(1, 1, 128, 64, 0, 0, *refs) == ela.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_split_choice(0, 1, 128, 64, 0, 152, *refs) == ela.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_split_choice(1, 1, 128, 96, 0, 152, *refs) == ela.ATTN_ERR_UNSUPPORTED
    assert lib.attn_fwd_split_choice(1, 1, 128, 64, 0, 152, None, *refs[1:]) == ela.ATTN_ERR_INVALID_ARG

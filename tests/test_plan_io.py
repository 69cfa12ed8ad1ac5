"""The tile planner's I/O count, pinned by walking the kernel's schedule (no GPU).

The planner (csrc/plan.cpp) prices a tiling with a closed form: per (batch,
head), Q read once, O and LSE written once, and K and V streamed once per unit
of q resident 128-row query tiles, or, under the causal mask, only up to each
unit's last query row (the I/O analysis of tall-and-skinny products in the
AttenIO abstract, and the tiling rule of the IO-Aware Algorithms page). Here
the same bytes are counted the slow way instead: every unit is visited, and
the rows it reads and writes are added up, with the K/V rows rounded up to
whole K/V tiles as the kernel streams them. The closed form must equal that
count wherever the tiles divide the sequence. Where they do not (a ragged
causal sequence), the two must stay within the last unit's slack. The planner's
I/O optimum must be the least-traffic tiling that fits the SM (shared memory,
tensor memory, registers) and runs its S = Q K^T product at the full tensor
rate; that is the tiling the kernel is compiled for, at both head dimensions.
"""
import math

import pytest

import exact_long_sequence_gb300 as ela

BR = 128
SMEM_LIMIT = 232448       # opt-in dynamic shared memory per CTA on sm_100-family SMs
TMEM_COLS = 512           # fp32 columns of tensor memory per SM


@pytest.fixture(scope="module", autouse=True)
def lib():
    return ela.load_library()


def walked_bytes(N, d, q, causal, Bc=128):
    """Bytes one (batch, head) moves under a tiling of q query tiles per unit, by enumeration."""
    rows_per_unit = q * BR
    total = 0
    for r0 in range(0, N, rows_per_unit):
        r1 = min(N, r0 + rows_per_unit)
        total += (r1 - r0) * d * 2       # Q rows read (bf16)
        total += (r1 - r0) * d * 2       # O rows written (bf16)
        total += (r1 - r0) * 4           # LSE written (fp32)
        kv_rows = min(N, -(-r1 // Bc) * Bc) if causal else N
        total += 2 * kv_rows * d * 2     # K and V rows streamed (bf16)
    return total


def plan(B, H, N, d, causal):
    return ela.attn_plan(B, H, N, d, causal, num_sms=152)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [256, 1024, 4096, 16384, 65536])
def test_closed_form_equals_the_walk_on_whole_units(N, d, causal):
    B, H = 2, 3
    p = plan(B, H, N, d, causal)
    assert p["l2_bytes"] == pytest.approx(B * H * walked_bytes(N, d, 2, causal), rel=1e-12)


@pytest.mark.parametrize("N", [1, 127, 129, 300, 1000, 4097, 9000])
@pytest.mark.parametrize("d", [64, 128])
def test_closed_form_equals_the_walk_on_ragged_non_causal(N, d):
    p = plan(1, 2, N, d, False)
    assert p["l2_bytes"] == pytest.approx(2 * walked_bytes(N, d, 2, False), rel=1e-12)


@pytest.mark.parametrize("N", [129, 300, 1000, 4097, 9000, 16000])
@pytest.mark.parametrize("d", [64, 128])
def test_ragged_causal_stays_within_the_last_units_slack(N, d):
    """The closed form treats the last unit as full; the walk streams only what exists."""
    p = plan(1, 1, N, d, True)
    walked = walked_bytes(N, d, 2, True)
    units = math.ceil(N / (2 * BR))
    missing = 2 * BR * units - N                  # rows the last unit lacks
    assert p["l2_bytes"] <= walked
    # the closed form averages the units' K/V spans as if the last unit were full,
    # which prices each unit at most `missing` rows of K and of V short.
    assert walked - p["l2_bytes"] <= units * 2 * missing * d * 2
    assert (walked - p["l2_bytes"]) / walked < 2 * BR / N


REGS_PER_SM = 65536


def fits(q, Bc, d, stages=3):
    """The SM's capacity for a tiling, stated from the limits: q resident query tiles and a
    K/V ring of at least three stages in shared memory (plus alignment slack, barriers and
    flags), S and O of every resident tile in tensor memory, and the register file for
    q + 1 warpgroups whose softmax threads hold a row of Bc fp32 scores (plus 40 registers
    of state)."""
    smem = q * BR * d * 2 + stages * (Bc * d * 2 + 16) + 1024 + 19 * 8 + 16
    regs = Bc + 40
    return q * (Bc + d) <= TMEM_COLS and smem <= SMEM_LIMIT and regs <= 255 and 128 * (q + 1) * regs <= REGS_PER_SM


def full_rate(Bc):
    """S = Q K^T with both operands in shared memory: per 16-deep step, Bc / 2 cycles of
    arithmetic (2 * 128 * Bc * 16 FLOP at 8192 per cycle) against (128 + Bc) / 4 cycles of
    operand reads ((128 + Bc) * 16 * 2 bytes at 128 per cycle)."""
    return Bc / 2 >= (128 + Bc) / 4


def least_traffic(N, d, causal, rate_limited=True):
    best = None
    for q in (1, 2, 3, 4):
        for Bc in (64, 128, 256):
            if not fits(q, Bc, d) or (rate_limited and not full_rate(Bc)):
                continue
            key = (walked_bytes(N, d, q, causal, Bc), -q, -Bc)
            if best is None or key < best[0]:
                best = (key, q, Bc)
    return best


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d,N", [(64, 4096), (64, 16384), (128, 16384), (128, 65536)])
def test_io_optimum_is_the_least_walked_traffic_that_fits(d, N, causal):
    best = least_traffic(N, d, causal)
    p = plan(1, 1, N, d, causal)
    assert (p["io_opt_q_tiles"], p["io_opt_Bc"]) == (best[1], best[2])
    assert p["io_opt_l2_bytes"] == pytest.approx(best[0][0], rel=1e-12)
    # the planner arrives at the compiled tiling and reports it
    assert (p["q_tiles"], p["Bc"]) == (best[1], best[2]) == (2, 128)


@pytest.mark.parametrize("N", [4096, 16384, 65536])
def test_tensor_rate_is_what_rules_out_more_resident_tiles_at_d64(N):
    """Without the rate constraint the count alone picks three resident tiles with Bc = 64 at
    d = 64 (four no longer fit the register file); with it, two tiles of Bc = 128."""
    for causal in (False, True):
        unconstrained = least_traffic(N, 64, causal, rate_limited=False)
        assert (unconstrained[1], unconstrained[2]) == (3, 64)
        assert not full_rate(64) and full_rate(128)
        assert (least_traffic(N, 64, causal)[1], least_traffic(N, 64, causal)[2]) == (2, 128)


@pytest.mark.parametrize("d,N", [(64, 4096), (128, 16384), (128, 65536)])
def test_more_resident_rows_never_stream_more(d, N):
    """The I/O analysis' premise: K/V traffic falls as resident query rows grow."""
    for causal in (False, True):
        t = [walked_bytes(N, d, q, causal) for q in (1, 2, 4)]
        assert t[0] > t[1] > t[2]


@pytest.mark.parametrize("N,d", [(4096, 64), (16384, 128), (65536, 128), (262144, 128)])
def test_causal_head_groups_fit_half_of_l2(N, d):
    """A causal schedule group holds as many heads as keep their K and V within 64 MiB."""
    BH = 64
    g = plan(1, BH, N, d, True)["heads_per_group"]
    kv = 2 * N * d * 2
    assert 1 <= g <= BH
    assert g == 1 or g * kv <= 64 << 20
    assert g == BH or (g + 1) * kv > 64 << 20


@pytest.mark.parametrize("B,H,N,d,causal", [(1, 16, 16384, 128, False), (1, 8, 65536, 128, True),
                                            (4, 32, 8192, 128, True), (1, 8, 4096, 64, True)])
def test_hbm_model_is_the_io_bound_when_the_heads_in_flight_fit_l2(B, H, N, d, causal):
    p = plan(B, H, N, d, causal)
    assert p["kv_in_flight_bytes"] <= 96 << 20 and p["l2_fit"] == 1.0
    assert p["hbm_bytes"] == pytest.approx(p["io_bytes"], rel=1e-12)


def test_hbm_model_charges_re_reads_when_one_head_exceeds_l2():
    """N = 262144, d = 128: one head's K and V take 128 MiB, above the 96 MiB budget.  Its 1024
    units run in 1024 / 152 waves of CTAs; every wave after the first re-reads the quarter of the
    head's K/V that L2 does not hold."""
    N, d = 262144, 128
    p = plan(1, 1, N, d, True)
    kv = 2 * N * d * 2
    assert p["kv_in_flight_bytes"] == kv and p["l2_fit"] == pytest.approx(0.75)
    waves = (N // 256) / 152
    assert p["hbm_bytes"] == pytest.approx(p["io_bytes"] + kv * (waves - 1) * 0.25, rel=1e-9)

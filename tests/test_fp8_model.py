"""Model of the FP8 forward's arithmetic, against the fp64 oracle and the FP8 bound (no GPU).

The FP8 kernel (csrc/attn_fwd_fp8_kernel.cuh) multiplies E4M3 codes on the
tensor core with fp32 accumulation, folds the per-tensor scales of Q and K into
the exponent's factor, keeps the bf16 kernel's lazy reference maximum (moved
only when a tile's maximum exceeds it by more than 2^T, T = 8), sums P in fp32,
and rounds P to E4M3 (round to nearest even, saturating at 448) for O += P V.
The row ends with O = O_acc * v_scale / l in bf16 and LSE = ln 2 (m + log2 l).

This test replays that arithmetic in fp32 on sampled rows of seeded E4M3
inputs, the spiky recipe among them. It checks the per-element bound that the
GPU parity test derives from E4M3 rounding:
    |dO_ic| <= 2^-4 sum_j P_ij |v_jc| + 2^-10 sum_j |v_jc| max_j P_ij + 2^-8 |O_ic| + 1e-6,
with P the oracle's exact probabilities, and LSE's per-row 1e-3.

That bound charges every key 2^-10 for its rounding below E4M3's normal range,
so on long rows it grows with the number of keys. On the spiky rows at
N = 4096 its median is about 0.8, for outputs within [-1, 1]. A per-term bound
is just as rigorous and far tighter. Each term p_j = P_ij / max_j P_ij (the
worst case, a reference at the row maximum; a stale reference only scales the
terms up, which does not raise any term's error relative to the row sum) moves
by at most 2^-4 p_j in the normal range (p_j >= 2^-6). Below it, a term moves
by at most min(p_j, 2^-10): below 2^-10 it rounds to zero. So
    |dO_ic| <= max_j P_ij sum_j e_j |v_jc| + 2^-8 |O_ic| + 1e-6.
Both bounds rest on every term staying inside E4M3's range. The lazy reference
guarantees that only while 2^T <= 448. A threshold of 2^16, safe for bf16 P,
lets the spiky rows' terms saturate at 448. The per-term bound catches that,
and the loose one does not. The kernel's static_assert on the shared threshold
exists to rule that case out.
"""
import math

import numpy as np
import pytest
import torch

from exact_long_sequence_gb300 import workloads
from fp8_bound import NEAR_CEILING_OFFSETS, fp8_output_bounds, near_ceiling_inputs

LOG2E = 1.4426950408889634
BC = 128
E4M3_MAX = 448.0


def f32(x):
    return torch.tensor(x, dtype=torch.float32)


def codes_value(c):
    """The E4M3 value of each uint8 code, as fp32 (exact)."""
    return c.view(torch.float8_e4m3fn).float()


def fp8_forward_replay(q8, k8, v8, scales, rows, causal, scale, T=8.0):
    """q8, k8, v8: [N, d] uint8 codes. Returns (O [R, d] of the bf16 output, LSE [R])."""
    N = k8.shape[0]
    qs, ks, vs = scales
    sl2 = f32(scale) * f32(qs) * f32(ks) * f32(LOG2E)
    S = codes_value(q8)[rows] @ codes_value(k8).T
    if causal:
        S = S.masked_fill(torch.arange(N)[None, :] > rows[:, None], float("-inf"))
    vf = codes_value(v8)
    R = len(rows)
    m = torch.full((R,), float("-inf"))
    l = torch.zeros(R)
    O = torch.zeros(R, vf.shape[1])
    for j in range((N + BC - 1) // BC):
        st = S[:, j * BC:(j + 1) * BC]
        if causal and bool(torch.isinf(st).all()):
            break
        mt = st.max(1).values * sl2
        grow = mt > m + T
        alpha = torch.where(grow, torch.exp2(m - mt), torch.ones(R))
        m = torch.where(grow, mt, m)
        m_use = torch.where(torch.isinf(m), torch.zeros(R), m)
        p = torch.exp2(st * sl2 - m_use[:, None])
        l = l * alpha + p.sum(1)
        p8 = p.clamp(max=E4M3_MAX).to(torch.float8_e4m3fn).float()  # cvt.rn.satfinite
        O = O * alpha[:, None] + p8 @ vf[j * BC:(j + 1) * BC]
    out = (O * (f32(vs) / l)[:, None]).to(torch.bfloat16).double().numpy()
    lse = ((m + torch.log2(l)) * math.log(2.0)).double().numpy()
    return out, lse


CASES = [  # N, causal, Q/K recipe, V recipe, seed, sampled rows
    (2048, False, "normal", "normal", 21, 48),
    (2048, True, "normal", "normal", 22, 48),
    (4096, True, "normal_spiky", "uniform", 23, 256),
]


def bound_and_reference(oracle_mod, q8, k8, v8, scales, rows, causal, scale):
    """The oracle's O and LSE, the GPU test's bound and the per-term bound."""
    O, L, P = oracle_mod.attention_fp8(q8[None], k8[None], v8[None], causal, scale, scales=scales,
                                       rows=rows.numpy()[None], return_probs=True)
    O, L, P = O[0], L[0], P[0]
    vabs = np.abs(oracle_mod.decode_e4m3(v8, scales[2]))
    loose, tight = fp8_output_bounds(P, vabs, O)
    return O, L, loose, tight


@pytest.fixture(scope="module")
def cases():
    out = []
    for N, causal, qk, vd, seed, R in CASES:
        q8, k8, v8, scales = workloads.make_inputs_fp8(1, 1, N, 128, seed, qk, vd)
        rows = torch.sort(torch.randperm(N, generator=torch.Generator().manual_seed(seed))[:R]).values
        out.append((q8[0, 0], k8[0, 0], v8[0, 0], scales, rows, causal, qk))
    return out


def test_fp8_arithmetic_meets_both_bounds(oracle_mod, cases):
    scale = 1.0 / math.sqrt(128)
    for q8, k8, v8, scales, rows, causal, qk in cases:
        O_ref, L_ref, loose, tight = bound_and_reference(oracle_mod, q8, k8, v8, scales, rows, causal, scale)
        O, L = fp8_forward_replay(q8, k8, v8, scales, rows, causal, scale)
        err = np.abs(O - O_ref)
        assert (err <= loose).all(), (qk, causal, float((err / loose).max()))
        assert (err <= tight).all(), (qk, causal, float((err / tight).max()))
        assert (np.abs(L - L_ref) <= 1e-3 * np.abs(L_ref)).all(), (qk, causal)


def test_the_loose_bound_is_wide_on_long_peaked_rows(oracle_mod, cases):
    scale = 1.0 / math.sqrt(128)
    q8, k8, v8, scales, rows, causal, qk = cases[-1]
    _, _, loose, tight = bound_and_reference(oracle_mod, q8, k8, v8, scales, rows, causal, scale)
    assert np.median(loose) > 0.5 and np.median(tight) < 0.1


def test_a_threshold_beyond_e4m3_range_breaks_the_per_term_bound(oracle_mod, cases):
    """P above 448 saturates: the lazy reference must keep terms inside E4M3's range."""
    scale = 1.0 / math.sqrt(128)
    q8, k8, v8, scales, rows, causal, qk = cases[-1]
    assert qk == "normal_spiky"
    O_ref, _, loose, tight = bound_and_reference(oracle_mod, q8, k8, v8, scales, rows, causal, scale)
    O, _ = fp8_forward_replay(q8, k8, v8, scales, rows, causal, scale, T=16.0)
    err = np.abs(O - O_ref)
    assert (err > tight).any()
    assert (err <= loose).all()  # the loose bound misses it


def test_near_ceiling_terms_meet_the_bound_and_a_larger_threshold_saturates(oracle_mod):
    """The planted case's terms reach 2^8 (the stale reference at the threshold): exact rounding
    meets the per-term bound; a threshold of 16 lets the offsets above 8 reach 2^9 .. 2^12, which
    saturate at 448 and break it."""
    q8, k8, v8, scales, scale = near_ceiling_inputs()
    rows = torch.arange(256)
    O_ref, L_ref, loose, tight = bound_and_reference(oracle_mod, q8[0, 0], k8[0, 0], v8[0, 0], scales, rows,
                                                     False, scale)
    O, L = fp8_forward_replay(q8[0, 0], k8[0, 0], v8[0, 0], scales, rows, False, scale)
    assert (np.abs(O - O_ref) <= tight).all()
    assert (np.abs(L - L_ref) <= 1e-3 * np.abs(L_ref)).all()
    O16, _ = fp8_forward_replay(q8[0, 0], k8[0, 0], v8[0, 0], scales, rows, False, scale, T=16.0)
    bad = (np.abs(O16 - O_ref) > tight).any(1)
    offsets = np.array(NEAR_CEILING_OFFSETS * (256 // len(NEAR_CEILING_OFFSETS)))
    assert bad.any() and (offsets[bad] > 8.8).all()

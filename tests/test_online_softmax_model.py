"""Model of the forward kernel's online-softmax arithmetic, against the fp64 oracle (no GPU).

The kernel (csrc/attn_fwd_kernel.cuh) streams each query row's keys in tiles
of 128 and keeps, per row, a reference maximum m in log2 units (the scale
folded in). It moves m only when a tile's maximum exceeds it by more than
T (T = 32 in the bf16 kernel, 8 in the FP8 one, whose P is E4M3), rescaling l
and the O accumulator by 2^(m_old - m_new). Every
other tile's terms P = 2^(c s - m) are taken against the stale m and stay
below 2^T. P is summed into l in fp32, rounded to bf16 for O += P V (fp32
accumulation), and the row ends with O / l in bf16 and LSE = ln 2 (m + log2 l).
This is the streaming reformulation of the softmax (IO-Aware Algorithms page;
the FlashAttention structure of the AICF page, section 3), read with a lazy
reference.

The claim that makes the lazy reference exact is that O / l and LSE do not
depend on which m is used, up to rounding. This test replays the arithmetic in
fp32 and bf16 on sampled rows of the seeded workloads, the spiky one among
them, where the reference does move mid-row. It checks:
- the result is within the parity tolerances of the oracle, at T = 8, 32
  and 64;
- results for different T differ only by rounding;
- no term exceeds 2^T.
The model is not the kernel, whose own parity tests run on the GPU. It checks
the arithmetic the kernel is built on.
"""
import math

import numpy as np
import pytest
import torch

from exact_long_sequence_gb300 import workloads

LOG2E = 1.4426950408889634
BC = 128


def lazy_online_softmax(q, k, v, rows, causal, scale, T, rescale_o=True):
    """Replay of the kernel's per-row arithmetic. q, k, v: [N, d] bf16; rows: query positions.
    Returns (O [R, d] fp64 of the bf16 output, LSE [R], number of reference moves past the
    first tile, largest term seen). rescale_o=False plants a mistake: O keeps its old scale
    when the reference moves."""
    N = k.shape[0]
    c = torch.tensor(scale, dtype=torch.float32) * torch.tensor(LOG2E, dtype=torch.float32)
    S = q[rows].float() @ k.float().T                       # fp32 scores [R, N]
    if causal:
        S = S.masked_fill(torch.arange(N)[None, :] > rows[:, None], float("-inf"))
    R, d = len(rows), v.shape[1]
    m = torch.full((R,), float("-inf"))
    l = torch.zeros(R)
    O = torch.zeros(R, d)
    moves, top = 0, 0.0
    for j in range((N + BC - 1) // BC):
        st = S[:, j * BC:(j + 1) * BC]
        if causal and bool(torch.isinf(st).all()):
            break  # past every row's diagonal
        mt = st.max(1).values * c
        grow = mt > m + T
        alpha = torch.where(grow, torch.exp2(m - mt), torch.ones(R))
        if j > 0:
            moves += int(grow.sum())
        m = torch.where(grow, mt, m)
        m_use = torch.where(torch.isinf(m), torch.zeros(R), m)
        p = torch.exp2(st * c - m_use[:, None])              # fp32 terms against the (stale) reference
        top = max(top, float(p.max()))
        l = l * alpha + p.sum(1)
        if rescale_o:
            O = O * alpha[:, None]
        O = O + p.to(torch.bfloat16).float() @ v[j * BC:(j + 1) * BC].float()
    out = (O / l[:, None]).to(torch.bfloat16).double().numpy()
    lse = ((m + torch.log2(l)) * math.log(2.0)).double().numpy()
    return out, lse, moves, top


CASES = [  # workload, (b, h) pairs, rows per head
    ("b1h8n4096d64_causal", [(0, 0), (0, 5)], 64),
    ("b1h16n16384d128", [(0, 3)], 32),
    ("b4h32n8192d128_causal_spiky", [(0, 0), (2, 17), (3, 31)], 64),
]


@pytest.fixture(scope="module")
def case_inputs():
    cache = {}

    def get(name):
        if name not in cache:
            w = workloads.WORKLOADS[name]
            cache[name] = (w, workloads.workload_inputs(w))
        return cache[name]
    return get


@pytest.mark.parametrize("name,heads,R", CASES)
def test_lazy_reference_meets_the_parity_tolerances(oracle_mod, case_inputs, name, heads, R):
    w, (q, k, v) = case_inputs(name)
    g = torch.Generator().manual_seed(11)
    for b, h in heads:
        rows = torch.sort(torch.randperm(w.N, generator=g)[:R]).values
        O_ref, L_ref = oracle_mod.attention_rows(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1],
                                                 w.causal, w.scale, rows=rows.numpy()[None, :])
        O_ref, L_ref = O_ref[0], L_ref[0]
        results = {}
        for T in (8.0, 32.0, 64.0):
            O, L, moves, top = lazy_online_softmax(q[b, h], k[b, h], v[b, h], rows, w.causal, w.scale, T)
            assert np.abs(O - O_ref).max() <= 2e-2, (name, b, h, T)
            assert (np.abs(L - L_ref) <= 1e-3 * np.abs(L_ref)).all(), (name, b, h, T)
            assert top <= 2.0 ** T * (1 + 1e-6)
            results[T] = (O, L, moves)
        # different references change only rounding: within a few bf16 ulps of |O| <= max|V|
        vmax = float(v[b, h].float().abs().max())
        for T in (32.0, 64.0):
            assert np.abs(results[T][0] - results[8.0][0]).max() <= 4 * 2.0 ** -8 * vmax
            assert np.abs(results[T][1] - results[8.0][1]).max() <= 1e-5 * np.abs(L_ref).max()
        if w.qk_dist == "normal_spiky":
            assert results[8.0][2] > 0, "the spiky rows should move their reference mid-row"
            assert results[64.0][2] <= results[8.0][2]


def test_checker_finds_a_missing_o_rescale(oracle_mod, case_inputs):
    """Planted mistake: without the O rescale the spiky rows leave the O tolerance."""
    w, (q, k, v) = case_inputs("b4h32n8192d128_causal_spiky")
    rows = torch.sort(torch.randperm(w.N, generator=torch.Generator().manual_seed(11))[:64]).values
    O_ref, _ = oracle_mod.attention_rows(q[:1, :1], k[:1, :1], v[:1, :1], True, w.scale, rows=rows.numpy()[None, :])
    O, _, moves, _ = lazy_online_softmax(q[0, 0], k[0, 0], v[0, 0], rows, True, w.scale, 8.0, rescale_o=False)
    assert moves > 0 and np.abs(O - O_ref[0]).max() > 2e-2


def test_reference_moves_are_what_rescaling_is_for():
    """A row whose maximum rises by far more than 2^T moves its reference, and the result is
    still the softmax: the largest key takes (almost) all the weight."""
    d, N = 64, 512
    g = torch.Generator().manual_seed(5)
    k = torch.randn(N, d, generator=g).to(torch.bfloat16)
    v = torch.randn(N, d, generator=g).to(torch.bfloat16)
    q = torch.zeros(1, d, dtype=torch.bfloat16)
    q[0, 0] = 64.0
    k[:, 0] = 0.0
    k[400, 0] = 16.0  # in the fourth tile: a logit of 64 * 16 * scale, far above the rest
    O, L, moves, top = lazy_online_softmax(q, k, v, torch.tensor([0]), False, 0.125, 8.0)
    assert moves == 1 and top <= 2.0 ** 8
    np.testing.assert_allclose(O[0], v[400].double().numpy(), atol=2 ** -8 * 4)
    assert abs(L[0] - 64 * 16 * 0.125) < 1e-3 * 128

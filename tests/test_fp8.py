"""GPU parity of the FP8 (E4M3) forward (attn_fwd_fp8) against the fp64 oracle
on the decoded inputs.

Tolerance (a reading: the pages fix no FP8 tolerance).  S is accumulated in
fp32 from exact code products, so LSE keeps the bf16 path's per-row bound
|dLSE| <= 1e-3 |LSE|.  O differs from the exact result through the rounding of
P to E4M3 before the second product.  Every element is held to the per-term
bound of fp8_bound.py, computed from the oracle's exact P:
    |dO_ic| <= max_j P_ij sum_j e_ij |v_jc| + 2^-8 |O_ic| + 1e-6,
    e_ij = 2^-4 p_ij in E4M3's normal range (p_ij = P_ij / max_j P_ij >= 2^-6),
           min(p_ij, 2^-10) below it,
which does not grow with the row length, and the test prints the worst ratio
of error to bound.  The cases include long spiky causal rows (the stress
recipe at N = 4096), where the older per-element bound was loose enough to
pass a saturation bug, and a planted case whose terms reach 2^8, the largest
the stale-maximum threshold allows, with V at E4M3's largest magnitudes.  A
one-hot attention case (every query attends to one key with weight 1, which
E4M3 holds exactly) pins the layout of P and of the transposed V to the exact
answer.  Launches with fewer units than SMs, or a partial last wave, are cut
into K/V segments as in the bf16 forward and merged by the same combine
kernel; their cases are held to the same bound.
"""
import ctypes

import numpy as np
import pytest
import torch

import exact_long_sequence_gb300 as ela
from exact_long_sequence_gb300 import workloads
from fp8_bound import fp8_output_bounds, near_ceiling_inputs

pytestmark = pytest.mark.gpu
D = 128


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from exact_long_sequence_gb300 import _build

    _build.build()
    ela.load_library()


def run(q8, k8, v8, scales, causal, scale=None):
    o, lse = ela.attn_fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), scales, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert ela.last_device_error() == ela.ATTN_OK
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def check(oracle_mod, q8, k8, v8, scales, causal, rows=None, label="", scale=None):
    B, H, N, d = q8.shape
    BH = B * H
    scale = ela.default_scale(d) if scale is None else scale
    o, lse = run(q8, k8, v8, scales, causal, scale)
    o, lse = o.reshape(BH, N, d), lse.reshape(BH, N)
    O, L, P = oracle_mod.attention_fp8(q8, k8, v8, causal, scale, scales=scales, rows=rows, return_probs=True)
    idx = np.arange(N)[None, :].repeat(BH, 0) if rows is None else np.asarray(rows).reshape(BH, -1)
    vabs = np.abs(oracle_mod.decode_e4m3(v8, scales[2]).reshape(BH, N, d))
    _, bound = fp8_output_bounds(P, vabs, O)
    og = np.take_along_axis(o, idx[..., None], 1)
    lg = np.take_along_axis(lse, idx, 1)
    assert np.isfinite(og).all() and np.isfinite(lg).all(), label
    ratio = np.abs(og - O) / bound
    print(f"{label}: worst |dO| / per-term bound = {ratio.max():.3f}, max |dO| = {np.abs(og - O).max():.3e}")
    assert (ratio <= 1).all(), f"{label}: O error above the per-term E4M3 bound by {ratio.max():.3f}x"
    rel = np.abs(lg - L) / np.maximum(np.abs(L), 1e-30)
    assert (np.abs(lg - L) <= 1e-3 * np.abs(L) + 1e-6).all(), f"{label}: LSE rel err {rel.max():.3e}"
    return np.abs(og - O).max()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 17, 128, 129, 300, 1000])
def test_fp8_parity_small(oracle_mod, N, causal):
    q8, k8, v8, sc = workloads.make_inputs_fp8(1, 2, N, D, seed=600 + N)
    check(oracle_mod, q8, k8, v8, sc, causal, label=f"N={N} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [300, 1000])
def test_fp8_one_hot_attention_is_exact(N, causal):
    """Q = K = +-4 codes: the diagonal score (16 d scale ~ 181) beats every other
    one by more than 100, so P is one-hot and O_i = v_i up to the bf16 output."""
    g = torch.Generator().manual_seed(N)
    sign = torch.randint(0, 2, (1, 1, N, D), generator=g, dtype=torch.uint8)
    qk = torch.where(sign == 1, torch.tensor(0x48, dtype=torch.uint8), torch.tensor(0xC8, dtype=torch.uint8))
    v8 = torch.randint(0, 0x7E, (1, 1, N, D), generator=g, dtype=torch.uint8) | (sign << 7)
    sv = 0.125
    o, _ = run(qk, qk.clone(), v8, (1.0, 1.0, sv), causal)
    want = v8.view(torch.float8_e4m3fn).double().numpy() * sv
    np.testing.assert_allclose(o, want, rtol=2.0 ** -8, atol=1e-6)


@pytest.mark.parametrize("name, rows_per_head", [("b1h16n16384d128", 64), ("b1h8n65536d128_causal", 48),
                                                 ("b4h32n8192d128_causal_spiky", 8)])
def test_fp8_workloads_sampled(oracle_mod, name, rows_per_head):
    w = workloads.WORKLOADS[name]
    q8, k8, v8, sc = workloads.make_inputs_fp8(w.B, w.H, w.N, w.d, w.seed, w.qk_dist, w.v_dist)
    rows = workloads.sample_rows(w.B * w.H, w.N, rows_per_head, w.seed)
    err = check(oracle_mod, q8, k8, v8, sc, w.causal, rows=rows.numpy(), label=name)
    assert err < 0.1


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_spiky_long_rows(oracle_mod, causal):
    """The stress recipe (1% of Q and K entries x10, V ~ U(-1, 1)) at N = 4096: long rows
    whose reference maximum moves mid-row; 256 sampled rows per head, first and last included."""
    q8, k8, v8, sc = workloads.make_inputs_fp8(1, 2, 4096, D, 23, "normal_spiky", "uniform")
    rows = workloads.sample_rows(2, 4096, 254, seed=23)
    rows = torch.cat([torch.tensor([[0, 4095]] * 2), rows], dim=1).sort(dim=1).values
    check(oracle_mod, q8, k8, v8, sc, causal, rows=rows.numpy(), label=f"spiky N=4096 causal={causal}")


def test_fp8_terms_at_the_threshold_with_v_at_the_ceiling(oracle_mod):
    """Planted rows whose second key tile scores 6 .. 12 (log2 units) above the first: up to 8
    the reference maximum stays stale and P reaches 2^8 (E4M3 holds up to 448); above 8 it moves.
    V codes are E4M3's largest magnitudes.  A kernel whose terms saturated would break the bound."""
    q8, k8, v8, sc, scale = near_ceiling_inputs()
    check(oracle_mod, q8, k8, v8, sc, False, label="near the E4M3 ceiling", scale=scale)


@pytest.mark.parametrize("B,H,N,causal", [(1, 1, 4096, False), (1, 1, 8192, True), (3, 1, 7000, True),
                                           (1, 13, 3000, False)])
def test_fp8_split_launches(oracle_mod, B, H, N, causal):
    """Launches that take the bf16 forward's work schedule with K/V segments: 16 units cut into
    four, a causal mask with the heaviest units cut, a ragged causal shape whose segments are
    claimed dynamically, and a partial last wave (156 units).  The combine kernel merges the
    segments; every row's result must meet the same per-term bound, and a second launch into
    fresh outputs must give the same bits."""
    lib = ela.load_library()
    segs = [ctypes.c_int() for _ in range(4)]
    assert lib.attn_fwd_split_choice(B, H, N, D, int(causal), torch.cuda.get_device_properties(0).multi_processor_count,
                                     *[ctypes.byref(x) for x in segs]) == ela.ATTN_OK
    assert segs[0].value > 1, "this shape is meant to split"
    q8, k8, v8, sc = workloads.make_inputs_fp8(B, H, N, D, seed=640 + N)
    rows = workloads.sample_rows(B * H, N, 62, seed=N)
    rows = torch.cat([torch.tensor([[0, N - 1]]).repeat(B * H, 1), rows], dim=1).sort(dim=1).values
    check(oracle_mod, q8, k8, v8, sc, causal, rows=rows.numpy(), label=f"split B={B} H={H} N={N} causal={causal}")
    a = ela.attn_fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), sc, causal=causal)
    b = ela.attn_fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), sc, causal=causal,
                         out=torch.full((B, H, N, D), float("nan"), dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_fp8_rejects_bad_arguments():
    q8 = torch.zeros(1, 1, 128, 64, dtype=torch.uint8, device="cuda")
    with pytest.raises(ela.AttnError):
        ela.attn_fwd_fp8(q8, q8, q8, (1.0, 1.0, 1.0))  # d = 64 is not supported
    q8 = torch.zeros(1, 1, 128, D, dtype=torch.uint8, device="cuda")
    for bad in ((0.0, 1.0, 1.0), (1.0, float("nan"), 1.0), (1.0, 1.0, -1.0)):
        with pytest.raises(ela.AttnError):
            ela.attn_fwd_fp8(q8, q8, q8, bad)


@pytest.mark.parametrize("B,H,N", [(1, 2, 300), (1, 8, 8192)])
def test_fp8_outputs_and_workspace_stay_inside_their_buffers(B, H, N):
    """Causal; the second shape (256 units) takes the dynamic schedule, whose counter sits at the
    end of the workspace."""
    q8, k8, v8, sc = workloads.make_inputs_fp8(B, H, N, D, seed=11)
    n = B * H * N * D
    o_buf = torch.full((n + 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    l_buf = torch.full((B * H * N + 1024,), 7.0, dtype=torch.float32, device="cuda")
    need = ela.load_library().attn_fwd_fp8_workspace_bytes(B, H, N, D)
    ws = torch.full((need + 4096,), 0x5A, dtype=torch.uint8, device="cuda")
    o = o_buf[:n].view(B, H, N, D)
    lse = l_buf[: B * H * N].view(B, H, N)
    ela.attn_fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), sc, causal=True, out=o, lse=lse, workspace=ws[:need])
    torch.cuda.synchronize()
    assert ela.last_device_error() == ela.ATTN_OK
    assert (o_buf[n:] == 7.0).all() and (l_buf[B * H * N:] == 7.0).all() and (ws[need:] == 0x5A).all()

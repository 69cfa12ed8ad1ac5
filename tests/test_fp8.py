"""GPU parity of the FP8 (E4M3) forward (attn_fwd_fp8) against the fp64 oracle
on the decoded inputs.

Tolerance (a reading: the pages fix no FP8 tolerance).  S is accumulated in
fp32 from exact code products, so LSE keeps the bf16 path's per-row bound
|dLSE| <= 1e-3 |LSE|.  O differs from the exact result through the rounding of
P to E4M3 before the second product.  The kernel's P is p_j = 2^(c s_j - m)
with m at most the row maximum, so its row sum l is at least
L_i = sum_j exp(s_ij - max_j s_ij) = 1 / max_j P_ij.  E4M3 rounding moves a
value by at most 2^-4 of itself in the normal range and by at most 2^-10 below
it, which gives, per element,
    |dO_ic| <= 2^-4 sum_j P_ij |v_jc| + 2^-10 sum_j |v_jc| / L_i + 2^-8 |O_ic| + 1e-6,
the last two terms covering the bf16 output and the fp32 sums.  The bound is
computed from the oracle's exact P.  On long peaked rows it is loose (its
second term grows with the number of keys); test_fp8_model.py derives a
per-term bound from the same rounding facts and checks the kernel's arithmetic
against both on the CPU.  A one-hot attention case (every query
attends to one key with weight 1, which E4M3 holds exactly) pins the layout of
P and of the transposed V to the exact answer.
"""
import numpy as np
import pytest
import torch

import exact_long_sequence_gb300 as ela
from exact_long_sequence_gb300 import workloads

pytestmark = pytest.mark.gpu
D = 128


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from exact_long_sequence_gb300 import _build

    _build.build()
    ela.load_library()


def run(q8, k8, v8, scales, causal):
    o, lse = ela.attn_fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), scales, causal=causal)
    torch.cuda.synchronize()
    assert ela.last_device_error() == ela.ATTN_OK
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def check(oracle_mod, q8, k8, v8, scales, causal, rows=None, label=""):
    B, H, N, d = q8.shape
    BH = B * H
    o, lse = run(q8, k8, v8, scales, causal)
    o, lse = o.reshape(BH, N, d), lse.reshape(BH, N)
    O, L, P = oracle_mod.attention_fp8(q8, k8, v8, causal, ela.default_scale(d), scales=scales, rows=rows,
                                       return_probs=True)
    idx = np.arange(N)[None, :].repeat(BH, 0) if rows is None else np.asarray(rows).reshape(BH, -1)
    vabs = np.abs(oracle_mod.decode_e4m3(v8, scales[2]).reshape(BH, N, d))
    bound = (2.0 ** -4 * np.einsum("brn,bnd->brd", P, vabs)
             + 2.0 ** -10 * vabs.sum(1)[:, None, :] * P.max(-1)[..., None]
             + 2.0 ** -8 * np.abs(O) + 1e-6)
    og = np.take_along_axis(o, idx[..., None], 1)
    lg = np.take_along_axis(lse, idx, 1)
    assert np.isfinite(og).all() and np.isfinite(lg).all(), label
    excess = np.abs(og - O) - bound
    assert (excess <= 0).all(), f"{label}: O error above the E4M3 bound by {excess.max():.3e}"
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

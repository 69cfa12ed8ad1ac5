"""GPU parity of the K/V split (attn_fwd_split).

Problems with fewer work units than SMs cut the K/V range of their long units
into segments that run on different CTAs; a second kernel merges the segments'
partial results of each row by their LSE weights.  Causal problems may take the
dynamic schedule for their segments.  The result is the same operation as
attn_fwd, so the forward's tolerances apply unchanged: against the fp64 oracle
max |dO| <= 2e-2 and per-row |dLSE| <= 1e-3 |LSE|.  The shapes below are chosen
so that the launch splits units into 2, 3 and 4 segments on a 152-SM GB300 (the
test checks the split the library reports is the expected one), with causal
masks, ragged lengths, several schedule groups, units left whole beside split
ones, and split items claimed dynamically.  A second launch into fresh outputs
with the same workspace must give the same bits.

Causal problems with more units than SMs take the same entry's dynamic
schedule instead: CTAs claim units from a counter in the workspace.  Each unit
is computed as by attn_fwd, so those outputs must equal attn_fwd's bit for bit.
"""
import pytest
import torch

import exact_long_sequence_gb300 as ela
from exact_long_sequence_gb300 import workloads

pytestmark = pytest.mark.gpu

O_TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from exact_long_sequence_gb300 import _build

    _build.build()
    ela.load_library()


def chosen_split(B, H, N, d, causal):
    """Segments per split unit that the library chose (1: no split)."""
    return ela.split_segments(B, H, N, d, causal)


# (B, H, N, d, causal, segments per split unit expected on 152 SMs).  With fewer
# units than SMs, the heaviest units are split, as many as the idle SMs allow.
# With more (equal, non-causal) units, the units of the last partial wave are.
CASES = [
    (1, 8, 4096, 64, True, 2),     # the causal d = 64 workload: 128 units, 120 halved, claimed dynamically
    (1, 4, 6000, 128, True, 2),    # ragged causal, 96 units: the 56 heaviest halved in one wave
    (3, 1, 7000, 128, True, 3),    # ragged causal, three schedule groups, 72 units in thirds, dynamic
    (3, 1, 7000, 64, True, 3),     # ragged causal, three schedule groups, dynamic
    (1, 2, 8192, 128, False, 2),   # 64 equal units, all split
    (1, 1, 1000, 64, False, 3),    # 4 units of 8 K/V tiles, ragged length
    (1, 5, 3000, 64, True, 3),     # ragged causal, 60 units of which 45 split
    (2, 1, 2000, 128, True, 3),    # ragged causal, two batches in two schedule groups
    (1, 1, 4096, 128, False, 4),   # 16 units of 32 K/V tiles
    (1, 1, 8192, 64, True, 4),     # causal, 32 units of which 26 split
    # more equal units than SMs: the last, partial wave's units are split
    (1, 10, 4096, 128, False, 4),  # 160 units: 8 split into 4, spread over all SMs
    (1, 13, 3000, 128, False, 4),  # 156 units, ragged length
    (1, 16, 16384, 128, False, 4), # the long-sequence workload: 1024 units, the last 112 split
]


@pytest.mark.parametrize("B,H,N,d,causal,segs", CASES)
def test_split_parity(oracle_mod, B, H, N, d, causal, segs):
    needs_152_sms()
    assert chosen_split(B, H, N, d, causal) == segs
    q, k, v = workloads.make_inputs(B, H, N, d, seed=900 + N + H)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    ws = torch.empty(ela.split_workspace_bytes(B, H, N, d, causal), dtype=torch.uint8, device="cuda")
    o, lse = ela.attn_fwd(qd, kd, vd, causal=causal, workspace=ws)
    o2 = torch.full_like(o, float("nan"))
    lse2 = torch.full_like(lse, float("nan"))
    ela.attn_fwd(qd, kd, vd, causal=causal, workspace=ws, out=o2, lse=lse2)
    o1, lse1 = ela.attn_fwd(qd, kd, vd, causal=causal, split=False)
    torch.cuda.synchronize()
    assert ela.last_device_error() == ela.ATTN_OK
    assert torch.equal(o, o2) and torch.equal(lse, lse2), "a second launch on the same workspace differs"
    # every row of the small cases, sampled rows (with the first and last) of the long ones
    R = N if B * H * N <= 16384 else 48
    rows = None
    if R < N:
        rows = workloads.sample_rows(B * H, N, R - 2, seed=N)
        ends = torch.tensor([[0, N - 1]]).repeat(B * H, 1)
        rows = torch.cat([ends, rows], dim=1).sort(dim=1).values
    O_ref, L_ref = oracle_mod.attention_rows(q, k, v, causal, ela.default_scale(d),
                                             rows=None if rows is None else rows.numpy())
    for out, lout, label in ((o, lse, "split"), (o1, lse1, "unsplit")):
        oo = out.reshape(B * H, N, d)
        ll = lout.reshape(B * H, N)
        if rows is not None:
            idx = rows.cuda()
            oo = torch.gather(oo, 1, idx[:, :, None].expand(-1, -1, d))
            ll = torch.gather(ll, 1, idx)
        oo = oo.double().cpu().numpy()
        ll = ll.double().cpu().numpy()
        err = abs(oo - O_ref).max()
        rel = (abs(ll - L_ref) / abs(L_ref)).max()
        assert err <= O_TOL, f"{label}: max|dO| = {err:.3e}"
        assert rel <= 1e-3, f"{label}: max rel dLSE = {rel:.3e}"
    # the split and the single kernel agree to the bf16 output's rounding
    assert (o.float() - o1.float()).abs().max().item() <= 2 ** -7 * max(1.0, o1.float().abs().max().item())


def test_no_split_when_it_would_not_pay():
    """Causal launches with more units than SMs, equal units that fill the SMs exactly or whose
    last wave does not pay to split, or units the idle SMs cannot all split: no split."""
    needs_152_sms()
    for shape in ((1, 8, 65536, 128, True), (1, 8, 4096, 64, False), (1, 1, 256, 64, False),
                  (1, 19, 2048, 64, False), (2, 9, 4096, 64, False)):
        assert chosen_split(*shape) == 1
    # non-causal: no workspace at all (152 units fill the SMs exactly; 288 units: no split pays);
    # causal with more units than SMs: the schedule counter only
    assert ela.split_workspace_bytes(1, 19, 2048, 64, False) == 0
    assert ela.split_workspace_bytes(2, 9, 4096, 64, False) == 0
    assert ela.split_workspace_bytes(1, 8, 65536, 128, True) == 256


@pytest.mark.parametrize("B,H,N,d", [(2, 8, 8192, 64), (1, 5, 20000, 128), (3, 40, 1000, 64)])
def test_dynamic_schedule_is_bit_identical(oracle_mod, B, H, N, d):
    """Causal, more units than SMs: CTAs claim units dynamically; every unit is computed as by
    the static schedule of attn_fwd, so O and LSE are equal bit for bit (and match the oracle)."""
    needs_152_sms()
    assert ela.split_workspace_bytes(B, H, N, d, True) == 256
    q, k, v = workloads.make_inputs(B, H, N, d, seed=700 + N)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    ws = torch.full((4096,), 0x5A, dtype=torch.uint8, device="cuda")
    o, lse = ela.attn_fwd(qd, kd, vd, causal=True, workspace=ws[:256])
    o_again, lse_again = ela.attn_fwd(qd, kd, vd, causal=True, workspace=ws[:256])
    o1, lse1 = ela.attn_fwd(qd, kd, vd, causal=True, split=False)
    torch.cuda.synchronize()
    assert ela.last_device_error() == ela.ATTN_OK
    assert torch.equal(o, o1) and torch.equal(lse, lse1)
    assert torch.equal(o_again, o1) and torch.equal(lse_again, lse1)
    assert (ws[256:] == 0x5A).all()  # nothing written past the counter block
    rows = workloads.sample_rows(B * H, N, 6, seed=N)
    O_ref, L_ref = oracle_mod.attention_rows(q, k, v, True, ela.default_scale(d), rows=rows.numpy())
    idx = rows.cuda()
    og = torch.gather(o.reshape(B * H, N, d), 1, idx[:, :, None].expand(-1, -1, d)).double().cpu().numpy()
    lg = torch.gather(lse.reshape(B * H, N), 1, idx).double().cpu().numpy()
    assert abs(og - O_ref).max() <= O_TOL
    assert (abs(lg - L_ref) / abs(L_ref)).max() <= 1e-3


def needs_152_sms():
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the shapes split on 152 SMs")


def test_split_rejects_a_missing_or_short_workspace():
    needs_152_sms()
    lib = ela.load_library()
    B, H, N, d = 1, 8, 4096, 64
    need = ela.split_workspace_bytes(B, H, N, d, True)
    assert need > 0
    q = torch.zeros(B, H, N, d, dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
    ws = torch.empty(need + 64, dtype=torch.uint8, device="cuda")
    args = (q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d, 1, 0.125)
    assert lib.attn_fwd_split(*args, None, 0, None) == ela.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_split(*args, ws.data_ptr(), need - 1, None) == ela.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_split(*args, ws.data_ptr() + 4, need, None) == ela.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_split(*args, ws.data_ptr(), need, None) == ela.ATTN_OK
    torch.cuda.synchronize()
    assert ela.last_device_error() == ela.ATTN_OK
    # no split for this shape: a NULL workspace is accepted
    small = (q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 1, 256, d, 0, 0.125)
    assert ela.split_workspace_bytes(1, 1, 256, d, False) == 0
    assert lib.attn_fwd_split(*small, None, 0, None) == ela.ATTN_OK
    torch.cuda.synchronize()


def test_split_stays_inside_its_buffers():
    """Guard canaries after O, LSE and the workspace stay untouched by a split launch."""
    needs_152_sms()
    B, H, N, d = 1, 5, 3000, 64
    need = ela.split_workspace_bytes(B, H, N, d, True)
    assert need > 0
    q, k, v = (t.cuda() for t in workloads.make_inputs(B, H, N, d, seed=5))
    o_buf = torch.full((B * H * N * d + 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    l_buf = torch.full((B * H * N + 1024,), 7.0, dtype=torch.float32, device="cuda")
    w_buf = torch.full((need + 8192,), 0x5A, dtype=torch.uint8, device="cuda")
    o = o_buf[: B * H * N * d].view(B, H, N, d)
    lse = l_buf[: B * H * N].view(B, H, N)
    ela.attn_fwd(q, k, v, causal=True, out=o, lse=lse, workspace=w_buf[:need])
    torch.cuda.synchronize()
    assert ela.last_device_error() == ela.ATTN_OK
    assert (o_buf[B * H * N * d:] == 7.0).all() and (l_buf[B * H * N:] == 7.0).all()
    assert (w_buf[need:] == 0x5A).all()

"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded bf16 inputs.

Tolerances (fixed by the target, not tuned): max |O_gpu - O_oracle| <= 2e-2 over
every compared element, and per row |LSE_gpu - LSE_oracle| <= 1e-3 |LSE_oracle|.
"""
import numpy as np
import pytest
import torch

import exact_long_sequence_gb300 as ela
from exact_long_sequence_gb300 import workloads

pytestmark = pytest.mark.gpu

O_TOL = 2e-2
LSE_RTOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from exact_long_sequence_gb300 import _build

    _build.build()
    ela.load_library()


def compare(o, lse, q, k, v, causal, scale, rows, oracle_mod, label=""):
    """Check GPU outputs against the oracle on `rows` ([BH, R] or None = all)."""
    B, H, N, d = q.shape
    O_ref, L_ref = oracle_mod.attention_rows(q, k, v, causal, scale, rows=None if rows is None else rows.numpy())
    o = o.reshape(B * H, N, d)
    lse = lse.reshape(B * H, N)
    if rows is None:
        o_cmp = o.double().cpu().numpy()
        l_cmp = lse.double().cpu().numpy()
    else:
        idx = rows.to(o.device)
        o_cmp = torch.gather(o, 1, idx[:, :, None].expand(-1, -1, d)).double().cpu().numpy()
        l_cmp = torch.gather(lse, 1, idx).double().cpu().numpy()
    assert np.isfinite(o_cmp).all() and np.isfinite(l_cmp).all(), f"{label}: non-finite output"
    err_o = np.abs(o_cmp - O_ref).max()
    dl = np.abs(l_cmp - L_ref)
    # per row |dLSE| <= 1e-3 |LSE|; a row whose exact LSE is 0 (one visible key at a zero
    # score) must then be exact
    rel_l = np.divide(dl, np.abs(L_ref), out=np.where(dl == 0, 0.0, np.inf), where=L_ref != 0)
    worst = np.unravel_index(np.argmax(rel_l), rel_l.shape)
    assert err_o <= O_TOL, f"{label}: max|dO| = {err_o:.3e}"
    assert (dl <= LSE_RTOL * np.abs(L_ref)).all(), (f"{label}: worst rel dLSE = {rel_l.max():.3e} at row {worst} "
                                                    f"(|LSE| = {abs(L_ref[worst]):.3e})")
    return err_o, rel_l.max()


def run(q, k, v, causal, scale=None, prefill=float("nan")):
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.full_like(qd, prefill)
    lse = torch.full(q.shape[:3], prefill, dtype=torch.float32, device=dev)
    ela.attn_fwd(qd, kd, vd, causal=causal, scale=scale, out=o, lse=lse)
    assert ela.last_device_error() == ela.ATTN_OK
    return o, lse


@pytest.mark.parametrize("name", list(workloads.WORKLOADS))
def test_workload_parity(oracle_mod, name):
    """Every named workload, at full size; large ones on the sampled query rows."""
    w = workloads.WORKLOADS[name]
    q, k, v = workloads.workload_inputs(w)
    o, lse = run(q, k, v, w.causal, w.scale)
    rows = workloads.workload_rows(w)
    # every element is written (NaN pre-fill), not just the compared rows
    assert not torch.isnan(o).any() and not torch.isnan(lse).any()
    err_o, err_l = compare(o, lse, q, k, v, w.causal, w.scale, rows, oracle_mod, name)
    print(f"{name}: max|dO|={err_o:.3e} max rel dLSE={err_l:.3e}")


EDGE_N = [1, 2, 17, 127, 128, 129, 255, 256, 257, 383, 1000]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", EDGE_N)
def test_ragged_lengths(oracle_mod, N, causal, d):
    """Lengths that end inside a tile, at a tile edge, or leave the second query tile of a pair empty."""
    q, k, v = workloads.make_inputs(1, 3, N, d, seed=100 + N)
    o, lse = run(q, k, v, causal)
    assert not torch.isnan(o).any() and not torch.isnan(lse).any()
    compare(o, lse, q, k, v, causal, ela.default_scale(d), None, oracle_mod, f"N={N} d={d} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_more_units_than_sms(oracle_mod, causal):
    """B*H*pairs well above the SM count: every persistent CTA runs several units."""
    q, k, v = workloads.make_inputs(3, 70, 300, 64, seed=7)
    o, lse = run(q, k, v, causal)
    compare(o, lse, q, k, v, causal, ela.default_scale(64), None, oracle_mod, "many units")


@pytest.mark.parametrize("N,d", [(1 << 20, 64), (1 << 19, 128)])
def test_longest_sequences(oracle_mod, N, d):
    """Million-token causal attention: sampled rows, always including the first and last."""
    q, k, v = workloads.make_inputs(1, 1, N, d, seed=50 + d)
    o, lse = run(q, k, v, True)
    rows = workloads.sample_rows(1, N, 14, seed=50 + d)
    rows = torch.cat([torch.tensor([[0, N - 1]]), rows], dim=1).sort(dim=1).values
    compare(o, lse, q, k, v, True, ela.default_scale(d), rows, oracle_mod, f"N={N} d={d}")


def test_many_heads(oracle_mod):
    """16384 (batch, head) pairs of 64 tokens: every persistent CTA runs over a hundred units."""
    B, H, N, d = 128, 128, 64, 64
    q, k, v = workloads.make_inputs(B, H, N, d, seed=60)
    o, lse = run(q, k, v, False)
    rows = workloads.sample_rows(B * H, N, 3, seed=60)
    compare(o, lse, q, k, v, False, ela.default_scale(d), rows, oracle_mod, "many heads")


def test_outputs_stay_inside_their_buffers():
    """Guard canaries after O and LSE stay untouched."""
    B, H, N, d = 1, 2, 300, 128
    q, k, v = (t.cuda() for t in workloads.make_inputs(B, H, N, d, seed=3))
    o_buf = torch.full((B * H * N * d + 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    l_buf = torch.full((B * H * N + 1024,), 7.0, dtype=torch.float32, device="cuda")
    o = o_buf[: B * H * N * d].view(B, H, N, d)
    lse = l_buf[: B * H * N].view(B, H, N)
    ela.attn_fwd(q, k, v, causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    assert (o_buf[B * H * N * d:] == 7.0).all() and (l_buf[B * H * N:] == 7.0).all()


def test_invariants_on_gpu():
    """Constant V gives constant O; N = 1 gives O = V and LSE = scale q.k;
    non-causal output is invariant under a shared K/V row permutation."""
    q, k, _ = workloads.make_inputs(1, 2, 500, 128, seed=5)
    v = torch.full_like(q, 0.625)
    o, _ = run(q, k, v, True)
    assert (o.float() - 0.625).abs().max().item() <= O_TOL

    q1, k1, v1 = workloads.make_inputs(2, 2, 1, 64, seed=6)
    o, lse = run(q1, k1, v1, False, 0.125)
    assert torch.equal(o.cpu(), v1)
    ref = 0.125 * (q1.double() * k1.double()).sum(-1)
    assert torch.allclose(lse.double().cpu(), ref, rtol=1e-5, atol=1e-6)

    q, k, v = workloads.make_inputs(1, 1, 700, 64, seed=8)
    perm = torch.randperm(700, generator=torch.Generator().manual_seed(1))
    o1, l1 = run(q, k, v, False)
    o2, l2 = run(q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous(), False)
    assert (o1.float() - o2.float()).abs().max().item() <= 2e-2
    assert ((l1 - l2).abs() / l1.abs()).max().item() <= 1e-5


def test_deterministic():
    q, k, v = (t.cuda() for t in workloads.make_inputs(1, 4, 1100, 128, seed=9))
    a = ela.attn_fwd(q, k, v, causal=True)
    b = ela.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_host_buffer_entry_matches_device_entry():
    q, k, v = workloads.make_inputs(1, 3, 777, 128, seed=10)
    qp, kp, vp = (t.pin_memory() for t in (q, k, v))
    stream = torch.cuda.Stream()
    o_h, l_h = ela.attn_fwd_host(qp, kp, vp, causal=True, stream=stream)
    stream.synchronize()
    # the host entry runs the single-kernel attn_fwd on each chunk: the same bits
    o_d, l_d = ela.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, split=False)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(l_h, l_d.cpu())


@pytest.mark.parametrize("B,H,N,causal", [(2, 9, 333, True), (1, 1, 200, False), (3, 6, 1024, False)])
def test_host_buffer_entry_chunks(oracle_mod, B, H, N, causal):
    """The host-buffer entry splits (batch, head) pairs into chunks with overlapped
    copies; results equal the oracle and the device entry for uneven chunk sizes."""
    q, k, v = workloads.make_inputs(B, H, N, 64, seed=40 + N)
    qp, kp, vp = (t.pin_memory() for t in (q, k, v))
    o_h, l_h = ela.attn_fwd_host(qp, kp, vp, causal=causal)
    torch.cuda.current_stream().synchronize()
    compare(o_h, l_h, q, k, v, causal, ela.default_scale(64), None, oracle_mod, "host entry")
    o_d, l_d = ela.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, split=False)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(l_h, l_d.cpu())


def test_side_stream_and_scale(oracle_mod):
    q, k, v = workloads.make_inputs(2, 2, 200, 64, seed=11)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
        o, lse = ela.attn_fwd(qd, kd, vd, causal=False, scale=0.3, stream=s)
    s.synchronize()
    compare(o, lse, q, k, v, False, 0.3, None, oracle_mod, "side stream")


@pytest.mark.parametrize("scale", [-0.125, -0.3, 0.0])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("split", [False, True])
def test_negative_and_zero_scale(oracle_mod, scale, d, causal, split):
    """Any finite scale: a negative one runs as |scale| on the negated scores (the MMA's
    negate bit), so the running maximum follows the largest scaled score; zero gives the
    plain average of the visible values and LSE = ln(#visible).  Ragged length; with
    split=True the launch takes the K/V split and its in-kernel merge."""
    q, k, v = workloads.make_inputs(1, 3, 300, d, seed=170 + d)
    dev = torch.device("cuda")
    o = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device=dev)
    ela.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=scale, out=o, lse=lse, split=split)
    assert ela.last_device_error() == ela.ATTN_OK
    compare(o, lse, q, k, v, causal, scale, None, oracle_mod, f"scale={scale} d={d} causal={causal}")


def test_negative_scale_on_a_spiky_long_row(oracle_mod):
    """The stress recipe's large entries with a negative scale: the smallest raw scores
    become the largest scaled ones, and the running maximum must move with them."""
    q, k, v = workloads.make_inputs(1, 2, 4096, 128, seed=180, qk_dist="normal_spiky", v_dist="uniform")
    o, lse = run(q, k, v, True, -ela.default_scale(128))
    rows = workloads.sample_rows(2, 4096, 128, seed=180)
    compare(o, lse, q, k, v, True, -ela.default_scale(128), rows, oracle_mod, "spiky negative scale")


def test_bounded_wait_reports_timeout_and_context_survives(oracle_mod):
    """A wait nobody satisfies gives up after its limit: the kernel records a
    timeout, exits normally, and the next launch still works."""
    assert ela.debug_wait_timeout(50_000_000) == ela.ATTN_OK
    assert ela.last_device_error() == ela.ATTN_ERR_TIMEOUT
    assert ela.last_device_error() == ela.ATTN_OK  # the read cleared it
    q, k, v = workloads.make_inputs(1, 1, 256, 64, seed=12)
    o, lse = run(q, k, v, True)
    compare(o, lse, q, k, v, True, ela.default_scale(64), None, oracle_mod, "after timeout")


def test_rejects_bad_tensors():
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        ela.attn_fwd(q.float(), q.float(), q.float())
    with pytest.raises(ela.AttnError) as e:
        ela.attn_fwd(q, q, q, scale=float("nan"))
    assert e.value.status == ela.ATTN_ERR_INVALID_ARG
    x = torch.zeros(1, 1, 128, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ela.AttnError) as e:
        ela.attn_fwd(x, x, x)
    assert e.value.status == ela.ATTN_ERR_UNSUPPORTED

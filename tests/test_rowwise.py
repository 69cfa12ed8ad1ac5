"""GPU parity of the standalone streaming row softmax and layer normalisation
against the fp64 oracle.

Tolerances (a reading; the pages fix none for these operations).  The kernels
compute in fp32 and round the output to bf16 (2^-9 relative).  fp32 errors
(exp2, sums over at most 2^20 elements, the normalisation) stay well below
2^-12 relative, so softmax is held to |dy| <= 2^-8 |y| + 1e-37 (the absolute
term covers results below fp32's normal range, which are flushed to zero), and
layer normalisation to |dy| <= 2^-8 |y| + 2e-3 |gamma_i| + 1e-6 (the second
term covers the fp32 cancellation in x - mean for rows with an offset).
"""
import numpy as np
import pytest
import torch

import exact_long_sequence_gb300 as ela
from exact_long_sequence_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from exact_long_sequence_gb300 import _build

    _build.build()
    ela.load_library()


def rows(R, N, seed, scale=3.0, offset=0.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(R, N, generator=g) * scale + offset).to(torch.bfloat16)


def check_softmax(oracle_mod, x, y):
    ref = oracle_mod.softmax_rows(x)
    got = y.double().cpu().numpy()
    err = np.abs(got - ref) - (2.0 ** -8 * np.abs(ref) + 1e-37)
    assert (err <= 0).all(), f"softmax error above bound by {err.max():.3e}"
    np.testing.assert_allclose(got.sum(-1), 1.0, atol=2.0 ** -7)


@pytest.mark.parametrize("R,N", [(1, 8), (3, 64), (5, 1000), (7, 16384), (2, 65536), (3, 65544), (2, 200000),
                                 (1, 1 << 20), (2, (1 << 20) + 8), (4096, 1024)])
def test_softmax_rows_parity(oracle_mod, R, N):
    N = (N + 7) // 8 * 8
    x = rows(R, N, seed=R * 7 + N)
    check_softmax(oracle_mod, x, ela.softmax_rows(x.cuda()))


def test_softmax_rows_large_offset_and_in_place(oracle_mod):
    x = rows(6, 4096, seed=3, offset=1000.0)
    xd = x.cuda()
    ela.softmax_rows(xd, out=xd)
    check_softmax(oracle_mod, x, xd)


def check_layernorm(oracle_mod, x, g, b, eps, y):
    ref = oracle_mod.layernorm_rows(x, g, b, eps)
    got = y.double().cpu().numpy()
    gabs = np.abs(g.double().numpy())[None, :]
    err = np.abs(got - ref) - (2.0 ** -8 * np.abs(ref) + 2e-3 * gabs + 1e-6)
    assert (err <= 0).all(), f"layernorm error above bound by {err.max():.3e}"


@pytest.mark.parametrize("R,N", [(3, 8), (4, 1024), (64, 4096), (16, 8192), (5, 24000), (2, 65536)])
def test_layernorm_rows_parity(oracle_mod, R, N):
    x = rows(R, N, seed=N + R, scale=1.0, offset=3.0)
    gen = torch.Generator().manual_seed(N)
    g = (1 + 0.2 * torch.randn(N, generator=gen)).to(torch.bfloat16)
    b = (0.3 * torch.randn(N, generator=gen)).to(torch.bfloat16)
    y = ela.layernorm_rows(x.cuda(), g.cuda(), b.cuda(), eps=1e-5)
    check_layernorm(oracle_mod, x, g, b, 1e-5, y)


@pytest.mark.parametrize("R,N", [(2000, 8), (3001, 1000), (1000, 2048), (700, 11264), (700, 11272)])
def test_layernorm_many_rows_parity(oracle_mod, R, N):
    """Many rows (several waves of one CTA per row), rows of one to 1409 chunks."""
    x = rows(R, N, seed=N + 3 * R, scale=1.0, offset=3.0)
    gen = torch.Generator().manual_seed(N + 1)
    g = (1 + 0.2 * torch.randn(N, generator=gen)).to(torch.bfloat16)
    b = (0.3 * torch.randn(N, generator=gen)).to(torch.bfloat16)
    y = ela.layernorm_rows(x.cuda(), g.cuda(), b.cuda(), eps=1e-5)
    check_layernorm(oracle_mod, x, g, b, 1e-5, y)


def test_layernorm_constant_rows_give_beta_and_in_place(oracle_mod):
    N = 512
    x = torch.full((3, N), -2.5, dtype=torch.bfloat16)
    g = torch.linspace(0.5, 1.5, N).to(torch.bfloat16)
    b = torch.linspace(-1, 1, N).to(torch.bfloat16)
    xd = x.cuda()
    ela.layernorm_rows(xd, g.cuda(), b.cuda(), eps=1e-3, out=xd)
    torch.testing.assert_close(xd.cpu(), b.expand(3, N), rtol=0, atol=0)


@pytest.mark.parametrize("name", list(workloads.ROW_WORKLOADS))
def test_row_workloads_sampled(oracle_mod, name):
    """The benchmarked row workloads at full size, on the benchmark's seeded host inputs and in
    its call (the softmax with the workspace its segmented path asks for): 64 sampled rows
    against the oracle, and every row's softmax sum."""
    kind, R, N = workloads.ROW_WORKLOADS[name]
    inp = workloads.row_inputs(kind, R, N, seed=1)
    rows_idx = torch.sort(torch.randperm(R, generator=torch.Generator().manual_seed(7))[:64]).values
    if kind == "softmax":
        need = ela.load_library().attn_softmax_rows_workspace_bytes(R, N)
        ws = torch.empty(max(need, 8), dtype=torch.uint8, device="cuda") if need else None
        y = ela.softmax_rows(inp.cuda(), workspace=ws)
        torch.cuda.synchronize()
        sums = y.float().sum(-1)
        assert (sums - 1).abs().max().item() <= 2.0 ** -7
        check_softmax(oracle_mod, inp[rows_idx], y[rows_idx.cuda()])
    else:
        x, g, b = inp
        y = ela.layernorm_rows(x.cuda(), g.cuda(), b.cuda(), eps=1e-5)
        torch.cuda.synchronize()
        check_layernorm(oracle_mod, x[rows_idx], g, b, 1e-5, y[rows_idx.cuda()])


def test_row_ops_reject_bad_shapes():
    x = torch.zeros(4, 12, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ela.AttnError):
        ela.softmax_rows(x)  # N not a multiple of 8
    x = torch.zeros(2, 65544, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(65544, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ela.AttnError):
        ela.layernorm_rows(x, g, g)  # longer than one CTA holds


@pytest.mark.parametrize("N", [1000, 65544, (1 << 20) + 8])
def test_row_outputs_and_workspace_stay_inside_their_buffers(N):
    N = (N + 7) // 8 * 8
    R = 3
    x = rows(R, N, seed=N).cuda()
    y_buf = torch.full((R * N + 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    need = ela.load_library().attn_softmax_rows_workspace_bytes(R, N)
    ws = torch.full((need + 4096,), 0x5A, dtype=torch.uint8, device="cuda")
    ela.softmax_rows(x, out=y_buf[: R * N].view(R, N), workspace=ws[:need] if need else None)
    torch.cuda.synchronize()
    assert (y_buf[R * N:] == 7.0).all() and (ws[need:] == 0x5A).all()
    g = torch.ones(N, dtype=torch.bfloat16, device="cuda")
    if N <= 65536:
        ela.layernorm_rows(x, g, g, out=y_buf[: R * N].view(R, N))
        torch.cuda.synchronize()
        assert (y_buf[R * N:] == 7.0).all()

"""GPU parity of the forward with part of its exp2s on the FMA pipes.

The library is built a second time with ELS_EXP2_POLY_PER32=8: in every 32
scores of a row, the first eight exponentials are evaluated by exp2_poly.h's
range reduction and polynomial (packed f32x2 arithmetic) instead of the
special-function unit, a quarter of them, the largest share the build offers.
The polynomial's own error is pinned on the host (test_exp2_poly.py); here the
whole kernel built with it meets the oracle at the parity tolerances on the
named workloads (sampled rows for the large ones), ragged lengths, both head
dimensions, the causal mask, the K/V split, the dynamic schedule and a
negative scale.
"""
import pytest
import torch

import exact_long_sequence_gb300 as ela
from exact_long_sequence_gb300 import workloads
from test_parity import compare

pytestmark = pytest.mark.gpu

PER32 = 8


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from exact_long_sequence_gb300 import _build

    path = _build.build_variant(f"exp2poly{PER32}", {"ELS_EXP2_POLY_PER32": PER32})
    return ela.load_library(path)


def run(lib, q, k, v, causal, scale=None, split=True):
    dev = torch.device("cuda")
    o = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device=dev)
    ela.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=scale, out=o, lse=lse, split=split, lib=lib)
    assert ela.last_device_error(lib=lib) == ela.ATTN_OK
    assert not torch.isnan(o).any() and not torch.isnan(lse).any()
    return o, lse


@pytest.mark.parametrize("name,rows_per_head", [("b1h1n256d64", None), ("b1h8n4096d64_causal", None),
                                                ("b1h16n16384d128", 256), ("b1h8n65536d128_causal", 128),
                                                ("b4h32n8192d128_causal_spiky", 32)])
def test_offload_workload_parity(lib, oracle_mod, name, rows_per_head):
    w = workloads.WORKLOADS[name]
    q, k, v = workloads.workload_inputs(w)
    o, lse = run(lib, q, k, v, w.causal, w.scale)
    rows = None if rows_per_head is None else workloads.sample_rows(w.B * w.H, w.N, rows_per_head, w.seed)
    compare(o, lse, q, k, v, w.causal, w.scale, rows, oracle_mod, f"offload {name}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 17, 129, 257, 1000])
def test_offload_ragged_lengths(lib, oracle_mod, N, causal, d):
    q, k, v = workloads.make_inputs(1, 3, N, d, seed=500 + N)
    o, lse = run(lib, q, k, v, causal)
    compare(o, lse, q, k, v, causal, ela.default_scale(d), None, oracle_mod, f"offload N={N} d={d} causal={causal}")


def test_offload_negative_scale_and_single_kernel(lib, oracle_mod):
    q, k, v = workloads.make_inputs(2, 2, 700, 128, seed=510)
    o, lse = run(lib, q, k, v, True, scale=-0.2, split=False)
    compare(o, lse, q, k, v, True, -0.2, None, oracle_mod, "offload negative scale")

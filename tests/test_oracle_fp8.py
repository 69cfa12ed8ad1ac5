"""Pins for the FP8 (E4M3) side of the oracle: the exact decoder and the forward
on decoded inputs.

The decoder is checked against torch's own float8_e4m3fn conversion (an
independent implementation of the same OCP format) over all 256 codes, and
against values the format's definition fixes.  The FP8 forward is checked
against the pinned bf16 forward: every E4M3 value is also a bf16 value, so on
the same decoded inputs the two must agree exactly.
"""
import math

import numpy as np
import pytest
import torch

from exact_long_sequence_gb300 import workloads


def test_decoder_matches_torch_on_every_code(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    got = oracle_mod.decode_e4m3(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert nan.sum() == 2  # S.1111.111 for both signs
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    # signed zero included
    assert math.copysign(1.0, got[0x80]) == -1.0


def test_decoder_fixed_values_and_scale(oracle_mod):
    table = {0x38: 1.0, 0x7E: 448.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
             0x30: 0.5, 0x40: 2.0, 0x44: 3.0, 0xB8: -1.0, 0xFE: -448.0, 0x00: 0.0}
    codes = np.array(list(table), dtype=np.uint8)
    np.testing.assert_array_equal(oracle_mod.decode_e4m3(codes), np.array(list(table.values())))
    np.testing.assert_array_equal(oracle_mod.decode_e4m3(codes, 0.25), 0.25 * np.array(list(table.values())))


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_equals_bf16_forward_on_the_same_values(oracle_mod, causal):
    q8, k8, v8, _ = workloads.make_inputs_fp8(1, 2, 90, 32, seed=5)
    scales = (0.5, 2.0, 0.25)  # powers of two: the scaled values stay exact in bf16
    as_bf16 = [torch.from_numpy(oracle_mod.decode_e4m3(x, s)).to(torch.bfloat16) for x, s in zip((q8, k8, v8), scales)]
    for t, x, s in zip(as_bf16, (q8, k8, v8), scales):
        np.testing.assert_array_equal(t.double().numpy(), oracle_mod.decode_e4m3(x, s))  # exact in bf16
    O1, L1 = oracle_mod.attention_rows(*as_bf16, causal, 0.3)
    O2, L2 = oracle_mod.attention_fp8(q8, k8, v8, causal, 0.3, scales=scales)
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(L1, L2)


def test_row_selection_of_the_double_forward(oracle_mod):
    rng = np.random.default_rng(6)
    q, k, v = (rng.standard_normal((2, 40, 8)) for _ in range(3))
    O, L = oracle_mod.attention_f64(q, k, v, True, 0.4)
    rows = np.array([[0, 7, 39], [3, 4, 20]])
    Os, Ls, P = oracle_mod.attention_rows_f64(q, k, v, True, 0.4, rows=rows, return_probs=True)
    for b in range(2):
        np.testing.assert_array_equal(Os[b], O[b, rows[b]])
        np.testing.assert_array_equal(Ls[b], L[b, rows[b]])
    np.testing.assert_allclose(P.sum(-1), 1.0, atol=1e-12)


def test_quantiser_round_trip():
    g = torch.Generator().manual_seed(7)
    x = torch.randn(4, 300, generator=g) * 3
    codes, scale = workloads.quantize_e4m3(x)
    assert codes.dtype == torch.uint8
    back = codes.view(torch.float8_e4m3fn).to(torch.float64) * scale
    assert abs(float(back.abs().max()) - float(x.abs().max())) <= 2 ** -4 * float(x.abs().max())
    normal = x.abs() / scale >= 2 ** -6
    rel = ((back - x.double()).abs() / x.double().abs())[normal]
    assert float(rel.max()) <= 2 ** -4 + 1e-7

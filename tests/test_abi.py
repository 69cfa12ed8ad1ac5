"""Host-side checks of the C ABI: the library builds, loads and exports every
declared symbol; the planner's arithmetic; argument validation. No GPU needed:
every call here either launches nothing or fails validation before touching a
device."""
import ctypes
import math
import os
import re

import pytest
import torch

import exact_long_sequence_gb300 as ela
from exact_long_sequence_gb300 import _build, workloads

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "exact_attn.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return ela.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(attn_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_binding_symbols():
    assert declared_functions() == sorted(ela.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    # the library links no oracle code
    syms = os.popen(f"nm -D --defined-only {ela.LIB_PATH}").read()
    assert "oracle" not in syms


def test_strerror_covers_every_status(lib):
    for s in range(7):
        assert lib.attn_strerror(s).decode() not in ("", "unknown status")
    assert lib.attn_strerror(99).decode() == "unknown status"


def plan(B, H, N, d, causal, sms=152):
    return ela.attn_plan(B, H, N, d, causal, num_sms=sms)


@pytest.mark.parametrize("name", sorted(workloads.WORKLOADS))
def test_plan_matches_workload_arithmetic(lib, name):
    w = workloads.WORKLOADS[name]
    p = plan(w.B, w.H, w.N, w.d, w.causal)
    assert (p["Br"], p["Bc"], p["q_tiles"], p["threads"], p["tmem_cols"]) == (128, 128, 2, 384, 512)
    units = w.B * w.H * math.ceil(math.ceil(w.N / 128) / 2)
    assert p["num_units"] == units and p["grid"] == min(units, 152)
    assert p["flops"] == pytest.approx(w.flops, rel=1e-12)
    assert p["io_bytes"] == pytest.approx(w.io_bytes, rel=1e-12)
    assert p["smem_bytes"] <= 232448 and 2 * p["smem_bytes"] > 233472  # one CTA per SM
    assert p["kv_stages"] == (5 if w.d == 128 else 8)
    assert 1 <= p["heads_per_group"] <= w.B * w.H
    # K/V streamed once per pair of query tiles (half as often when causal)
    nd = w.N * w.d
    u = math.ceil(w.N / 256)
    passes = 0.5 * (u + 1) if w.causal else u
    assert p["l2_bytes"] == pytest.approx(w.B * w.H * (2 * (2 * nd + 2 * nd * passes) + 4 * w.N), rel=1e-12)


def test_planner_io_optimum(lib):
    # d=128: TMEM (q*(Bc+d) <= 512) allows two resident 128-row tiles with Bc=128: the compiled tiling.
    p = plan(1, 16, 16384, 128, False)
    assert (p["io_opt_q_tiles"], p["io_opt_Bc"]) == (2, 128)
    assert p["io_opt_l2_bytes"] == pytest.approx(p["l2_bytes"])
    # d=64: more resident tiles would need Bc=64, whose S product cannot run at the full
    # tensor rate from shared memory: the optimum is the compiled tiling too.
    p = plan(1, 8, 4096, 64, True)
    assert (p["io_opt_q_tiles"], p["io_opt_Bc"]) == (2, 128)
    assert p["io_opt_l2_bytes"] == pytest.approx(p["l2_bytes"])


def test_plan_rejects_bad_shapes(lib):
    out = ela.AttnPlan()
    assert lib.attn_plan(1, 1, 128, 96, 0, 152, ctypes.byref(out)) == ela.ATTN_ERR_UNSUPPORTED
    assert lib.attn_plan(0, 1, 128, 64, 0, 152, ctypes.byref(out)) == ela.ATTN_ERR_INVALID_ARG
    assert lib.attn_plan(1, 1, 0, 64, 0, 152, ctypes.byref(out)) == ela.ATTN_ERR_INVALID_ARG
    assert lib.attn_plan(1 << 16, 1 << 10, 1 << 10, 64, 0, 152, ctypes.byref(out)) == ela.ATTN_ERR_INVALID_ARG
    assert lib.attn_plan(1, 1, 128, 64, 0, 152, None) == ela.ATTN_ERR_INVALID_ARG


def call_fwd(lib, q=0x1000, k=0x2000, v=0x3000, o=0x4000, lse=0x5000, B=1, H=1, N=128, d=64, causal=0, scale=0.125):
    return lib.attn_fwd(q, k, v, o, lse, B, H, N, d, causal, scale, None)


def test_fwd_argument_validation(lib):
    assert call_fwd(lib, q=None) == ela.ATTN_ERR_INVALID_ARG
    assert call_fwd(lib, lse=None) == ela.ATTN_ERR_INVALID_ARG
    assert call_fwd(lib, N=0) == ela.ATTN_ERR_INVALID_ARG
    assert call_fwd(lib, B=-1) == ela.ATTN_ERR_INVALID_ARG
    assert call_fwd(lib, B=1 << 12, H=1 << 12, N=1 << 8) == ela.ATTN_ERR_INVALID_ARG
    for bad in (float("nan"), float("inf"), float("-inf")):
        assert call_fwd(lib, scale=bad) == ela.ATTN_ERR_INVALID_ARG
    # any finite scale passes validation (negative: negated scores; zero: uniform weights)
    if not torch.cuda.is_available():
        for ok in (0.0, -0.125, -3.0):
            assert call_fwd(lib, scale=ok) in (ela.ATTN_ERR_NO_DEVICE, ela.ATTN_ERR_CUDA)
    assert call_fwd(lib, d=96) == ela.ATTN_ERR_UNSUPPORTED
    assert call_fwd(lib, d=256) == ela.ATTN_ERR_UNSUPPORTED
    assert call_fwd(lib, k=0x2008) == ela.ATTN_ERR_MISALIGNED
    assert call_fwd(lib, o=0x4004) == ela.ATTN_ERR_MISALIGNED
    assert call_fwd(lib, lse=0x5002) == ela.ATTN_ERR_MISALIGNED


def test_host_entry_validation_and_workspace_size(lib):
    assert lib.attn_fwd_host_workspace_bytes(1, 2, 100, 64) == 4 * ((1 * 2 * 100 * 64 * 2 + 255) // 256 * 256) + 800
    assert lib.attn_fwd_host_workspace_bytes(0, 2, 100, 64) == 0
    args = (0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 1, 1, 128, 64, 0, 0.125)
    assert lib.attn_fwd_host(*args, None, 1 << 20, None) == ela.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_host(*args, 0x6008, 1 << 20, None) == ela.ATTN_ERR_MISALIGNED
    assert lib.attn_fwd_host(*args, 0x6000, 16, None) == ela.ATTN_ERR_INVALID_ARG
    assert lib.attn_debug_wait_timeout(0, None) == ela.ATTN_ERR_INVALID_ARG
    assert lib.attn_debug_wait_timeout(11_000_000_000, None) == ela.ATTN_ERR_INVALID_ARG
    # the abort hook's limit: 1 us .. 1 s (checked before anything else, no device needed)
    assert lib.attn_debug_arm_timeout(0) == ela.ATTN_ERR_INVALID_ARG
    assert lib.attn_debug_arm_timeout(999) == ela.ATTN_ERR_INVALID_ARG
    assert lib.attn_debug_arm_timeout(1_000_000_001) == ela.ATTN_ERR_INVALID_ARG


def test_split_entry_validation(lib):
    """attn_fwd_split checks its tensor arguments like attn_fwd; its size query is 0 for invalid shapes."""
    for shape in ((0, 1, 128, 64), (1, 1, 0, 64), (1, 1, 128, 96), (1 << 16, 1 << 8, 1 << 8, 64)):
        assert lib.attn_fwd_split_workspace_bytes(*shape, 1) == 0
    args = (0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 1, 1, 128, 96, 0, 0.125)
    assert lib.attn_fwd_split(*args, None, 0, None) in (ela.ATTN_ERR_INVALID_ARG, ela.ATTN_ERR_UNSUPPORTED)
    args = (0x1000, 0x2008, 0x3000, 0x4000, 0x5000, 1, 1, 128, 64, 0, 0.125)
    assert lib.attn_fwd_split(*args, None, 0, None) == ela.ATTN_ERR_MISALIGNED


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_valid_call_without_gpu_reports_no_device(lib):
    assert call_fwd(lib) in (ela.ATTN_ERR_NO_DEVICE, ela.ATTN_ERR_CUDA)
    assert lib.attn_last_device_error(None) in (ela.ATTN_ERR_NO_DEVICE, ela.ATTN_ERR_CUDA)
    assert lib.attn_noalloc_last_device_error(None) in (ela.ATTN_ERR_NO_DEVICE, ela.ATTN_ERR_CUDA)
    assert lib.attn_fwd_noalloc(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 1, 1, 128, 64, 0, -0.125, None) in (
        ela.ATTN_ERR_NO_DEVICE, ela.ATTN_ERR_CUDA)


def test_python_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        ela.load_library(str(tmp_path / "missing.so"))


def test_package_does_not_import_the_oracle():
    src_dir = os.path.dirname(ela.__file__)
    for root, _, files in os.walk(src_dir):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".cpp", ".h")):
                text = open(os.path.join(root, f)).read()
                assert "import oracle" not in text and "from oracle" not in text and "attn_oracle" not in text, f


def test_fp8_entry_validation(lib):
    args = (0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 1, 1, 128)
    ws = (0x6000, 1 << 20, None)
    assert lib.attn_fwd_fp8(*args, 64, 0, 0.125, 1.0, 1.0, 1.0, *ws) == ela.ATTN_ERR_UNSUPPORTED
    for bad in ((0.0, 1.0, 1.0), (1.0, float("inf"), 1.0), (1.0, 1.0, -2.0)):
        assert lib.attn_fwd_fp8(*args, 128, 0, 0.125, *bad, *ws) == ela.ATTN_ERR_INVALID_ARG
    for bad in (0.0, -0.125):  # the FP8 kernel takes a positive score scale only
        assert lib.attn_fwd_fp8(*args, 128, 0, bad, 1.0, 1.0, 1.0, *ws) == ela.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_fp8(*args, 128, 0, 0.125, 1.0, 1.0, 1.0, None, 1 << 20, None) == ela.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_fp8(*args, 128, 0, 0.125, 1.0, 1.0, 1.0, 0x6000, 16, None) == ela.ATTN_ERR_INVALID_ARG
    # the transposed V codes (rows padded to 16), 256-byte aligned, then the schedule counter block
    assert lib.attn_fwd_fp8_workspace_bytes(2, 3, 100, 128) == (2 * 3 * 128 * 112 + 255) // 256 * 256 + 256


def test_row_ops_validation(lib):
    assert lib.attn_softmax_rows(None, 0x2000, 4, 64, None, 0, None) == ela.ATTN_ERR_INVALID_ARG
    assert lib.attn_softmax_rows(0x1000, 0x2000, 0, 64, None, 0, None) == ela.ATTN_ERR_INVALID_ARG
    assert lib.attn_softmax_rows(0x1000, 0x2000, 4, 60, None, 0, None) == ela.ATTN_ERR_UNSUPPORTED
    assert lib.attn_softmax_rows(0x1008, 0x2000, 4, 64, None, 0, None) == ela.ATTN_ERR_MISALIGNED
    # long rows need the segment workspace: R * ceil(N / 16384) (m, l) pairs of 8 bytes
    assert lib.attn_softmax_rows_workspace_bytes(3, 1 << 16) == 0
    assert lib.attn_softmax_rows_workspace_bytes(3, (1 << 16) + 8) == 3 * 5 * 8
    assert lib.attn_softmax_rows(0x1000, 0x2000, 3, (1 << 16) + 8, None, 0, None) == ela.ATTN_ERR_INVALID_ARG
    g, b = 0x3000, 0x4000
    assert lib.attn_layernorm_rows(0x1000, g, b, 0x2000, 4, (1 << 16) + 8, 1e-5, None) == ela.ATTN_ERR_UNSUPPORTED
    assert lib.attn_layernorm_rows(0x1000, g, b, 0x2000, 4, 64, -1.0, None) == ela.ATTN_ERR_INVALID_ARG
    assert lib.attn_layernorm_rows(0x1000, None, b, 0x2000, 4, 64, 1e-5, None) == ela.ATTN_ERR_INVALID_ARG
    assert lib.attn_layernorm_rows(0x1000, 0x3004, b, 0x2000, 4, 64, 1e-5, None) == ela.ATTN_ERR_MISALIGNED

"""GB300 (sm_103a) exact self-attention forward: Python binding of the C ABI.

This module only marshals arguments: every step of the computation runs in the
CUDA kernels of ``libexact_attn.so`` (see ``include/exact_attn.h``). PyTorch is
used for device memory and streams. There is no fallback: if the library is
not built, or no sm_103 GPU is present, the calls raise.

    import exact_long_sequence_gb300 as ela
    o, lse = ela.attn_fwd(q, k, v, causal=True)   # q, k, v: bf16 [B, H, N, d] on cuda

The operation is O = softmax(scale * Q K^T + mask) V with the per-row natural
log-sum-exp LSE, computed as the streaming tiled pass of "From Attention Graph
to FlashAttention - A Memory-Centric Compilation Approach in AICF", section 3.
"""
from __future__ import annotations

import ctypes
import math
import os

from . import workloads  # noqa: F401  (seeded synthetic inputs; no attention arithmetic)

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libexact_attn.so")

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_MISALIGNED = 3
ATTN_ERR_CUDA = 4
ATTN_ERR_TIMEOUT = 5
ATTN_ERR_NO_DEVICE = 6

# Every symbol include/exact_attn.h declares.
EXPORTED_SYMBOLS = (
    "attn_fwd",
    "attn_fwd_host",
    "attn_fwd_host_workspace_bytes",
    "attn_fwd_split",
    "attn_fwd_split_workspace_bytes",
    "attn_fwd_split_segments",
    "attn_fwd_split_choice",
    "attn_plan",
    "attn_last_device_error",
    "attn_last_cuda_error",
    "attn_strerror",
    "attn_debug_wait_timeout",
    "attn_debug_arm_timeout",
    "attn_fwd_noalloc",
    "attn_noalloc_last_device_error",
    "attn_bwd",
    "attn_bwd_workspace_bytes",
    "attn_fwd_fp8",
    "attn_fwd_fp8_workspace_bytes",
    "attn_softmax_rows",
    "attn_softmax_rows_workspace_bytes",
    "attn_layernorm_rows",
)


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str, lib=None):
        msg = f"{what}: status {status}"
        if lib is not None:
            msg += f" ({lib.attn_strerror(status).decode()})"
            if status == ATTN_ERR_CUDA:
                msg += f", cudaError {lib.attn_last_cuda_error()}"
        super().__init__(msg)
        self.status = status


class AttnPlan(ctypes.Structure):
    _fields_ = [
        ("Br", ctypes.c_int), ("Bc", ctypes.c_int), ("q_tiles", ctypes.c_int), ("kv_stages", ctypes.c_int),
        ("tmem_cols", ctypes.c_int), ("smem_bytes", ctypes.c_int), ("threads", ctypes.c_int),
        ("num_units", ctypes.c_int), ("grid", ctypes.c_int), ("heads_per_group", ctypes.c_int),
        ("flops", ctypes.c_double), ("io_bytes", ctypes.c_double), ("l2_bytes", ctypes.c_double),
        ("hbm_bytes", ctypes.c_double), ("io_opt_q_tiles", ctypes.c_int), ("io_opt_Bc", ctypes.c_int),
        ("io_opt_l2_bytes", ctypes.c_double), ("kv_in_flight_bytes", ctypes.c_double), ("l2_fit", ctypes.c_double),
    ]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


_lib = None


def load_library(path: str | None = None):
    """Load the CUDA library (built by ``__graft_entry__.build()``); raise if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(p)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
    lib.attn_fwd.restype = i
    lib.attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, ctypes.c_size_t, vp]
    lib.attn_fwd_host.restype = i
    lib.attn_fwd_host_workspace_bytes.argtypes = [i, i, i, i]
    lib.attn_fwd_host_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_fwd_split.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, ctypes.c_size_t, vp]
    lib.attn_fwd_split.restype = i
    lib.attn_fwd_split_workspace_bytes.argtypes = [i, i, i, i, i]
    lib.attn_fwd_split_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_fwd_split_segments.argtypes = [i, i, i, i, i]
    lib.attn_fwd_split_segments.restype = i
    ip = ctypes.POINTER(ctypes.c_int)
    lib.attn_fwd_split_choice.argtypes = [i, i, i, i, i, i, ip, ip, ip, ip]
    lib.attn_fwd_split_choice.restype = i
    lib.attn_plan.argtypes = [i, i, i, i, i, i, ctypes.POINTER(AttnPlan)]
    lib.attn_plan.restype = i
    lib.attn_last_device_error.argtypes = [vp]
    lib.attn_last_device_error.restype = i
    lib.attn_last_cuda_error.argtypes = []
    lib.attn_last_cuda_error.restype = i
    lib.attn_strerror.argtypes = [i]
    lib.attn_strerror.restype = ctypes.c_char_p
    lib.attn_debug_wait_timeout.argtypes = [ctypes.c_uint64, vp]
    lib.attn_debug_wait_timeout.restype = i
    lib.attn_debug_arm_timeout.argtypes = [ctypes.c_uint64]
    lib.attn_debug_arm_timeout.restype = i
    lib.attn_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
    lib.attn_fwd_noalloc.restype = i
    lib.attn_noalloc_last_device_error.argtypes = [vp]
    lib.attn_noalloc_last_device_error.restype = i
    lib.attn_bwd.argtypes = [vp] * 9 + [i, i, i, i, i, f, vp, ctypes.c_size_t, vp]
    lib.attn_bwd.restype = i
    lib.attn_bwd_workspace_bytes.argtypes = [i, i, i, i]
    lib.attn_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_fwd_fp8.argtypes = [vp] * 5 + [i, i, i, i, i, f, f, f, f, vp, ctypes.c_size_t, vp]
    lib.attn_fwd_fp8.restype = i
    lib.attn_fwd_fp8_workspace_bytes.argtypes = [i, i, i, i]
    lib.attn_fwd_fp8_workspace_bytes.restype = ctypes.c_size_t
    i64 = ctypes.c_int64
    lib.attn_softmax_rows.argtypes = [vp, vp, i64, i, vp, ctypes.c_size_t, vp]
    lib.attn_softmax_rows.restype = i
    lib.attn_softmax_rows_workspace_bytes.argtypes = [i64, i]
    lib.attn_softmax_rows_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_layernorm_rows.argtypes = [vp, vp, vp, vp, i64, i, f, vp]
    lib.attn_layernorm_rows.restype = i
    if path is None:
        _lib = lib
    return lib


def _check(status: int, what: str):
    if status != ATTN_OK:
        raise AttnError(status, what, _lib)


def default_scale(d: int) -> float:
    """1/sqrt(d), computed in double and rounded once to fp32."""
    import torch

    return float(torch.tensor(1.0 / math.sqrt(d), dtype=torch.float32).item())


def _stream_handle(stream):
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def split_workspace_bytes(B: int, H: int, N: int, d: int, causal: bool) -> int:
    """Device bytes attn_fwd_split needs for this shape on the current device (0: none)."""
    return int(load_library().attn_fwd_split_workspace_bytes(B, H, N, d, int(bool(causal))))


def split_choice(B: int, H: int, N: int, d: int, causal: bool, num_sms: int | None = None) -> dict:
    """The work split attn_fwd_split uses (host only): segments per split unit (1: none), the
    first split unit, the number of split units, and whether the dynamic schedule runs (a
    counter-zeroing kernel then precedes the attention kernel).  num_sms: the current device's
    by default."""
    import ctypes

    import torch

    if num_sms is None:
        num_sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    out = [ctypes.c_int(0) for _ in range(4)]
    st = load_library().attn_fwd_split_choice(B, H, N, d, int(bool(causal)), int(num_sms),
                                              *[ctypes.byref(x) for x in out])
    _check(st, "attn_fwd_split_choice")
    return {"segs": out[0].value, "first": out[1].value, "units": out[2].value, "dynamic": bool(out[3].value)}


def split_segments(B: int, H: int, N: int, d: int, causal: bool) -> int:
    """K/V segments per split unit attn_fwd_split chooses (1: no split; 0: invalid or no device)."""
    return int(load_library().attn_fwd_split_segments(B, H, N, d, int(bool(causal))))


def attn_fwd(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None, stream=None,
             split: bool = True, workspace=None, lib=None):
    """O, LSE = attention(q, k, v) on the GPU through the C ABI.

    q, k, v   : bf16 CUDA tensors [B, H, N, d], contiguous, d in {64, 128}
    out       : optional bf16 [B, H, N, d] output buffer; lse: optional fp32 [B, H, N]
    stream    : torch.cuda.Stream (default: the current stream); the call is asynchronous.
    split     : allow attn_fwd_split: the K/V split for problems with fewer work units than SMs,
                and the dynamic schedule for causal problems with more (False: always attn_fwd)
    workspace : optional uint8 CUDA tensor of at least split_workspace_bytes() bytes for the
                split (allocated here when needed and not given)
    lib       : a library handle from load_library(path) (a compile-time variant); default: the
                library built in-tree
    """
    import torch

    lib = lib or load_library()
    if q.dim() != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must share a [B, H, N, d] shape")
    for t in (q, k, v):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous bf16 CUDA tensors")
    B, H, N, d = q.shape
    if scale is None:
        scale = default_scale(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor shaped like q")
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, H, N] tensor")
    with torch.cuda.device(q.device):
        need = int(lib.attn_fwd_split_workspace_bytes(B, H, N, d, int(bool(causal)))) if split else 0
        if need == 0:
            st = lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                              B, H, N, d, int(bool(causal)), float(scale), _stream_handle(stream))
            _check(st, "attn_fwd")
            return out, lse
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
            if stream is not None:
                workspace.record_stream(stream)
        if workspace.dtype != torch.uint8 or not workspace.is_cuda or workspace.numel() < need:
            raise ValueError(f"workspace must be a uint8 CUDA tensor of at least {need} bytes")
        st = lib.attn_fwd_split(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                B, H, N, d, int(bool(causal)), float(scale), workspace.data_ptr(),
                                workspace.numel(), _stream_handle(stream))
    _check(st, "attn_fwd_split")
    return out, lse


def attn_bwd(q, k, v, o, lse, do, causal: bool = False, scale: float | None = None, workspace=None, stream=None):
    """dQ, dK, dV = gradients of attn_fwd for the upstream gradient `do`.

    q, k, v, o, do : bf16 CUDA tensors [B, H, N, d] (o, lse from attn_fwd on the same inputs)
    lse            : fp32 [B, H, N]
    """
    import torch

    lib = load_library()
    for t in (q, k, v, o, do):
        if t.shape != q.shape or t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v, o, do must be contiguous bf16 CUDA tensors of one [B, H, N, d] shape")
    B, H, N, d = q.shape
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, H, N] tensor")
    if scale is None:
        scale = default_scale(d)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    need = lib.attn_bwd_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        st = lib.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                          dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, int(bool(causal)), float(scale),
                          workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(st, "attn_bwd")
    return dq, dk, dv


def attn_fwd_fp8(q8, k8, v8, scales, causal: bool = False, scale: float | None = None, out=None, lse=None,
                 workspace=None, stream=None, lib=None):
    """FP8 forward: q8, k8, v8 are uint8 CUDA tensors [B, H, N, d] of E4M3 codes and
    `scales` = (q_scale, k_scale, v_scale), the real inputs being scale * e4m3(code).
    Returns (o bf16 [B, H, N, d], lse fp32 [B, H, N]).  d must be 128.  `lib`: a library handle
    from load_library(path) (a compile-time variant); default: the library built in-tree."""
    import torch

    lib = lib or load_library()
    for t in (q8, k8, v8):
        if t.shape != q8.shape or t.dtype != torch.uint8 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q8, k8, v8 must be contiguous uint8 (E4M3 code) CUDA tensors of one [B, H, N, d] shape")
    B, H, N, d = q8.shape
    if scale is None:
        scale = default_scale(d)
    if out is None:
        out = torch.empty(q8.shape, dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    need = lib.attn_fwd_fp8_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q8.device)
    sq, sk, sv = (float(x) for x in scales)
    with torch.cuda.device(q8.device):
        st = lib.attn_fwd_fp8(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, N, d,
                              int(bool(causal)), float(scale), sq, sk, sv, workspace.data_ptr(),
                              workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(st, "attn_fwd_fp8")
    return out, lse


def softmax_rows(x, out=None, workspace=None, stream=None):
    """Row softmax over the last axis of a contiguous bf16 CUDA tensor (last axis a multiple of 8)."""
    import torch

    lib = load_library()
    if x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous bf16 CUDA tensor")
    N = x.shape[-1]
    R = x.numel() // N
    if out is None:
        out = torch.empty_like(x)
    need = lib.attn_softmax_rows_workspace_bytes(R, N)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    with torch.cuda.device(x.device):
        st = lib.attn_softmax_rows(x.data_ptr(), out.data_ptr(), R, N,
                                   workspace.data_ptr() if workspace is not None else None,
                                   workspace.numel() if workspace is not None else 0, _stream_handle(stream))
    _check(st, "attn_softmax_rows")
    return out


def layernorm_rows(x, gamma, beta, eps: float = 1e-5, out=None, stream=None):
    """Layer normalisation over the last axis (bf16 x, gamma, beta on CUDA; last axis a multiple of 8, <= 65536)."""
    import torch

    lib = load_library()
    for t in (x, gamma, beta):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("x, gamma, beta must be contiguous bf16 CUDA tensors")
    N = x.shape[-1]
    if gamma.shape != (N,) or beta.shape != (N,):
        raise ValueError("gamma and beta must have the row length")
    if out is None:
        out = torch.empty_like(x)
    with torch.cuda.device(x.device):
        st = lib.attn_layernorm_rows(x.data_ptr(), gamma.data_ptr(), beta.data_ptr(), out.data_ptr(),
                                     x.numel() // N, N, float(eps), _stream_handle(stream))
    _check(st, "attn_layernorm_rows")
    return out


def attn_fwd_noalloc(q, k, v, out, lse, causal: bool = False, scale: float | None = None, stream=None):
    """attn_fwd through the entry point that never allocates device memory.

    For callers that cannot let the library cudaMalloc (their own pool owns all
    of device memory, or their path cannot take cudaMalloc's implicit device
    synchronisation): the kernel's error word lives in a fixed array compiled
    into the library instead. The caller passes the outputs `out` (bf16, shaped
    like q) and `lse` (fp32 [B, H, N]); calls that overlap on the GPU race on
    the shared word, so serialise them.
    """
    lib = load_library()
    B, H, N, d = q.shape
    if scale is None:
        scale = default_scale(d)
    for t in (q, k, v, out):
        if t.shape != q.shape or not t.is_contiguous():
            raise ValueError("q, k, v, out must be contiguous tensors of one [B, H, N, d] shape")
    if lse.shape != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous [B, H, N] tensor")
    st = lib.attn_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                              B, H, N, d, int(bool(causal)), float(scale), _stream_handle(stream))
    _check(st, "attn_fwd_noalloc")
    return out, lse


def attn_fwd_host(q_h, k_h, v_h, causal: bool = False, scale: float | None = None, out_h=None, lse_h=None,
                  workspace=None, stream=None):
    """Same operation on HOST tensors (pin them for asynchronous copies): the library
    copies Q, K, V in, runs the kernel and copies O, LSE out on `stream`. Synchronise the
    stream before reading the outputs."""
    import torch

    lib = load_library()
    B, H, N, d = q_h.shape
    if scale is None:
        scale = default_scale(d)
    if out_h is None:
        out_h = torch.empty_like(q_h, pin_memory=q_h.is_pinned())
    if lse_h is None:
        lse_h = torch.empty((B, H, N), dtype=torch.float32, pin_memory=q_h.is_pinned())
    need = lib.attn_fwd_host_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device="cuda")
    st = lib.attn_fwd_host(q_h.data_ptr(), k_h.data_ptr(), v_h.data_ptr(), out_h.data_ptr(), lse_h.data_ptr(),
                           B, H, N, d, int(bool(causal)), float(scale), workspace.data_ptr(),
                           workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(st, "attn_fwd_host")
    return out_h, lse_h


def host_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(load_library().attn_fwd_host_workspace_bytes(B, H, N, d))


def attn_plan(B: int, H: int, N: int, d: int, causal: bool, num_sms: int = 0) -> dict:
    """The planner's tiling for a shape (host only; num_sms=0 asks the current GPU)."""
    lib = load_library()
    plan = AttnPlan()
    _check(lib.attn_plan(B, H, N, d, int(bool(causal)), num_sms, ctypes.byref(plan)), "attn_plan")
    return plan.as_dict()


def last_device_error(stream=None, lib=None) -> int:
    """Synchronise `stream` and return (and clear) the kernel error status."""
    return (lib or load_library()).attn_last_device_error(_stream_handle(stream))


def debug_wait_timeout(timeout_ns: int, stream=None) -> int:
    """Launch the bounded-wait test kernel (waits on a barrier nobody arrives on)."""
    return load_library().attn_debug_wait_timeout(int(timeout_ns), _stream_handle(stream))


def debug_arm_timeout(timeout_ns: int) -> int:
    """Arm the one-shot abort hook: the next forward launch runs with this wait limit and
    withholds one of CTA 0's query-tile copies, so its wait runs out (test use only)."""
    return load_library().attn_debug_arm_timeout(int(timeout_ns))


def noalloc_last_device_error(stream=None) -> int:
    """Synchronise `stream` and return (and clear) attn_fwd_noalloc's error status."""
    return load_library().attn_noalloc_last_device_error(_stream_handle(stream))

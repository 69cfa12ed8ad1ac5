"""fp64 CPU oracle for exact self-attention forward (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg use this package. The CUDA library never imports, links or calls it, and
it shares no code with it: the arithmetic lives in ``attn_oracle.c`` (plain C,
fp64), which follows the attention graph of "From Attention Graph to
FlashAttention - A Memory-Centric Compilation Approach in AICF", section 1:
Scores = Q x K^T, Mask, Softmax, Output = Scores x V.

Every function here is pinned by ``tests/test_oracle.py`` against closed forms
and invariants of that definition, not against itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into a shared library with gcc; return its path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        # -ffp-contract=off: keep every product and sum a separate, correctly
        # rounded fp64 operation, the same on x86 and Arm.
        cmd = ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared",
               "-pthread", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _open(path: str):
    lib = ctypes.CDLL(path)
    lib.oracle_attn_rows.restype = ctypes.c_int
    lib.oracle_attn_rows.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_double,
        ctypes.c_void_p, ctypes.c_int64,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
    ]
    dp = ctypes.POINTER(ctypes.c_double)
    lib.oracle_attn_f64.restype = ctypes.c_int
    lib.oracle_attn_f64.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int64] * 3 + [ctypes.c_int, ctypes.c_double,
                                                                                     ctypes.c_void_p, ctypes.c_void_p]
    lib.oracle_attn_rows_f64.restype = ctypes.c_int
    lib.oracle_attn_rows_f64.argtypes = lib.oracle_attn_rows.argtypes
    lib.oracle_decode_e4m3.restype = ctypes.c_int
    lib.oracle_decode_e4m3.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p]
    lib.oracle_softmax_rows.restype = ctypes.c_int
    lib.oracle_softmax_rows.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
    lib.oracle_layernorm_rows.restype = ctypes.c_int
    lib.oracle_layernorm_rows.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int64, ctypes.c_int64, ctypes.c_double,
                                                                   ctypes.c_void_p]
    lib.oracle_attn_bwd_f64.restype = ctypes.c_int
    lib.oracle_attn_bwd_f64.argtypes = ([ctypes.c_void_p] * 4 + [ctypes.c_int64] * 3 + [ctypes.c_int, ctypes.c_double]
                                        + [ctypes.c_void_p] * 3 + [ctypes.c_int])
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _open(build())
    return _lib


def _as_bf16_bits(x) -> np.ndarray:
    """Accept a torch bf16 tensor (any device) or a numpy uint16 array of bf16 bits."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("numpy input must hold bf16 bit patterns as uint16")
        return np.ascontiguousarray(x)
    import torch

    if x.dtype != torch.bfloat16:
        raise TypeError("oracle inputs are bf16 tensors")
    return x.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def attention_rows(q, k, v, causal: bool, scale: float, rows=None, nthreads: int | None = None,
                   return_probs: bool = False, _lib_handle=None):
    """Exact attention for selected query rows, in fp64.

    q, k, v : [B, H, N, d] (or [BH, N, d]) bf16 inputs.
    scale   : the softmax scale; it is used as given (pass the fp32 value the
              GPU receives, widened to double).
    rows    : None for every row, or an int array [B*H, R] of query positions.
    Returns (O [BH, R, d] float64, LSE [BH, R] float64[, P [BH, R, N]]).
    """
    qb, kb, vb = _as_bf16_bits(q), _as_bf16_bits(k), _as_bf16_bits(v)
    if qb.shape != kb.shape or qb.shape != vb.shape or qb.ndim not in (3, 4):
        raise ValueError("q, k, v must share a [B,H,N,d] or [BH,N,d] shape")
    N, d = qb.shape[-2], qb.shape[-1]
    BH = int(np.prod(qb.shape[:-2]))
    if rows is None:
        R = N
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(BH, -1))
        R = rows_arr.shape[1]
    O = np.empty((BH, R, d), dtype=np.float64)
    LSE = np.empty((BH, R), dtype=np.float64)
    P = np.empty((BH, R, N), dtype=np.float64) if return_probs else None
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    lib = _lib_handle if _lib_handle is not None else _load()
    rc = lib.oracle_attn_rows(
        qb.ctypes.data, kb.ctypes.data, vb.ctypes.data, BH, N, d, int(bool(causal)), float(scale),
        rows_arr.ctypes.data if rows_arr is not None else None, R,
        O.ctypes.data, LSE.ctypes.data, P.ctypes.data if P is not None else None, int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_attn_rows failed with status {rc}")
    return (O, LSE, P) if return_probs else (O, LSE)


def _as_f64(x) -> np.ndarray:
    """bf16 torch tensors are decoded exactly; float arrays are taken as given."""
    if isinstance(x, np.ndarray):
        return np.ascontiguousarray(x, dtype=np.float64)
    import torch

    return np.ascontiguousarray(x.detach().to("cpu").to(torch.float64).numpy())


def attention_f64(q, k, v, causal: bool, scale: float, _lib_handle=None):
    """Forward on double inputs, every row: (O [BH, N, d], LSE [BH, N])."""
    qd, kd, vd = _as_f64(q), _as_f64(k), _as_f64(v)
    N, d = qd.shape[-2], qd.shape[-1]
    BH = int(np.prod(qd.shape[:-2]))
    O = np.empty((BH, N, d))
    LSE = np.empty((BH, N))
    lib = _lib_handle if _lib_handle is not None else _load()
    rc = lib.oracle_attn_f64(qd.ctypes.data, kd.ctypes.data, vd.ctypes.data, BH, N, d, int(bool(causal)),
                             float(scale), O.ctypes.data, LSE.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_attn_f64 failed with status {rc}")
    return O, LSE


def attention_rows_f64(q, k, v, causal: bool, scale: float, rows=None, nthreads: int | None = None,
                       return_probs: bool = False, _lib_handle=None):
    """attention_rows on double inputs (float arrays are used as given)."""
    qd, kd, vd = _as_f64(q), _as_f64(k), _as_f64(v)
    N, d = qd.shape[-2], qd.shape[-1]
    BH = int(np.prod(qd.shape[:-2]))
    if rows is None:
        R, rows_arr = N, None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(BH, -1))
        R = rows_arr.shape[1]
    O = np.empty((BH, R, d))
    LSE = np.empty((BH, R))
    P = np.empty((BH, R, N)) if return_probs else None
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    lib = _lib_handle if _lib_handle is not None else _load()
    rc = lib.oracle_attn_rows_f64(qd.ctypes.data, kd.ctypes.data, vd.ctypes.data, BH, N, d, int(bool(causal)),
                                  float(scale), rows_arr.ctypes.data if rows_arr is not None else None, R,
                                  O.ctypes.data, LSE.ctypes.data, P.ctypes.data if P is not None else None,
                                  int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_attn_rows_f64 failed with status {rc}")
    return (O, LSE, P) if return_probs else (O, LSE)


def decode_e4m3(codes, scale: float = 1.0, _lib_handle=None) -> np.ndarray:
    """scale * value of each E4M3 code (uint8 array or tensor), exactly, as float64."""
    if not isinstance(codes, np.ndarray):
        codes = codes.detach().to("cpu").contiguous().view(-1).numpy().view(np.uint8).reshape(tuple(codes.shape))
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    lib = _lib_handle if _lib_handle is not None else _load()
    rc = lib.oracle_decode_e4m3(c.ctypes.data, c.size, float(scale), out.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_decode_e4m3 failed with status {rc}")
    return out


def attention_fp8(q8, k8, v8, causal: bool, scale: float, scales=(1.0, 1.0, 1.0), rows=None,
                  nthreads: int | None = None, return_probs: bool = False, _lib_handle=None):
    """Forward for E4M3 inputs: Q = scales[0] * e4m3(q8), likewise K and V; then the
    same graph as attention_rows on the decoded values."""
    q, k, v = (decode_e4m3(x, s_, _lib_handle=_lib_handle) for x, s_ in zip((q8, k8, v8), scales))
    return attention_rows_f64(q, k, v, causal, scale, rows=rows, nthreads=nthreads, return_probs=return_probs,
                              _lib_handle=_lib_handle)


def softmax_rows(x, _lib_handle=None) -> np.ndarray:
    """Row softmax over the last axis (bf16 tensors decoded exactly; float arrays as given)."""
    xd = _as_f64(x)
    N = xd.shape[-1]
    R = xd.size // N
    y = np.empty(xd.shape)
    lib = _lib_handle if _lib_handle is not None else _load()
    rc = lib.oracle_softmax_rows(xd.ctypes.data, R, N, y.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_softmax_rows failed with status {rc}")
    return y


def layernorm_rows(x, gamma, beta, eps: float, _lib_handle=None) -> np.ndarray:
    """Layer normalisation over the last axis with per-column gamma, beta."""
    xd, gd, bd = _as_f64(x), _as_f64(gamma), _as_f64(beta)
    N = xd.shape[-1]
    R = xd.size // N
    if gd.shape != (N,) or bd.shape != (N,):
        raise ValueError("gamma and beta must have the row length")
    y = np.empty(xd.shape)
    lib = _lib_handle if _lib_handle is not None else _load()
    rc = lib.oracle_layernorm_rows(xd.ctypes.data, gd.ctypes.data, bd.ctypes.data, R, N, float(eps), y.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_layernorm_rows failed with status {rc}")
    return y


def attention_bwd(q, k, v, do, causal: bool, scale: float, nthreads: int | None = None, _lib_handle=None):
    """Backward for upstream gradient dO: (dQ, dK, dV), each [BH, N, d] float64.
    bf16 tensors are decoded exactly; float arrays are used as given."""
    qd, kd, vd, dod = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(do)
    N, d = qd.shape[-2], qd.shape[-1]
    BH = int(np.prod(qd.shape[:-2]))
    dQ, dK, dV = (np.empty((BH, N, d)) for _ in range(3))
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    lib = _lib_handle if _lib_handle is not None else _load()
    rc = lib.oracle_attn_bwd_f64(qd.ctypes.data, kd.ctypes.data, vd.ctypes.data, dod.ctypes.data, BH, N, d,
                                 int(bool(causal)), float(scale), dQ.ctypes.data, dK.ctypes.data, dV.ctypes.data,
                                 int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_attn_bwd_f64 failed with status {rc}")
    return dQ, dK, dV


class OracleBuild:
    """The same Python interface over another build of the C source (used by the
    mutation tests, which compile deliberately broken copies of the oracle)."""

    def __init__(self, lib_path: str):
        self._lib = _open(lib_path)

    def attention_rows(self, *args, **kwargs):
        return attention_rows(*args, _lib_handle=self._lib, **kwargs)

    def attention_f64(self, *args, **kwargs):
        return attention_f64(*args, _lib_handle=self._lib, **kwargs)

    def attention_bwd(self, *args, **kwargs):
        return attention_bwd(*args, _lib_handle=self._lib, **kwargs)

    def attention_rows_f64(self, *args, **kwargs):
        return attention_rows_f64(*args, _lib_handle=self._lib, **kwargs)

    def decode_e4m3(self, *args, **kwargs):
        return decode_e4m3(*args, _lib_handle=self._lib, **kwargs)

    def attention_fp8(self, *args, **kwargs):
        return attention_fp8(*args, _lib_handle=self._lib, **kwargs)

    def softmax_rows(self, *args, **kwargs):
        return softmax_rows(*args, _lib_handle=self._lib, **kwargs)

    def layernorm_rows(self, *args, **kwargs):
        return layernorm_rows(*args, _lib_handle=self._lib, **kwargs)

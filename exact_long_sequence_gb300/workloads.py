"""Seeded synthetic attention inputs and the named workloads.

This module draws random numbers and nothing else: it holds none of the
attention arithmetic, so both the CUDA path and the fp64 oracle can take their
inputs from it. The pages measure on no public dataset; every workload here is
synthetic by definition, with the shapes, masks and value distributions listed
below.

Draw recipe (one ``torch.Generator('cpu')`` per workload, seeded):
  Q, K, V are drawn in that order as fp32 ``[B, H, N, d]`` tensors, N(0, 1) via
  ``torch.randn`` or U(-1, 1) via ``torch.rand * 2 - 1``. The softmax-stability
  stress workload then draws a Bernoulli(0.01) mask for Q and then one for K
  (``torch.rand < 0.01``) and multiplies those entries by 10. Finally each
  tensor is rounded to bf16 (round to nearest even).

Sampled query rows for the large workloads come from a second generator seeded
with ``1000 + seed``: per (b, h), ``torch.randperm(N)[:R]``, sorted.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    seed: int
    qk_dist: str = "normal"      # "normal" or "normal_spiky" (1% of entries x10)
    v_dist: str = "normal"       # "normal" or "uniform" (U(-1,1))
    oracle_rows: int | None = None  # None: every query row is checked

    @property
    def scale(self) -> float:
        """1/sqrt(d), computed in double and rounded once to fp32."""
        return float(torch.tensor(1.0 / math.sqrt(self.d), dtype=torch.float32).item())

    @property
    def flops(self) -> float:
        """Two GEMMs, 4*B*H*N^2*d; the causal mask halves it (the usual count)."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    @property
    def io_bytes(self) -> int:
        """The Theta(N*d) I/O bound: bf16 Q, K, V read once, bf16 O and fp32 LSE written once."""
        return 2 * 4 * self.B * self.H * self.N * self.d + 4 * self.B * self.H * self.N


WORKLOADS = {
    "b1h1n256d64": Workload("b1h1n256d64", 1, 1, 256, 64, False, 0),
    "b1h8n4096d64_causal": Workload("b1h8n4096d64_causal", 1, 8, 4096, 64, True, 1),
    "b1h16n16384d128": Workload("b1h16n16384d128", 1, 16, 16384, 128, False, 2, oracle_rows=1024),
    "b1h8n65536d128_causal": Workload("b1h8n65536d128_causal", 1, 8, 65536, 128, True, 3, oracle_rows=512),
    "b4h32n8192d128_causal_spiky": Workload("b4h32n8192d128_causal_spiky", 4, 32, 8192, 128, True, 4,
                                            qk_dist="normal_spiky", v_dist="uniform", oracle_rows=256),
}
# The long-sequence, tall-and-skinny case that throughput is quoted on.
HEADLINE = "b1h16n16384d128"


def _draw(B: int, H: int, N: int, d: int, seed: int, qk_dist: str, v_dist: str):
    """The fp32 draws of the recipe above, before any rounding."""
    g = torch.Generator("cpu").manual_seed(seed)
    shape = (B, H, N, d)
    q = torch.randn(shape, generator=g)
    k = torch.randn(shape, generator=g)
    if v_dist == "normal":
        v = torch.randn(shape, generator=g)
    elif v_dist == "uniform":
        v = torch.rand(shape, generator=g) * 2 - 1
    else:
        raise ValueError(v_dist)
    if qk_dist == "normal_spiky":
        mq = torch.rand(shape, generator=g) < 0.01
        mk = torch.rand(shape, generator=g) < 0.01
        q = torch.where(mq, q * 10, q)
        k = torch.where(mk, k * 10, k)
    elif qk_dist != "normal":
        raise ValueError(qk_dist)
    return q, k, v


def make_inputs(B: int, H: int, N: int, d: int, seed: int, qk_dist: str = "normal",
                v_dist: str = "normal"):
    """Return bf16 CPU tensors (Q, K, V), each [B, H, N, d], by the recipe above."""
    q, k, v = _draw(B, H, N, d, seed, qk_dist, v_dist)
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


E4M3_MAX = 448.0  # largest finite E4M3 value


def quantize_e4m3(x: torch.Tensor):
    """Per-tensor E4M3 quantisation of an fp32 tensor: (codes as uint8, scale) with
    scale = max|x| / 448, so that x ~= scale * e4m3(codes).  Rounding is torch's
    float8_e4m3fn conversion (round to nearest even, saturating at 448)."""
    amax = float(x.abs().max())
    scale = amax / E4M3_MAX if amax > 0 else 1.0
    codes = (x / scale).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.contiguous(), scale


def make_inputs_fp8(B: int, H: int, N: int, d: int, seed: int, qk_dist: str = "normal",
                    v_dist: str = "normal"):
    """The same draws as make_inputs, quantised per tensor to E4M3: returns
    (q8, k8, v8, (q_scale, k_scale, v_scale)) with uint8 code tensors [B, H, N, d]."""
    q, k, v = _draw(B, H, N, d, seed, qk_dist, v_dist)
    (q8, sq), (k8, sk), (v8, sv) = (quantize_e4m3(t) for t in (q, k, v))
    return q8, k8, v8, (sq, sk, sv)


def workload_inputs(w: Workload):
    return make_inputs(w.B, w.H, w.N, w.d, w.seed, w.qk_dist, w.v_dist)


def sample_rows(BH: int, N: int, R: int, seed: int) -> torch.Tensor:
    """[BH, R] int64 sorted query positions, per (b, h) a random R-subset of range(N)."""
    g = torch.Generator("cpu").manual_seed(1000 + seed)
    R = min(R, N)
    out = torch.empty((BH, R), dtype=torch.int64)
    for bh in range(BH):
        out[bh] = torch.sort(torch.randperm(N, generator=g)[:R]).values
    return out


def workload_rows(w: Workload):
    """Rows the oracle checks for a workload: None means all of them."""
    if w.oracle_rows is None:
        return None
    return sample_rows(w.B * w.H, w.N, w.oracle_rows, w.seed)


# Standalone streaming row operations: (R rows, N elements per row), bf16, seeded
# normal inputs (softmax: N(0, 3^2); layer normalisation: N(3, 1) with gamma
# ~ 1 + 0.2 N(0, 1) and beta ~ 0.3 N(0, 1)).  Sized well above L2 so that the
# rate measured is the HBM rate.
ROW_WORKLOADS = {
    "softmax_r16384_n16384": ("softmax", 16384, 16384),      # attention-score-shaped rows, 512 MiB each way
    "softmax_r64_n1048576": ("softmax", 64, 1 << 20),        # million-element rows: the segmented path
    "layernorm_r65536_n8192": ("layernorm", 65536, 8192),    # 1 GiB each way
}


def row_inputs(kind: str, R: int, N: int, seed: int = 0, device="cpu"):
    """Seeded inputs of a row workload: x, or (x, gamma, beta) for layer normalisation."""
    g = torch.Generator(device=device).manual_seed(seed)
    if kind == "softmax":
        return (torch.randn(R, N, generator=g, device=device) * 3).to(torch.bfloat16)
    x = (torch.randn(R, N, generator=g, device=device) + 3).to(torch.bfloat16)
    gamma = (1 + 0.2 * torch.randn(N, generator=g, device=device)).to(torch.bfloat16)
    beta = (0.3 * torch.randn(N, generator=g, device=device)).to(torch.bfloat16)
    return x, gamma, beta

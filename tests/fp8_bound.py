"""Error bounds of the FP8 forward's output, shared by its GPU parity test and its CPU model.

Both come from E4M3 rounding of P before the second product.  With P the
oracle's exact probabilities of one query row:

  loose    |dO_c| <= 2^-4 sum_j P_j |v_jc| + 2^-10 sum_j |v_jc| max_j P_j + 2^-8 |O_c| + 1e-6
  per-term |dO_c| <= max_j P_j sum_j e_j |v_jc| + 2^-8 |O_c| + 1e-6,
           e_j = 2^-4 p_j where p_j = P_j / max_j P_j >= 2^-6 (E4M3's normal range),
           e_j = min(p_j, 2^-10) below it (a term there moves by at most 2^-10, or
           rounds to zero).

p_j is the kernel's term with its reference maximum at the row maximum, the
worst case: a stale reference scales every term up by the same power of two,
which leaves a normal term's relative error at 2^-4 and can only lift a term out
of the subnormal range.  The 2^-8 |O| and 1e-6 terms cover the bf16 output and
the fp32 sums.  Both bounds hold only while every term stays inside E4M3's
range (at most 448): the kernel's stale-maximum threshold keeps terms at most
2^8.  The loose bound charges every key 2^-10, so it grows with the row length;
the per-term one does not.
"""
import numpy as np


def fp8_output_bounds(P, vabs, O):
    """P: [..., R, N] exact probabilities; vabs: [..., N, d] |decoded V|; O: [..., R, d] exact output.
    Returns (loose, per_term), each shaped like O."""
    pmax = P.max(-1, keepdims=True)
    loose = (2.0 ** -4 * P @ vabs + 2.0 ** -10 * vabs.sum(-2)[..., None, :] * pmax
             + 2.0 ** -8 * np.abs(O) + 1e-6)
    p = P / pmax
    e = np.where(p >= 2.0 ** -6, 2.0 ** -4 * p, np.minimum(p, 2.0 ** -10))
    per_term = (e @ vabs) * pmax + 2.0 ** -8 * np.abs(O) + 1e-6
    return loose, per_term


# Row offsets (log2 units) of the near-ceiling case: the second key tile's scores sit this far
# above the first tile's, which fixes the kernel's reference maximum.  Up to 8 the reference stays
# stale and the terms reach 2^8 = 256 (E4M3's largest finite value is 448); above 8 it moves.
NEAR_CEILING_OFFSETS = (6.0, 6.5, 7.0, 7.5, 8.0, 9.0, 10.0, 12.0)


def near_ceiling_inputs(seed: int = 5):
    """E4M3 codes (q8, k8, v8) [1, 1, 256, 128], scales and the score scale of the near-ceiling case.

    With scale = ln 2 and unit Q and K scales, the scaled score in log2 units is q . k.  Q row r
    holds the offset delta_r (cycling through NEAR_CEILING_OFFSETS) in its first component and zeros
    elsewhere.  Keys 0-127 are zero, so the first tile's scores are 0; keys 128-255 hold 1 (even)
    or 1/2 (odd) in their first component, so the second tile's scores are delta_r and delta_r / 2.
    V holds codes of magnitude 352 to 448 with random signs, scaled by 1/448."""
    import torch

    N, d = 256, 128
    g = torch.Generator().manual_seed(seed)
    deltas = torch.tensor(NEAR_CEILING_OFFSETS).repeat(N // len(NEAR_CEILING_OFFSETS))
    q = torch.zeros(N, d)
    q[:, 0] = deltas
    k = torch.zeros(N, d)
    k[128::2, 0] = 1.0
    k[129::2, 0] = 0.5
    q8, k8 = (t.to(torch.float8_e4m3fn).view(torch.uint8) for t in (q, k))
    assert torch.equal(q8.view(torch.float8_e4m3fn).float(), q)  # every offset is an E4M3 value
    mags = torch.tensor([0x7B, 0x7C, 0x7D, 0x7E], dtype=torch.uint8)  # 352, 384, 416, 448
    v8 = mags[torch.randint(0, 4, (N, d), generator=g)] | (torch.randint(0, 2, (N, d), generator=g,
                                                                           dtype=torch.uint8) << 7)
    scales = (1.0, 1.0, 1.0 / 448.0)
    scale = float(torch.tensor(0.6931471805599453, dtype=torch.float32))
    shape = (1, 1, N, d)
    return q8.reshape(shape), k8.reshape(shape), v8.reshape(shape), scales, scale

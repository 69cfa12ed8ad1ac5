"""The K/V split's merge rule, pinned with the fp64 oracle (no GPU).

A split launch computes, for each segment s of a row's keys, the attention over
those keys alone (O_s, normalised, and LSE_s), and merges them by
    LSE = log sum_s exp(LSE_s),   O = sum_s exp(LSE_s - LSE) O_s.
This holds exactly because softmax over a union of disjoint key sets is the
LSE-weighted mixture of the softmaxes over the parts.  The test computes each
segment's attention in fp64 (numpy) on key segments laid out as the kernel
lays them out (whole 128-key tiles, the last one ragged), merges them with that
rule, and compares with the oracle's attention over all keys: equal to fp64
rounding.
"""
import numpy as np
import pytest

from exact_long_sequence_gb300 import workloads


def segment_attention(q, k, v, scale):
    """Attention of every query row over the given keys alone (fp64): (O [N, d], LSE [N])."""
    s = scale * (q @ k.T)
    m = s.max(1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(1, keepdims=True)
    return (e / l) @ v, (m + np.log(l))[:, 0]


def merge(parts):
    lse = np.stack([p[1] for p in parts])            # [S, rows]
    m = lse.max(0)
    w = np.exp(lse - m)                              # [S, rows]
    total = w.sum(0)
    O = sum(w[s][:, None] * parts[s][0] for s in range(len(parts))) / total[:, None]
    return O, m + np.log(total)


@pytest.mark.parametrize("N,segs", [(300, 2), (1000, 3), (1000, 4), (513, 2)])
def test_merge_of_segments_equals_full_attention(oracle_mod, N, segs):
    d = 64
    q, k, v = workloads.make_inputs(1, 1, N, d, seed=N + segs)
    scale = 0.125
    O_full, L_full = oracle_mod.attention_rows(q, k, v, False, scale)
    qd, kd, vd = (t.double().numpy().reshape(N, d) for t in (q, k, v))  # bf16 values, exactly
    ntiles = -(-N // 128)
    c = -(-ntiles // segs)  # K/V tiles per segment, as the kernel cuts them
    parts = []
    for s in range(segs):
        a, b = s * c * 128, min(N, (s + 1) * c * 128)
        assert a < b
        parts.append(segment_attention(qd, kd[a:b], vd[a:b], scale))
    O, L = merge(parts)
    assert np.abs(O - O_full.reshape(N, d)).max() <= 1e-12
    assert np.abs(L - L_full.reshape(N)).max() <= 1e-12 * np.abs(L_full).max()


def test_merge_weights_a_segment_by_its_mass():
    """A segment whose logits are all far below the others' contributes nothing."""
    d, N = 64, 256
    q, k, v = workloads.make_inputs(1, 1, N, d, seed=3)
    qd, kd, vd = (t.double().numpy().reshape(N, d) for t in (q, k, v))
    O_a, L_a = segment_attention(qd, kd[:128], vd[:128], 0.125)
    parts = [(O_a, L_a), (np.full((N, d), 7.0), L_a - 800.0)]
    O, L = merge(parts)
    np.testing.assert_allclose(O, O_a, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, L_a, rtol=1e-15, atol=0)

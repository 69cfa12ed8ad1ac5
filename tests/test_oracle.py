"""Pins for the fp64 oracle: closed forms and invariants of the attention definition.

The definition is the attention graph of "From Attention Graph to
FlashAttention - A Memory-Centric Compilation Approach in AICF", section 1:
Scores = Q x K^T (scaled), Mask, Softmax, Output = Scores x V, plus the
natural-log normaliser LSE. None of these tests re-types the oracle's formula:
each one checks a value the mathematics fixes independently (a closed form, an
invariant, a special case, or an independent library routine), chosen so that
a dropped term, a wrong sign or index, a transposed operand or an off-by-one
mask fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

from exact_long_sequence_gb300 import workloads

pytestmark = []


def bf16(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def f64(t):
    return t.to(torch.float64).numpy()


def rand_qkv(B, H, N, d, seed, v_dist="normal"):
    return workloads.make_inputs(B, H, N, d, seed, v_dist=v_dist)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_give_uniform_weights(oracle_mod, causal):
    """Q = 0 makes every logit 0: P is uniform over the visible keys, so O_i is
    the mean of the visible values and LSE_i = ln(#visible)."""
    N, d = 37, 8
    _, _, v = rand_qkv(1, 1, N, d, 11)
    q = torch.zeros_like(v)
    k = rand_qkv(1, 1, N, d, 12)[1]
    O, LSE = oracle_mod.attention_rows(q, k, v, causal, 0.125)
    V = f64(v)[0, 0]
    for i in range(N):
        nvis = i + 1 if causal else N
        np.testing.assert_allclose(O[0, i], V[:nvis].mean(axis=0), rtol=0, atol=1e-13)
        assert abs(LSE[0, i] - math.log(nvis)) < 1e-13


def test_two_keys_closed_form(oracle_mod):
    """d=1, N=2: the first weight is sigmoid(scale*q*(k1-k2)) and
    LSE = scale*q*k2 + log(1 + exp(scale*q*(k1-k2)))."""
    q = bf16([[1.5], [-1.0]]).reshape(1, 1, 2, 1)
    k = bf16([[2.0], [-0.5]]).reshape(1, 1, 2, 1)
    v = bf16([[3.0], [-1.0]]).reshape(1, 1, 2, 1)
    scale = 0.5
    O, LSE = oracle_mod.attention_rows(q, k, v, False, scale)
    for i, qi in enumerate([1.5, -1.0]):
        t = scale * qi * (2.0 - (-0.5))
        p1 = 1.0 / (1.0 + math.exp(-t))
        assert abs(O[0, i, 0] - (p1 * 3.0 + (1 - p1) * (-1.0))) < 1e-14
        assert abs(LSE[0, i] - (scale * qi * (-0.5) + math.log1p(math.exp(t)))) < 1e-14


def test_two_keys_causal_closed_form(oracle_mod):
    """Causal, N=2: row 0 sees only key 0 (O = v0, LSE = scale*q0*k0); row 1 sees both."""
    q = bf16([[1.5], [-1.0]]).reshape(1, 1, 2, 1)
    k = bf16([[2.0], [-0.5]]).reshape(1, 1, 2, 1)
    v = bf16([[3.0], [-1.0]]).reshape(1, 1, 2, 1)
    O, LSE = oracle_mod.attention_rows(q, k, v, True, 0.5)
    assert O[0, 0, 0] == 3.0 and LSE[0, 0] == 0.5 * 1.5 * 2.0
    t = 0.5 * -1.0 * 2.5
    p1 = 1.0 / (1.0 + math.exp(-t))
    assert abs(O[0, 1, 0] - (p1 * 3.0 - (1 - p1))) < 1e-14


@pytest.mark.parametrize("causal", [False, True])
def test_probabilities_sum_to_one(oracle_mod, causal):
    """Each row of P is a probability distribution; masked keys get exactly 0."""
    q, k, v = rand_qkv(1, 2, 50, 16, 3)
    _, _, P = oracle_mod.attention_rows(q, k, v, causal, 0.25, return_probs=True)
    np.testing.assert_allclose(P.sum(axis=-1), 1.0, rtol=0, atol=1e-12)
    assert (P >= 0).all()
    if causal:
        upper = np.triu(np.ones((50, 50), dtype=bool), k=1)
        assert (P[:, upper] == 0).all()
        assert (P[:, ~upper] > 0).all()


@pytest.mark.parametrize("causal", [False, True])
def test_constant_values_give_constant_output(oracle_mod, causal):
    q, k, _ = rand_qkv(1, 1, 40, 8, 4)
    v = torch.full_like(q, 0.375)
    O, _ = oracle_mod.attention_rows(q, k, v, causal, 0.3)
    np.testing.assert_allclose(O, 0.375, rtol=1e-14, atol=0)


def test_single_key_returns_its_value(oracle_mod):
    """N = 1: softmax of one logit is 1, so O = v and LSE = scale * q.k."""
    q, k, v = rand_qkv(2, 3, 1, 64, 5)
    O, LSE = oracle_mod.attention_rows(q, k, v, False, 0.125)
    np.testing.assert_array_equal(O.reshape(2, 3, 1, 64), f64(v))
    qk = (f64(q) * f64(k)).sum(-1)  # exact enough: 64 products of bf16 values
    np.testing.assert_allclose(LSE.reshape(2, 3, 1), 0.125 * qk, rtol=1e-14, atol=1e-14)


def test_key_value_permutation_invariance(oracle_mod):
    """Non-causal attention does not depend on the order of the (key, value) pairs."""
    q, k, v = rand_qkv(1, 1, 64, 32, 6)
    perm = torch.randperm(64, generator=torch.Generator().manual_seed(0))
    O1, L1 = oracle_mod.attention_rows(q, k, v, False, 0.2)
    O2, L2 = oracle_mod.attention_rows(q, k[:, :, perm], v[:, :, perm], False, 0.2)
    np.testing.assert_allclose(O1, O2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(L1, L2, rtol=1e-14, atol=0)


def test_logit_shift_moves_lse_only(oracle_mod):
    """Adding the same t to every logit of a row leaves O unchanged and adds t to LSE.
    Q's first column is 1 and K's first column moves from 0 to 2, so every logit
    grows by exactly scale*2."""
    q, k, v = rand_qkv(1, 1, 30, 8, 7)
    q[..., 0] = 1.0
    k[..., 0] = 0.0
    k2 = k.clone()
    k2[..., 0] = 2.0
    scale = 0.25
    O1, L1 = oracle_mod.attention_rows(q, k, v, False, scale)
    O2, L2 = oracle_mod.attention_rows(q, k2, v, False, scale)
    np.testing.assert_allclose(O1, O2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(L2 - L1, scale * 2.0, rtol=0, atol=1e-13)


def test_causal_row_is_attention_over_its_prefix(oracle_mod):
    """Causal row i equals non-causal attention of query i over keys 0..i."""
    N = 20
    q, k, v = rand_qkv(1, 1, N, 16, 8)
    Oc, Lc = oracle_mod.attention_rows(q, k, v, True, 0.25)
    for i in [0, 1, 7, N - 1]:
        qi = q[:, :, : i + 1]
        Op, Lp = oracle_mod.attention_rows(qi, k[:, :, : i + 1], v[:, :, : i + 1], False, 0.25,
                                           rows=np.array([[i]]))
        np.testing.assert_allclose(Oc[0, i], Op[0, 0], rtol=0, atol=1e-14)
        assert abs(Lc[0, i] - Lp[0, 0]) < 1e-13


def test_heads_are_independent(oracle_mod):
    """Each (b, h) uses its own K and V: a head whose V is constant c returns c."""
    B, H, N, d = 2, 3, 17, 8
    q, k, _ = rand_qkv(B, H, N, d, 9)
    v = torch.empty_like(q)
    consts = torch.arange(B * H, dtype=torch.float32).reshape(B, H) - 2.5
    for b in range(B):
        for h in range(H):
            v[b, h] = consts[b, h]
    O, _ = oracle_mod.attention_rows(q, k, v, True, 0.3)
    np.testing.assert_allclose(O.reshape(B, H, N, d), consts.double().numpy()[:, :, None, None]
                               * np.ones((1, 1, N, d)), rtol=1e-14, atol=0)


def test_huge_logits_do_not_overflow(oracle_mod):
    """Logits of order 1e4: the max-subtracted softmax keeps O = v of the winning key
    and LSE = its logit (plus a negligible log(1 + ...))."""
    q = bf16([[100.0]]).reshape(1, 1, 1, 1).expand(1, 1, 3, 1).contiguous()
    k = bf16([[100.0], [-100.0], [50.0]]).reshape(1, 1, 3, 1)
    v = bf16([[1.0], [2.0], [3.0]]).reshape(1, 1, 3, 1)
    O, LSE = oracle_mod.attention_rows(q, k, v, False, 1.0)
    assert np.isfinite(O).all() and np.isfinite(LSE).all()
    np.testing.assert_allclose(O[0, :, 0], 1.0, rtol=0, atol=1e-300)
    np.testing.assert_allclose(LSE[0], 1e4, rtol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(1, 64), (7, 16), (130, 64), (257, 128)])
def test_matches_torch_fp64(oracle_mod, causal, N, d):
    """Independent library routine: torch fp64 softmax / logsumexp on the same bf16 inputs."""
    q, k, v = rand_qkv(1, 2, N, d, 10 + N)
    scale = workloads.Workload("t", 1, 2, N, d, causal, 0).scale
    O, LSE = oracle_mod.attention_rows(q, k, v, causal, scale)
    qd, kd, vd = (t.to(torch.float64) for t in (q, k, v))
    s = scale * (qd @ kd.transpose(-1, -2))
    if causal:
        s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    ref_o = torch.softmax(s, dim=-1) @ vd
    ref_l = torch.logsumexp(s, dim=-1)
    np.testing.assert_allclose(O.reshape(1, 2, N, d), ref_o.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(LSE.reshape(1, 2, N), ref_l.numpy(), rtol=1e-13, atol=1e-13)


def test_sampled_rows_equal_full_rows(oracle_mod):
    q, k, v = rand_qkv(1, 3, 90, 16, 13)
    rows = workloads.sample_rows(3, 90, 11, seed=13)
    Of, Lf = oracle_mod.attention_rows(q, k, v, True, 0.25)
    Os, Ls = oracle_mod.attention_rows(q, k, v, True, 0.25, rows=rows.numpy(), nthreads=3)
    for bh in range(3):
        np.testing.assert_array_equal(Os[bh], Of[bh, rows[bh].numpy()])
        np.testing.assert_array_equal(Ls[bh], Lf[bh, rows[bh].numpy()])


def test_bad_row_index_is_rejected(oracle_mod):
    q, k, v = rand_qkv(1, 1, 8, 8, 14)
    with pytest.raises(ValueError):
        oracle_mod.attention_rows(q, k, v, False, 0.3, rows=np.array([[8]]))


def test_workload_recipe_is_seeded_and_shaped():
    w = workloads.WORKLOADS["b1h1n256d64"]
    a = workloads.workload_inputs(w)
    b = workloads.workload_inputs(w)
    for x, y in zip(a, b):
        assert x.dtype == torch.bfloat16 and x.shape == (1, 1, 256, 64)
        assert torch.equal(x, y)
    rows = workloads.sample_rows(4, 1000, 10, seed=2)
    assert rows.shape == (4, 10)
    assert all(len(set(r.tolist())) == 10 and r.tolist() == sorted(r.tolist()) for r in rows)
    assert workloads.Workload("x", 1, 1, 8, 128, False, 0).scale == np.float32(1 / math.sqrt(128))


def test_spiky_recipe_has_about_one_percent_outliers():
    q, k, v = workloads.make_inputs(1, 2, 2048, 64, 4, qk_dist="normal_spiky", v_dist="uniform")
    assert v.abs().max() <= 1.0
    frac = (q.float().abs() > 6).float().mean().item()  # N(0,1) almost never exceeds 6
    assert 0.005 < frac < 0.012

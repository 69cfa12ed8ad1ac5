"""Pins for the backward oracle (dQ, dK, dV for an upstream gradient dO).

The backward is the derivative of the attention definition; it is pinned here
against finite differences of the forward, an independent autograd routine,
closed forms and invariants, never against a re-typed copy of its formulas.
"""
import math

import numpy as np
import pytest
import torch

from exact_long_sequence_gb300 import workloads


def rnd(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def loss(oracle_mod, q, k, v, do, causal, scale, lib=None):
    fn = oracle_mod.attention_f64
    O, _ = fn(q, k, v, causal, scale)
    return float((O * do.reshape(O.shape)).sum())


def test_f64_forward_equals_bf16_forward(oracle_mod):
    """The double-input forward used by the backward is the pinned bf16 forward on decoded inputs."""
    for causal in (False, True):
        q, k, v = workloads.make_inputs(1, 2, 70, 32, seed=3)
        O1, L1 = oracle_mod.attention_rows(q, k, v, causal, 0.2)
        O2, L2 = oracle_mod.attention_f64(q, k, v, causal, 0.2)
        np.testing.assert_array_equal(O1, O2)
        np.testing.assert_array_equal(L1, L2)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_finite_differences(oracle_mod, causal):
    """dL/dx for L = sum(O * dO), by central differences of the forward, for every input entry."""
    N, d, scale = 5, 3, 0.7
    q, k, v, do = (rnd((1, 1, N, d), s) for s in (1, 2, 3, 4))
    dQ, dK, dV = oracle_mod.attention_bwd(q, k, v, do, causal, scale)
    eps = 1e-6
    for name, x, g in (("q", q, dQ), ("k", k, dK), ("v", v, dV)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            lp = loss(oracle_mod, args["q"], args["k"], args["v"], do, causal, scale)
            args[name] = xm
            lm = loss(oracle_mod, args["q"], args["k"], args["v"], do, causal, scale)
            fd[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(g.reshape(x.shape), fd, rtol=1e-6, atol=1e-8, err_msg=name)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(1, 8), (33, 16), (130, 64)])
def test_backward_matches_torch_autograd(oracle_mod, causal, N, d):
    """Independent library routine: torch fp64 autograd through softmax(scale Q K^T + mask) V."""
    q, k, v, do = (torch.tensor(rnd((2, N, d), s)) for s in (5, 6, 7, 8))
    scale = 1 / math.sqrt(d)
    qt, kt, vt = (t.clone().requires_grad_(True) for t in (q, k, v))
    s = scale * qt @ kt.transpose(-1, -2)
    if causal:
        s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    (torch.softmax(s, -1) @ vt).backward(do)
    dQ, dK, dV = oracle_mod.attention_bwd(q.numpy(), k.numpy(), v.numpy(), do.numpy(), causal, scale)
    for got, ref in ((dQ, qt.grad), (dK, kt.grad), (dV, vt.grad)):
        np.testing.assert_allclose(got, ref.numpy(), rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_changes_no_gradient(oracle_mod, causal):
    """Adding one vector u to every key adds q_i.u to all of row i's logits: the softmax,
    and with it every gradient, is unchanged (rows of dS sum to zero)."""
    q, k, v, do = (rnd((1, 1, 40, 8), s) for s in (9, 10, 11, 12))
    u = rnd((8,), 13)
    g1 = oracle_mod.attention_bwd(q, k, v, do, causal, 0.4)
    g2 = oracle_mod.attention_bwd(q, k + u, v, do, causal, 0.4)
    for a, b in zip(g1, g2):
        np.testing.assert_allclose(a, b, rtol=1e-9, atol=1e-11)


@pytest.mark.parametrize("causal", [False, True])
def test_key_gradients_sum_to_zero(oracle_mod, causal):
    """sum_j dK_j = scale * sum_i (sum_j dS_ij) q_i = 0."""
    q, k, v, do = (rnd((2, 50, 16), s) for s in (14, 15, 16, 17))
    _, dK, _ = oracle_mod.attention_bwd(q, k, v, do, causal, 0.3)
    np.testing.assert_allclose(dK.sum(axis=1), 0.0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_uniform_attention_value_gradient(oracle_mod, causal):
    """Q = 0: P is uniform over the visible keys, so dV_j = sum over the queries i that see j
    of dO_i / #visible(i), and dK = 0 (every score's gradient is scaled by q_i = 0)."""
    N, d = 23, 4
    q = np.zeros((1, N, d))
    k, v, do = (rnd((1, N, d), s) for s in (18, 19, 20))
    dQ, dK, dV = oracle_mod.attention_bwd(q, k, v, do, causal, 0.5)
    ref = np.zeros((N, d))
    for i in range(N):
        vis = range(i + 1) if causal else range(N)
        for j in vis:
            ref[j] += do[0, i] / len(vis)
    np.testing.assert_allclose(dV[0], ref, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dK, 0.0, atol=0)


def test_zero_upstream_gradient(oracle_mod):
    q, k, v = (rnd((1, 20, 8), s) for s in (21, 22, 23))
    for g in oracle_mod.attention_bwd(q, k, v, np.zeros_like(q), True, 0.3):
        assert (g == 0).all()


def test_single_visible_key_has_no_score_gradient(oracle_mod):
    """A query that sees one key has P = 1 whatever its score, so its score gradient is 0:
    with N = 1, dQ = dK = 0 and dV = dO; with the causal mask, query 0 sees only key 0,
    so dQ_0 = 0, and the last key is seen only by the last query: dV_{N-1} = P_{N-1,N-1} dO_{N-1}."""
    q, k, v, do = (rnd((1, 1, 6), s) for s in (24, 25, 26, 27))
    dQ, dK, dV = oracle_mod.attention_bwd(q, k, v, do, False, 0.4)
    assert (dQ == 0).all() and (dK == 0).all()
    np.testing.assert_array_equal(dV[0], do[0])
    N, d, scale = 9, 5, 0.45
    q, k, v, do = (rnd((1, N, d), s) for s in (28, 29, 30, 31))
    dQ, dK, dV = oracle_mod.attention_bwd(q, k, v, do, True, scale)
    assert (dQ[0, 0] == 0).all()
    s = scale * q[0, -1] @ k[0].T
    p_last = math.exp(s[-1] - s.max()) / np.exp(s - s.max()).sum()
    np.testing.assert_allclose(dV[0, -1], p_last * do[0, -1], rtol=1e-13)

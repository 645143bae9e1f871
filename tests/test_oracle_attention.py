"""Pins of the value-projection estimator oracle (oracle/attention.py)
against special cases, invariances and its large-population limit."""
import numpy as np
import pytest

import oracle


def _case(nseq=2, H=2, L=6, dv=4, d_in=3, seed=0):
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((nseq, H, L, L))
    logits = np.where(np.tril(np.ones((L, L))) > 0, logits, -np.inf)
    P = np.exp(logits - logits.max(-1, keepdims=True))
    P /= P.sum(-1, keepdims=True)
    T = nseq * L
    E = rng.standard_normal((T, H * dv))
    x = rng.standard_normal((T, d_in))
    return P, E, x, L


def test_identity_attention_own_token_is_the_projection_estimator():
    # P = I and gamma = 0: dl_{i,s} = sigma <E_s, a_{i,s}>, so
    # g_s = (1/K) sum_i (<E_s, a_i> - mean_j <E_s, a_j>) a_i.
    P, E, x, L = _case()
    nseq, H = P.shape[:2]
    P = np.broadcast_to(np.eye(L), P.shape).copy()
    K, sigma = 11, 0.3
    T, C = E.shape
    a = np.stack([oracle.noise(5, 2, i, 0, T, C) for i in range(K)])  # K x T x C
    proj = (a * E[None]).sum(-1)  # K x T
    proj -= proj.mean(0, keepdims=True)
    want = (proj[..., None] * a).sum(0) / K
    got = oracle.attn_value_estimate(P, E, x, L, sigma, 0.0, K, 5, 2)["g"]
    np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-12)


def test_sigma_cancels_exactly():
    P, E, x, L = _case(seed=1)
    g1 = oracle.attn_value_estimate(P, E, x, L, 0.5, 0.9, 6, 7, 2)["g"]
    g2 = oracle.attn_value_estimate(P, E, x, L, 1e-3, 0.9, 6, 7, 2)["g"]
    np.testing.assert_allclose(g1, g2, rtol=1e-9, atol=1e-12)


def test_first_token_error_only_reaches_the_first_token():
    # dl_s depends on E_s alone and r_t sums s >= t: changing E of the first
    # token of a sequence changes g only at that token.
    P, E, x, L = _case(seed=2)
    g1 = oracle.attn_value_estimate(P, E, x, L, 0.1, 0.95, 5, 3, 2)["g"]
    E2 = E.copy()
    E2[L] += 1.0  # first token of sequence 1
    g2 = oracle.attn_value_estimate(P, E2, x, L, 0.1, 0.95, 5, 3, 2)["g"]
    diff = np.abs(g1 - g2).max(axis=1)
    assert diff[L] > 1e-3
    assert np.all(np.delete(diff, L) < 1e-12)


def test_large_population_approaches_backprop_through_the_values():
    # With gamma = 1 the expectation is d/dv_t sum_s <E_s, o_s> =
    # sum_{s >= t} P_{s,t} E_s per head (the values' backprop gradient).
    P, E, x, L = _case(nseq=1, H=1, L=5, dv=3, seed=4)
    want = np.zeros_like(E)
    for t in range(L):
        for s in range(t, L):
            want[t] += P[0, 0, s, t] * E[s]
    g = oracle.attn_value_estimate(P, E, x, L, 0.1, 1.0, 20000, 11, 2)["g"]
    cos = (g * want).sum() / np.linalg.norm(g) / np.linalg.norm(want)
    assert cos > 0.99, cos


def _gate_case(T=8, C=12, d_in=3, seed=0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((T, C)), rng.standard_normal((T, C)),
            rng.standard_normal((T, C)), rng.standard_normal((T, d_in)))


def test_gate_small_sigma_limit_is_the_projection_onto_the_noise():
    # sig(z + d) - sig(z) = sig(z)(1 - sig(z)) d + O(d^2): with gamma = 0, g_s
    # -> (1/K) sum_i (<w_s, a_i> - mean) a_i, w = E sig(z)(1 - sig(z)) o.
    z, o, E, x = _gate_case()
    T, C = z.shape
    K, sigma = 9, 1e-5
    sg = 1.0 / (1.0 + np.exp(-z))
    wgt = E * sg * (1.0 - sg) * o
    a = np.stack([oracle.noise(8, 3, i, 0, T, C) for i in range(K)])
    proj = (a * wgt[None]).sum(-1)
    proj -= proj.mean(0, keepdims=True)
    want = (proj[..., None] * a).sum(0) / K
    got = oracle.attn_gate_estimate(z, o, E, x, T, sigma, 0.0, K, 8, 3)["g"]
    assert np.linalg.norm(got - want) / np.linalg.norm(want) < 1e-4


def test_gate_with_zero_output_estimates_nothing():
    z, o, E, x = _gate_case(seed=1)
    got = oracle.attn_gate_estimate(z, np.zeros_like(o), E, x, 8, 0.1, 0.9, 5, 8, 3)
    assert np.all(got["dl"] == 0.0) and np.all(got["g"] == 0.0)


def test_gate_change_is_the_difference_of_gated_outputs():
    # dl equals <E, sig(z + sigma a) o - sig(z) o> computed as two full gated
    # outputs (no shared intermediate).
    z, o, E, x = _gate_case(T=4, C=8, seed=2)
    sigma = 0.7
    dl = oracle.attn_gate_delta_loss(z, o, E, sigma, 2, 31, 3)
    for i in range(2):
        a = oracle.noise(31, 3, i, 0, 4, 8)
        out1 = o / (1.0 + np.exp(-(z + sigma * a)))
        out0 = o / (1.0 + np.exp(-z))
        np.testing.assert_allclose(dl[i], (E * out1).sum(1) - (E * out0).sum(1), rtol=1e-10,
                                   atol=1e-13)

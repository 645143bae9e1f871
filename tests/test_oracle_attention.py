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

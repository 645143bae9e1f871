"""Pins of the query and key estimator oracle (oracle/attention.py): the clean
forward against scipy's softmax, a two-token closed form valid at any sigma,
the first-order limit against the textbook attention gradient, invariances of
softmax attention, and the large-population limit of g."""
import numpy as np
import pytest
from scipy.special import softmax

import oracle


def _qkv(nseq=2, H=2, L=5, dv=4, d_in=3, seed=0):
    rng = np.random.default_rng(seed)
    T, C = nseq * L, H * dv
    Q, Kk, V, E = (rng.standard_normal((T, C)) for _ in range(4))
    x = rng.standard_normal((T, d_in))
    return Q, Kk, V, E, x


def test_forward_matches_scipy_softmax_per_row():
    Q, Kk, V, E, x = _qkv(seed=1)
    L, H, dv = 5, 2, 4
    P, O = oracle.attn_forward(Q, Kk, V, L, H)
    for sq in range(2):
        for h in range(H):
            q = Q[sq * L:(sq + 1) * L, h * dv:(h + 1) * dv]
            k = Kk[sq * L:(sq + 1) * L, h * dv:(h + 1) * dv]
            v = V[sq * L:(sq + 1) * L, h * dv:(h + 1) * dv]
            for s in range(L):
                p = softmax(q[s] @ k[:s + 1].T / 2.0)  # sqrt(dv) = 2
                np.testing.assert_allclose(P[sq, h, s, :s + 1], p, rtol=1e-13)
                assert np.all(P[sq, h, s, s + 1:] == 0.0)
                np.testing.assert_allclose(O[sq * L + s, h * dv:(h + 1) * dv], p @ v[:s + 1],
                                           rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("which", [0, 1])
def test_two_tokens_closed_form_at_large_sigma(which):
    # One head, two tokens: token 0 attends to itself only (dO_0 = 0 whatever
    # the perturbation) and token 1 has O_1 = v0 + sig(D) (v1 - v0) with
    # D = (s_11 - s_10) = q1 . (k1 - k0) / sqrt(dv), sig the logistic function.
    dv, sigma, K = 4, 0.7, 3
    Q, Kk, V, E, x = _qkv(nseq=1, H=1, L=2, dv=dv, seed=2)
    dl = oracle.attn_qk_delta_loss(which, Q, Kk, V, E, 2, 1, sigma, K, 17, 4 + which)
    sig = lambda u: 1.0 / (1.0 + np.exp(-u))
    D = Q[1] @ (Kk[1] - Kk[0]) / 2.0
    for i in range(K):
        a = oracle.noise(17, 4 + which, i, 0, 2, dv)
        if which == 0:
            Dp = (Q[1] + sigma * a[1]) @ (Kk[1] - Kk[0]) / 2.0
        else:
            Dp = Q[1] @ ((Kk[1] + sigma * a[1]) - (Kk[0] + sigma * a[0])) / 2.0
        assert dl[i, 0] == 0.0
        want = (sig(Dp) - sig(D)) * (E[1] @ (V[1] - V[0]))
        np.testing.assert_allclose(dl[i, 1], want, rtol=1e-11, atol=1e-14)


@pytest.mark.parametrize("which", [0, 1])
def test_small_sigma_limit_is_the_attention_gradient(which):
    # dl_{i,s} / sigma -> the directional derivative of <E_s, O_s> along a_i:
    #   d/dq_s = (1/sqrt dv) sum_t P_st (<E_s, v_t> - <E_s, o_s>) k_t
    #   d/dk_t = (1/sqrt dv) P_st (<E_s, v_t> - <E_s, o_s>) q_s     (t <= s)
    nseq, H, L, dv = 2, 2, 6, 4
    Q, Kk, V, E, x = _qkv(nseq, H, L, dv, seed=3)
    T, C = Q.shape
    sigma, K = 1e-6, 3
    dl = oracle.attn_qk_delta_loss(which, Q, Kk, V, E, L, H, sigma, K, 5, 4 + which)
    for i in range(K):
        a = oracle.noise(5, 4 + which, i, 0, T, C)
        want = np.zeros(T)
        for sq in range(nseq):
            for h in range(H):
                r0, cs = sq * L, slice(h * dv, (h + 1) * dv)
                for s in range(L):
                    p = softmax(Q[r0 + s, cs] @ Kk[r0:r0 + s + 1, cs].T / 2.0)
                    o = p @ V[r0:r0 + s + 1, cs]
                    w = p * (V[r0:r0 + s + 1, cs] @ E[r0 + s, cs] - o @ E[r0 + s, cs]) / 2.0
                    if which == 0:
                        want[r0 + s] += (w @ Kk[r0:r0 + s + 1, cs]) @ a[r0 + s, cs]
                    else:
                        want[r0 + s] += w @ (a[r0:r0 + s + 1, cs] @ Q[r0 + s, cs])
        np.testing.assert_allclose(dl[i] / sigma, want, rtol=1e-4, atol=1e-6)


@pytest.mark.parametrize("which", [0, 1])
def test_shifting_every_value_changes_nothing(which):
    # softmax rows sum to one before and after the perturbation, so adding a
    # vector b to every value of a head adds b to O and O' alike.
    Q, Kk, V, E, x = _qkv(seed=4)
    b = np.tile(np.arange(1.0, 5.0), 2)
    d1 = oracle.attn_qk_delta_loss(which, Q, Kk, V, E, 5, 2, 0.3, 4, 9, 4 + which)
    d2 = oracle.attn_qk_delta_loss(which, Q, Kk, V + b, E, 5, 2, 0.3, 4, 9, 4 + which)
    np.testing.assert_allclose(d1, d2, rtol=1e-9, atol=1e-12)


def test_query_perturbation_ignores_a_common_key_shift():
    # Adding one vector c to every key of a head adds (q + sigma a) . c to a
    # whole score row, which the softmax removes; the key perturbation has no
    # such invariance (its noise is per key), so the shift is a query-only pin.
    Q, Kk, V, E, x = _qkv(seed=5)
    c = np.tile(np.array([0.5, -1.0, 2.0, 0.25]), 2)
    d1 = oracle.attn_qk_delta_loss(0, Q, Kk, V, E, 5, 2, 0.3, 4, 9, 4)
    d2 = oracle.attn_qk_delta_loss(0, Q, Kk + c, V, E, 5, 2, 0.3, 4, 9, 4)
    np.testing.assert_allclose(d1, d2, rtol=1e-9, atol=1e-12)


def test_zero_keys_make_the_queries_inert():
    # All scores zero whatever the query: the perturbed output is the clean one.
    Q, Kk, V, E, x = _qkv(seed=6)
    got = oracle.attn_qk_estimate(0, Q, np.zeros_like(Kk), V, E, x, 5, 2, 0.3, 0.9, 4, 9, 4)
    assert np.abs(got["dl"]).max() < 1e-15
    assert np.abs(got["g"]).max() < 1e-13


@pytest.mark.parametrize("which", [0, 1])
def test_large_population_approaches_backprop(which):
    # gamma = 1 and small sigma: E[g_t] = d/d(q_t or k_t) of sum_s <E_s, O_s>.
    nseq, H, L, dv = 1, 1, 4, 3
    Q, Kk, V, E, x = _qkv(nseq, H, L, dv, seed=7)
    want = np.zeros_like(Q)
    for s in range(L):
        p = softmax(Q[s] @ Kk[:s + 1].T / np.sqrt(dv))
        o = p @ V[:s + 1]
        w = p * (V[:s + 1] @ E[s] - o @ E[s]) / np.sqrt(dv)
        if which == 0:
            want[s] += w @ Kk[:s + 1]
        else:
            want[:s + 1] += np.outer(w, Q[s])
    g = oracle.attn_qk_estimate(which, Q, Kk, V, E, x, L, H, 1e-3, 1.0, 4000, 11, 4 + which)["g"]
    cos = (g * want).sum() / np.linalg.norm(g) / np.linalg.norm(want)
    assert cos > 0.98, cos

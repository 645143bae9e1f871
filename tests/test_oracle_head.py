"""Pins of the oracle's LM-head estimator (CPU only).

- The per-token loss change is checked against PyTorch's float64
  cross-entropy of the perturbed logits (a library routine the oracle does not
  use).
- gamma = 0 keeps the own token: the reward equals the centred decrease
  (hn.213312.xyz Dust translation §2.2).
- Closed-form statistics.  For small sigma one draw's estimate of the head
  error g_t = softmax(z_t) - onehot(y_t) has mean ((K-1)/K) g_t over K draws and
  covariance (|g_t|^2 I + g_t g_t^T) / K, so the outer product
  G_hat = sum_t g_hat_t x_t^T has cos(G_hat, G) ~ 1/sqrt(1 + c/K) with
  c = sum_t |x_t|^2 (V+1) |g_t|^2 / |G|_F^2 -- the two-parameter law
  cos(K) = c_max / sqrt(1 + c/K) the pages fit (hn.213312.xyz §4.2).  A wrong
  sign, scale, index or a dropped centring fails these.
- Brute-force unbiasedness on a tiny problem.
- Invariants: a per-token constant added to every loss change leaves g
  unchanged; g is linear in the reward; draws split by draw0 reproduce the
  single call.
"""
import math

import numpy as np
import pytest
import torch

from conftest import rel_l2


def _tiny(T=8, V=32, d=5, seed=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d)).astype(np.float32)
    W = (rng.standard_normal((V, d)) / math.sqrt(d)).astype(np.float32)
    z = (x.astype(np.float64) @ W.astype(np.float64).T).astype(np.float32)
    y = rng.integers(0, V, T).astype(np.int32)
    return x, W, z, y


def _analytic_head(z, y, x):
    z = np.asarray(z, np.float64)
    p = np.exp(z - z.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    g = p.copy()
    g[np.arange(len(y)), y] -= 1
    return g, g.T @ np.asarray(x, np.float64)


def test_delta_loss_matches_torch_cross_entropy(orc):
    x, W, z, y = _tiny()
    sigma, K, seed, layer = 0.3, 6, 77, 0
    dl = orc.head_delta_loss(z, y, sigma, K, seed, layer, draw0=3, token0=10)
    zt = torch.tensor(z, dtype=torch.float64)
    yt = torch.tensor(y, dtype=torch.long)
    ce0 = torch.nn.functional.cross_entropy(zt, yt, reduction="none")
    for i in range(K):
        a = torch.tensor(orc.noise(seed, layer, 3 + i, 10, z.shape[0], z.shape[1]))
        ce = torch.nn.functional.cross_entropy(zt + sigma * a, yt, reduction="none")
        np.testing.assert_allclose(dl[i], (ce - ce0).numpy(), rtol=1e-11, atol=1e-13)


def test_gamma_zero_is_own_token(orc):
    rng = np.random.default_rng(1)
    c = rng.standard_normal((5, 12))
    r = orc.reward(c, 0.0, 4)
    np.testing.assert_array_equal(r, c)
    r_lit = orc.reward(c, 0.0, 4, literal=True)
    np.testing.assert_array_equal(r_lit, c)


def test_center_is_mean_over_draws(orc):
    dl = np.random.default_rng(2).standard_normal((7, 9))
    c = orc.center(dl)
    np.testing.assert_allclose(c.sum(0), 0, atol=1e-14)
    np.testing.assert_allclose(c[0] - c[1], -(dl[0] - dl[1]), atol=1e-14)


def test_head_ghat_sign_and_scale_one_draw_pair(orc):
    """K = 2 by hand: c = -(dl - mean), g = -(c_0 a_0 + c_1 a_1) / (2 sigma)."""
    x, W, z, y = _tiny(T=3, V=8)
    sigma, seed = 0.1, 5
    out = orc.head_estimate(z, y, x, sigma, 2, seed, 0)
    a0 = orc.noise(seed, 0, 0, 0, 3, 8)
    a1 = orc.noise(seed, 0, 1, 0, 3, 8)
    d0, d1 = out["dl"]
    half = (d0 - d1) / 2.0        # c_1 = half, c_0 = -half
    expect = -(-half[:, None] * a0 + half[:, None] * a1) / (2 * sigma)
    np.testing.assert_allclose(out["g"], expect, rtol=1e-12, atol=1e-14)


@pytest.fixture(scope="module")
def head_tiny_runs(orc):
    """Config-1 shape: T=256, d=64, V=512, sigma=0.05; G_hat at several K."""
    import workloads
    w = workloads.head_workload(**workloads.HEAD_TINY)
    g, G = _analytic_head(w["z"], w["targets"], w["x"])
    res = {}
    for K in (64, 256, 1024, 4096):
        out = orc.head_estimate(w["z"], w["targets"], w["x"], 0.05, K, 1234, 0)
        res[K] = out
    return w, g, G, res


def test_cosine_law(head_tiny_runs):
    w, g, G, res = head_tiny_runs
    x = w["x"].astype(np.float64)
    V = w["V"]
    c_pred = float((np.sum(x * x, 1) * (V + 1) * np.sum(g * g, 1)).sum() / np.sum(G * G))
    cos = {}
    for K, out in res.items():
        Gh = out["G"]
        cos[K] = float(np.sum(Gh * G) / np.linalg.norm(Gh) / np.linalg.norm(G))
        pred = 1 / math.sqrt(1 + c_pred / K)
        assert abs(cos[K] - pred) <= 0.03, (K, cos[K], pred)
    Ks = sorted(cos)
    assert all(cos[a] < cos[b] for a, b in zip(Ks, Ks[1:]))
    # two-parameter fit of cos(K) = c_max / sqrt(1 + c/K): 1/cos^2 = (1 + c/K)/c_max^2
    A = np.stack([np.ones(len(Ks)), 1.0 / np.array(Ks, float)], 1)
    sol, *_ = np.linalg.lstsq(A, np.array([1 / cos[k] ** 2 for k in Ks]), rcond=None)
    c_max = 1 / math.sqrt(sol[0])
    c_fit = sol[1] / sol[0]
    assert 0.97 <= c_max <= 1.0 + 1e-2, c_max
    assert abs(c_fit - c_pred) <= 0.15 * c_pred, (c_fit, c_pred)


def test_projection_scale(head_tiny_runs):
    """<G_hat, G>/|G|^2 -> (K-1)/K, the centring by the mean over draws."""
    w, g, G, res = head_tiny_runs
    Gh = res[4096]["G"]
    s = float(np.sum(Gh * G) / np.sum(G * G))
    assert abs(s - 4095 / 4096) < 0.05, s


def test_ghat_per_token_matches_analytic_direction(head_tiny_runs):
    w, g, G, res = head_tiny_runs
    gh = res[4096]["g"]
    cos_t = np.sum(gh * g, 1) / np.linalg.norm(gh, axis=1) / np.linalg.norm(g, axis=1)
    # per token: c_t = (V+1) with |g|^2 cancelling -> cos ~ 1/sqrt(1 + (V+1)/K) = 0.94
    pred = 1 / math.sqrt(1 + (w["V"] + 1) / 4096)
    assert abs(np.median(cos_t) - pred) < 0.03


def test_unbiased_brute_force(orc):
    """Mean of g over many seeds equals ((K-1)/K) (softmax - onehot) within 4 SE."""
    x, W, z, y = _tiny(T=2, V=4, d=3, seed=3)
    g, _ = _analytic_head(z, y, x)
    K, sigma, nseed = 100, 0.01, 2000
    acc = []
    for s in range(nseed):
        out = orc.head_estimate(z, y, x, sigma, K, 10_000 + s, 0)
        acc.append(out["g"])
    acc = np.array(acc)
    mean = acc.mean(0)
    se = acc.std(0, ddof=1) / math.sqrt(nseed)
    target = (K - 1) / K * g
    assert np.all(np.abs(mean - target) <= 4 * se + 1e-4), (mean, target, se)


def test_constant_shift_invariance(orc):
    dl = np.random.default_rng(4).standard_normal((16, 6)) * 0.01
    shift = np.random.default_rng(5).standard_normal(6)
    c1 = orc.center(dl)
    c2 = orc.center(dl + shift[None, :])
    np.testing.assert_allclose(c1, c2, atol=1e-15)
    g1 = orc.ghat(orc.reward(c1, 0.0, 6), 10, 0.05, 3, 0)
    g2 = orc.ghat(orc.reward(c2, 0.0, 6), 10, 0.05, 3, 0)
    assert rel_l2(g1, g2) < 1e-12


def test_ghat_linear_in_reward(orc):
    rng = np.random.default_rng(6)
    r1, r2 = rng.standard_normal((2, 8, 5))
    g1 = orc.ghat(r1, 12, 0.05, 9, 1)
    g2 = orc.ghat(r2, 12, 0.05, 9, 1)
    g12 = orc.ghat(r1 + 2 * r2, 12, 0.05, 9, 1)
    np.testing.assert_allclose(g12, g1 + 2 * g2, rtol=1e-12, atol=1e-14)


def test_draw_chunks_reproduce_single_call(orc):
    """Draws [0,8) in one call equal draws [0,4) and [4,8) via draw0; the
    single-pass sums S1 = sum dl a, S0 = sum a recombine to the same g."""
    x, W, z, y = _tiny(T=4, V=16, d=3, seed=7)
    sigma, seed, K = 0.05, 21, 8
    full = orc.head_delta_loss(z, y, sigma, K, seed, 0)
    a = orc.head_delta_loss(z, y, sigma, 4, seed, 0, draw0=0)
    b = orc.head_delta_loss(z, y, sigma, 4, seed, 0, draw0=4)
    np.testing.assert_array_equal(full, np.concatenate([a, b]))
    g_full = orc.head_estimate(z, y, x, sigma, K, seed, 0)["g"]
    S1 = np.zeros((4, 16))
    S0 = np.zeros((4, 16))
    for i in range(K):
        an = orc.noise(seed, 0, i, 0, 4, 16)
        S1 += full[i][:, None] * an
        S0 += an
    m = full.mean(0)
    g_single_pass = (S1 - m[:, None] * S0) / (K * sigma)
    np.testing.assert_allclose(g_single_pass, g_full, rtol=1e-10, atol=1e-13)


def test_token_offset_slices(orc):
    """Noise is keyed by the global token index: a slice equals the full rows."""
    x, W, z, y = _tiny(T=6, V=16, d=3, seed=8)
    full = orc.head_delta_loss(z, y, 0.05, 3, 4, 0, token0=100)
    part = orc.head_delta_loss(z[2:5], y[2:5], 0.05, 3, 4, 0, token0=102)
    np.testing.assert_array_equal(full[:, 2:5], part)

"""Pins of the optimiser and exact-gradient oracle (oracle/optim.py) against
closed forms and hand-derived values, independent of its loops."""
import math

import numpy as np
import pytest

import oracle


def test_sgd_constant_gradient_closed_form():
    # b_k = g (1 - mu^k) / (1 - mu); W_t = W_0 - lr sum_k b_k
    W0, g, lr, mu, t = 1.5, 0.7, 0.1, 0.9, 6
    W, b = np.array([W0]), np.array([0.0])
    for _ in range(t):
        W, b = oracle.sgd_step(W, [g], b, lr, mu)
    total = (t - mu * (1 - mu ** t) / (1 - mu)) / (1 - mu)
    assert W[0] == pytest.approx(W0 - lr * g * total, rel=1e-14)
    assert b[0] == pytest.approx(g * (1 - mu ** t) / (1 - mu), rel=1e-14)


def test_sgd_momentum_on_quadratic_matches_matrix_power():
    # f(W) = a W^2 / 2: (W, b) evolves by a fixed 2 x 2 linear map.
    a, lr, mu, W0, t = 3.0, 0.05, 0.8, 2.0, 9
    M = np.array([[1 - lr * a, -lr * mu], [a, mu]])  # [W'; b'] = M [W; b]
    want = np.linalg.matrix_power(M, t) @ np.array([W0, 0.0])
    W, b = np.array([W0]), np.array([0.0])
    for _ in range(t):
        W, b = oracle.sgd_step(W, a * W, b, lr, mu)
    assert W[0] == pytest.approx(want[0], rel=1e-12)
    assert b[0] == pytest.approx(want[1], rel=1e-12)


def test_sgd_weight_decay_alone_shrinks_geometrically():
    W, b = np.array([2.0, -1.0]), np.zeros(2)
    for _ in range(5):
        W, b = oracle.sgd_step(W, [0.0, 0.0], b, 0.1, 0.0, wd=0.5)
    np.testing.assert_allclose(W, np.array([2.0, -1.0]) * 0.95 ** 5, rtol=1e-14)


def test_adam_constant_gradient_moves_lr_per_step():
    # m_hat = g and v_hat = g^2 at every step, so each step is lr g / (|g| + eps).
    g, lr, eps, t = np.array([0.3, -2.0]), 0.01, 1e-8, 10
    W, m, v = np.array([1.0, 1.0]), np.zeros(2), np.zeros(2)
    for k in range(1, t + 1):
        W, m, v = oracle.adam_step(W, g, m, v, k, lr, 0.9, 0.999, eps)
    np.testing.assert_allclose(W, 1.0 - t * lr * g / (np.abs(g) + eps), rtol=1e-12)


def test_adam_two_steps_by_hand():
    # b1 = b2 = 1/2, g = 1 then -1: step 1 m_hat = 1, v_hat = 1; step 2
    # m = -1/4, v = 3/4, bias corrections 3/4, so m_hat = -1/3, v_hat = 1.
    lr, eps = 0.1, 1e-6
    W, m, v = np.array([0.0]), np.zeros(1), np.zeros(1)
    W, m, v = oracle.adam_step(W, [1.0], m, v, 1, lr, 0.5, 0.5, eps)
    assert W[0] == pytest.approx(-lr / (1 + eps), rel=1e-14)
    W, m, v = oracle.adam_step(W, [-1.0], m, v, 2, lr, 0.5, 0.5, eps)
    assert m[0] == pytest.approx(-0.25) and v[0] == pytest.approx(0.75)
    assert W[0] == pytest.approx(-lr / (1 + eps) + lr * (1 / 3) / (1 + eps), rel=1e-13)


def test_adam_decoupled_weight_decay_with_zero_gradient():
    W, m, v = np.array([3.0]), np.zeros(1), np.zeros(1)
    for k in range(1, 5):
        W, m, v = oracle.adam_step(W, [0.0], m, v, k, 0.1, 0.9, 0.999, 1e-8, wd=0.2)
    assert W[0] == pytest.approx(3.0 * 0.98 ** 4, rel=1e-14)


def test_head_grad_rows_sum_to_zero_and_target_negative():
    rng = np.random.default_rng(0)
    z = rng.standard_normal((5, 17))
    y = rng.integers(0, 17, 5)
    g = oracle.head_grad_rows(z, y)
    np.testing.assert_allclose(g.sum(axis=1), 0.0, atol=1e-15)
    assert all(g[t, y[t]] < 0 for t in range(5))


def test_head_backprop_matches_finite_differences():
    # d/dW of sum_t CE(x_t W^T, y_t) by central differences on a tiny head.
    rng = np.random.default_rng(1)
    T, V, d = 6, 5, 3
    x = rng.standard_normal((T, d))
    Wh = rng.standard_normal((V, d)) * 0.5
    y = rng.integers(0, V, T)

    def loss(Wm):
        z = x @ Wm.T
        zmax = z.max(axis=1, keepdims=True)
        lse = zmax[:, 0] + np.log(np.exp(z - zmax).sum(axis=1))
        return float((lse - z[np.arange(T), y]).sum())

    G = oracle.head_backprop(x @ Wh.T, y, x)["G"]
    h = 1e-6
    num = np.zeros_like(Wh)
    for i in range(V):
        for j in range(d):
            E = np.zeros_like(Wh)
            E[i, j] = h
            num[i, j] = (loss(Wh + E) - loss(Wh - E)) / (2 * h)
    np.testing.assert_allclose(G, num, rtol=1e-6, atol=1e-8)


def test_es_estimate_on_a_linear_loss_is_the_sample_covariance_times_w():
    # L(theta + sigma eps) - mean = sigma w.(eps_i - mean eps), so
    # g = (1/K) sum_i (w.(eps_i - eps_bar)) eps_i = C w with the sample
    # moment matrix C = (1/K) sum_i (eps_i - eps_bar) eps_i^T.
    rng = np.random.default_rng(3)
    n, K, sigma = 6, 40, 0.01
    w = rng.standard_normal(n)
    theta = rng.standard_normal(n)
    eps = oracle.es_noise(n, K, 5, 9)
    losses = (theta[None] + sigma * eps) @ w
    C = ((eps - eps.mean(0)).T @ eps) / K
    np.testing.assert_allclose(oracle.es_estimate(losses, n, sigma, 5, 9), C @ w, rtol=1e-10)


def test_es_estimate_on_a_quadratic_tends_to_its_gradient():
    # For L = theta^T A theta / 2, Gaussian smoothing leaves the gradient A theta.
    rng = np.random.default_rng(4)
    n, K, sigma = 3, 20000, 0.1
    A = np.diag([1.0, 2.0, 3.0])
    theta = rng.standard_normal(n)
    th = theta[None] + sigma * oracle.es_noise(n, K, 6, 9)
    losses = 0.5 * np.einsum("ki,ij,kj->k", th, A, th)
    g = oracle.es_estimate(losses, n, sigma, 6, 9)
    cos = g @ (A @ theta) / np.linalg.norm(g) / np.linalg.norm(A @ theta)
    assert cos > 0.99, cos

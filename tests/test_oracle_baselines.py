"""Pins of the head estimator's leave-one-out and antithetic baselines
(oracle/baselines.py) against identities and limits that do not use its code."""
import numpy as np
import pytest

import oracle


def _inputs(T=6, V=40, d=5, seed=0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((T, V)), rng.integers(0, V, T).astype(np.int32),
            rng.standard_normal((T, d)))


def test_leave_one_out_is_K_over_K_minus_1_times_the_mean_baseline():
    # dl_i - mean_{j != i} dl_j = K/(K-1) (dl_i - mean_j dl_j), exactly.
    z, y, x = _inputs()
    K = 9
    loo = oracle.head_estimate_leave_one_out(z, y, x, 0.05, K, 1234, 0)
    mean = oracle.head_estimate(z, y, x, 0.05, K, 1234, 0)
    np.testing.assert_allclose(loo["g"], K / (K - 1) * mean["g"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(loo["G"], K / (K - 1) * mean["G"], rtol=1e-12, atol=1e-14)


def test_antithetic_small_sigma_limit_is_the_projection_onto_the_noise():
    # dl(+a) - dl(-a) = 2 sigma <grad, a> + O(sigma^3), so as sigma -> 0
    # g -> (1/K) sum_i <p_t - e_y, a_i> a_i, with an O(sigma^2) error.
    z, y, x = _inputs()
    T, V = z.shape
    K, sigma = 7, 1e-4
    grad = np.exp(z - z.max(1, keepdims=True))
    grad /= grad.sum(1, keepdims=True)
    grad[np.arange(T), y] -= 1.0
    want = np.zeros((T, V))
    for i in range(K):
        a = oracle.noise(1234, 0, i, 0, T, V)
        want += (grad * a).sum(1, keepdims=True) * a
    want /= K
    got = oracle.head_estimate_antithetic(z, y, x, sigma, K, 1234, 0)["g"]
    assert np.linalg.norm(got - want) / np.linalg.norm(want) < 1e-6


def test_antithetic_error_shrinks_as_sigma_squared():
    z, y, x = _inputs(seed=3)
    lim = oracle.head_estimate_antithetic(z, y, x, 1e-5, 5, 7, 0)["g"]
    e1 = np.linalg.norm(oracle.head_estimate_antithetic(z, y, x, 0.2, 5, 7, 0)["g"] - lim)
    e2 = np.linalg.norm(oracle.head_estimate_antithetic(z, y, x, 0.1, 5, 7, 0)["g"] - lim)
    assert 3.5 < e1 / e2 < 4.5, e1 / e2


def test_antithetic_pair_changes_are_cross_entropies_of_the_perturbed_logits():
    # c_i = -(CE(z + sigma a) - CE(z - sigma a)) / 2, each CE taken as
    # -log of the target's softmax probability.
    z, y, x = _inputs(T=3, V=11, seed=5)
    T, V = z.shape
    sigma = 0.3

    def ce(zz):
        p = np.exp(zz - zz.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        return -np.log(p[np.arange(T), y])
    c = oracle.head_estimate_antithetic(z, y, x, sigma, 2, 99, 0)["c"]
    for i in range(2):
        a = oracle.noise(99, 0, i, 0, T, V)
        np.testing.assert_allclose(c[i], -(ce(z + sigma * a) - ce(z - sigma * a)) / 2,
                                   rtol=1e-12, atol=1e-14)


def test_chunked_with_one_chunk_is_the_mean_estimator():
    z, y, x = _inputs(V=40)
    got = oracle.head_estimate_chunked(z, y, x, 0.05, 6, 1234, 0, 40)
    want = oracle.head_estimate(z, y, x, 0.05, 6, 1234, 0)
    np.testing.assert_allclose(got["g"], want["g"], rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(got["G"], want["G"], rtol=1e-9, atol=1e-12)


def test_chunked_small_sigma_limit_is_the_projection_per_chunk():
    # Each chunk's columns tend to (1/K_c) sum_i (<grad_c, a_i> - mean) a_i over
    # that chunk's draws, grad = p - e_y restricted to the chunk.
    z, y, x = _inputs(T=4, V=24)
    T, V = z.shape
    chunk, K, sigma = 8, 12, 1e-5
    nch = V // chunk
    grad = np.exp(z - z.max(1, keepdims=True))
    grad /= grad.sum(1, keepdims=True)
    grad[np.arange(T), y] -= 1.0
    want = np.zeros((T, V))
    for c in range(nch):
        cols = slice(c * chunk, (c + 1) * chunk)
        a = np.stack([oracle.noise(1234, 0, c + k * nch, 0, T, V)[:, cols] for k in range(K // nch)])
        proj = (a * grad[None, :, cols]).sum(-1)
        proj -= proj.mean(0, keepdims=True)
        want[:, cols] = (proj[..., None] * a).sum(0) / (K // nch)
    got = oracle.head_estimate_chunked(z, y, x, sigma, K, 1234, 0, chunk)["g"]
    assert np.linalg.norm(got - want) / np.linalg.norm(want) < 1e-4


def test_chunked_loss_change_uses_only_the_chunk():
    # A chunk that does not hold the target and whose logits are far below the
    # rest barely moves the loss: its columns of g stay tiny.
    z, y, x = _inputs(T=3, V=16)
    z[:, 8:] -= 30.0
    y = np.array([0, 1, 2], np.int32)
    g = oracle.head_estimate_chunked(z, y, x, 0.1, 8, 5, 0, 8)["g"]
    assert np.abs(g[:, 8:]).max() < 1e-9 < np.abs(g[:, :8]).max()

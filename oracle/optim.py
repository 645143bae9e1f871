"""fp64 oracle of what consumes the estimate: the optimiser step and the exact
head gradient the estimate is compared with.

TEST INFRASTRUCTURE ONLY, like the rest of oracle/: tests/ and the benchmark's
CPU-baseline leg are the only callers.

The pages train with SGD and momentum and report that Adam works on the
estimate unchanged (hn.213312.xyz Dust translation: experiment set-up, §3.3);
they tune by the single-batch cosine between the estimate and backprop's
gradient (§2.3, §4.2).  They fix no formula for either optimiser, so these are
the textbook ones, one element at a time:

    SGD with momentum (heavy ball, no dampening):
        b <- mu b + (G + wd W);  W <- W - lr b
    Adam (Kingma & Ba 2015, Algorithm 1) with decoupled weight decay
    (Loshchilov & Hutter 2019):
        m <- b1 m + (1 - b1) G;  v <- b2 v + (1 - b2) G^2
        m_hat = m / (1 - b1^t);  v_hat = v / (1 - b2^t)
        W <- W - lr (m_hat / (sqrt(v_hat) + eps) + wd W)

and the gradient of sum_t CE(z_t, y_t) with respect to the head weight:
    g_t = softmax(z_t) - e_{y_t};  G = sum_t g_t x_t^T.
"""
import math

import numpy as np


def sgd_step(W, G, b, lr, mu, wd=0.0):
    """Returns the new (W, b), float64, from float64 copies of the inputs."""
    W = np.array(W, np.float64).reshape(-1)
    G = np.asarray(G, np.float64).reshape(-1)
    b = np.array(b, np.float64).reshape(-1)
    for i in range(W.size):
        b[i] = mu * b[i] + (G[i] + wd * W[i])
        W[i] = W[i] - lr * b[i]
    return W, b


def adam_step(W, G, m, v, t, lr, b1, b2, eps, wd=0.0):
    """Returns the new (W, m, v), float64; t is the step number, from 1."""
    W = np.array(W, np.float64).reshape(-1)
    G = np.asarray(G, np.float64).reshape(-1)
    m = np.array(m, np.float64).reshape(-1)
    v = np.array(v, np.float64).reshape(-1)
    bc1 = 1.0 - b1 ** t
    bc2 = 1.0 - b2 ** t
    for i in range(W.size):
        m[i] = b1 * m[i] + (1.0 - b1) * G[i]
        v[i] = b2 * v[i] + (1.0 - b2) * G[i] * G[i]
        m_hat = m[i] / bc1
        v_hat = v[i] / bc2
        W[i] = W[i] - lr * (m_hat / (math.sqrt(v_hat) + eps) + wd * W[i])
    return W, m, v


def head_grad_rows(z, targets):
    """g_t = softmax(z_t) - e_{y_t}, row by row (float64)."""
    z = np.asarray(z, np.float64)
    T, V = z.shape
    g = np.empty((T, V), np.float64)
    for t in range(T):
        e = np.exp(z[t] - z[t].max())
        g[t] = e / e.sum()
        g[t, int(targets[t])] -= 1.0
    return g


def head_backprop(z, targets, x):
    """dict(g, G): the exact gradient of sum_t CE(z_t, y_t) with respect to the
    head weight, G = sum_t g_t x_t^T."""
    g = head_grad_rows(z, targets)
    G = g.T @ np.asarray(x, np.float64)
    return {"g": g, "G": G}


def es_noise(n, K, seed, layer, draw0=0, token0=0):
    """eps_i[j], K x n: the oracle's normals with parameter j as channel j of
    one token (the same counter scheme as the activation noise)."""
    from . import noise
    return np.stack([noise(seed, layer, draw0 + i, token0, 1, n)[0] for i in range(K)])


def es_estimate(losses, n, sigma, seed, layer, draw0=0, token0=0):
    """Weight-space ES for the residual-mixing scalars (hn.213312.xyz Dust
    translation §2.1 leaves them out of the activation method):
    g = (1/(K sigma)) sum_i (L_i - mean L) eps_i."""
    L = np.asarray(losses, np.float64)
    K = L.size
    eps = es_noise(n, K, seed, layer, draw0, token0)
    g = np.zeros(n)
    for i in range(K):
        g += (L[i] - L.mean()) * eps[i]
    return g / (K * sigma)


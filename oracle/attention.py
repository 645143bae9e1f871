"""fp64 oracle of the estimators inside attention: the value projection and
the gate of the attention output.

TEST INFRASTRUCTURE ONLY, like the rest of oracle/.

The pages score perturbations inside attention by the error of the attention
output, with a decay gamma close to 1 for later tokens (hn.213312.xyz Dust
translation §2.3; laoyaoba.com, section 机制拆解).  For the values, written out
in the method's order:

    a_i            noise of draw i, T x (H dv) (the oracle's Philox + Box-Muller)
    dO_{i,s}[h]    = sigma sum_{t <= s, same sequence} P[h]_{s,t} a_{i,t}[h]
    dl_{i,s}       = sum_h <E_s[h], dO_{i,s}[h]>      (first-order loss change)
    c, r, g, G     as for the interior layer: centring by the mean over draws,
                   r_t = sum_{s >= t} gamma^(s-t) c_s per sequence,
                   g_t = -(1/(K sigma)) sum_i r a,  G = g^T x.

The per-draw contraction P[h] a[h] is numpy's float64 matmul (a library step);
the causal mask is applied by zeroing P above the diagonal first.
"""
import numpy as np


def attn_value_delta_loss(P, E, sigma, K, seed, layer, draw0=0, token0=0):
    """K x T first-order loss changes dl_{i,s}."""
    from . import noise
    P = np.asarray(P, np.float64)
    E = np.asarray(E, np.float64)
    nseq, H, L, _ = P.shape
    T, C = E.shape
    dv = C // H
    mask = np.tril(np.ones((L, L)))
    dl = np.zeros((K, T), np.float64)
    for i in range(K):
        a = noise(seed, layer, draw0 + i, token0, T, C)
        for sq in range(nseq):
            rows = slice(sq * L, (sq + 1) * L)
            for h in range(H):
                cols = slice(h * dv, (h + 1) * dv)
                dO = sigma * ((P[sq, h] * mask) @ a[rows, cols])
                dl[i, rows] += (E[rows, cols] * dO).sum(axis=1)
    return dl


def attn_value_estimate(P, E, x, seq_len, sigma, gamma, K, seed, layer, draw0=0, token0=0):
    """dict(dl, c, r, g, G) of the value estimator."""
    from . import center, ghat, outer, reward
    dl = attn_value_delta_loss(P, E, sigma, K, seed, layer, draw0, token0)
    c = center(dl)
    r = reward(c, gamma, seq_len)
    C = np.asarray(E).shape[1]
    g = ghat(r, C, sigma, seed, layer, draw0, token0)
    return {"dl": dl, "c": c, "r": r, "g": g, "G": outer(g, np.asarray(x, np.float64))}


def attn_gate_delta_loss(z, o, E, sigma, K, seed, layer, draw0=0, token0=0):
    """K x T: dl_{i,s} = sum_c E (sig(z + sigma a) - sig(z)) o, the gated
    output's first-order loss change (sig the logistic function)."""
    from . import noise
    z = np.asarray(z, np.float64)
    o = np.asarray(o, np.float64)
    E = np.asarray(E, np.float64)
    T, C = z.shape
    sig = lambda u: 1.0 / (1.0 + np.exp(-u))
    dl = np.empty((K, T), np.float64)
    for i in range(K):
        a = noise(seed, layer, draw0 + i, token0, T, C)
        dl[i] = (E * (sig(z + sigma * a) - sig(z)) * o).sum(axis=1)
    return dl


def attn_gate_estimate(z, o, E, x, seq_len, sigma, gamma, K, seed, layer, draw0=0, token0=0):
    """dict(dl, c, r, g, G) of the gate estimator (the gated output sig(z) * o,
    scored by the error of the gated output)."""
    from . import center, ghat, outer, reward
    dl = attn_gate_delta_loss(z, o, E, sigma, K, seed, layer, draw0, token0)
    c = center(dl)
    r = reward(c, gamma, seq_len)
    g = ghat(r, np.asarray(z).shape[1], sigma, seed, layer, draw0, token0)
    return {"dl": dl, "c": c, "r": r, "g": g, "G": outer(g, np.asarray(x, np.float64))}


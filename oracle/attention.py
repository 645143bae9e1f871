"""fp64 oracle of the estimators inside attention: the value projection, the
gate of the attention output, and the queries and keys.

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



# ---------------------------------------------------------------------------
# Queries and keys.  The same scoring (the attention-output error, decay gamma)
# applied to a perturbation of every token's query, or of every token's key:
# the oracle re-runs the causal softmax attention with the perturbed operand
# and takes the difference of the outputs, no algebraic shortcut:
#
#   S[h]  = Q[h] K[h]^T / sqrt(dv), entries above the diagonal -inf
#   P[h]  = row softmax of S[h],  O[h] = P[h] V[h]
#   O'    = the same with Q + sigma a_i (queries) or K + sigma a_i (keys)
#   dl_{i,s} = sum_h <E_s[h], O'_s[h] - O_s[h]>
#
# then c, r, g and G exactly as for the values.
# ---------------------------------------------------------------------------
def attn_forward(Q, Kk, V, seq_len, H):
    """Clean causal attention, per sequence and head: (P, O) with P of shape
    (T/seq_len, H, seq_len, seq_len) (zero above the diagonal) and O T x H dv."""
    Q = np.asarray(Q, np.float64)
    Kk = np.asarray(Kk, np.float64)
    V = np.asarray(V, np.float64)
    T, C = Q.shape
    dv = C // H
    nseq, L = T // seq_len, seq_len
    upper = np.triu(np.ones((L, L), bool), 1)
    P = np.zeros((nseq, H, L, L))
    O = np.zeros((T, C))
    for sq in range(nseq):
        rows = slice(sq * L, (sq + 1) * L)
        for h in range(H):
            cols = slice(h * dv, (h + 1) * dv)
            S = Q[rows, cols] @ Kk[rows, cols].T / np.sqrt(dv)
            S[upper] = -np.inf
            S -= S.max(axis=1, keepdims=True)
            e = np.exp(S)
            P[sq, h] = e / e.sum(axis=1, keepdims=True)
            O[rows, cols] = P[sq, h] @ V[rows, cols]
    return P, O


def attn_qk_delta_loss(which, Q, Kk, V, E, seq_len, H, sigma, K, seed, layer, draw0=0,
                       token0=0):
    """K x T loss changes of the query (which 0) or key (which 1) perturbation."""
    from . import noise
    if which not in (0, 1):
        raise ValueError("which is 0 (queries) or 1 (keys)")
    Q = np.asarray(Q, np.float64)
    Kk = np.asarray(Kk, np.float64)
    E = np.asarray(E, np.float64)
    T, C = Q.shape
    _, O = attn_forward(Q, Kk, V, seq_len, H)
    dl = np.empty((K, T))
    for i in range(K):
        a = noise(seed, layer, draw0 + i, token0, T, C)
        if which == 0:
            _, Op = attn_forward(Q + sigma * a, Kk, V, seq_len, H)
        else:
            _, Op = attn_forward(Q, Kk + sigma * a, V, seq_len, H)
        dl[i] = (E * (Op - O)).sum(axis=1)
    return dl


def attn_qk_estimate(which, Q, Kk, V, E, x, seq_len, H, sigma, gamma, K, seed, layer, draw0=0,
                     token0=0):
    """dict(dl, c, r, g, G) of the query (which 0) or key (which 1) estimator."""
    from . import center, ghat, outer, reward
    dl = attn_qk_delta_loss(which, Q, Kk, V, E, seq_len, H, sigma, K, seed, layer, draw0, token0)
    c = center(dl)
    r = reward(c, gamma, seq_len)
    g = ghat(r, np.asarray(Q).shape[1], sigma, seed, layer, draw0, token0)
    return {"dl": dl, "c": c, "r": r, "g": g, "G": outer(g, np.asarray(x, np.float64))}

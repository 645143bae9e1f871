"""fp64 oracle of the LM-head estimator with the two other baselines.

TEST INFRASTRUCTURE ONLY, like the rest of oracle/.

The pages centre each draw's loss decrease by the mean over the draws
(hn.213312.xyz Dust translation, §2.2 credit assignment).  They describe no
other baseline; these are the two common variance-reduction ones, written out
as defined:

    leave-one-out:  c_i = -(dl_i - (1/(K-1)) sum_{j != i} dl_j)
    antithetic:     every draw's noise a_i is evaluated as +a_i and -a_i and
                    c_i = -(dl_i(+a_i) - dl_i(-a_i)) / 2

with dl(a) = CE(z_t + sigma a) - CE(z_t) on the cached logits, and then, as for
the mean, g_t = -(1/(K sigma)) sum_i c_i a_i and G_W = sum_t g_t x_t^T.  The
noise is the oracle's own Philox + Box-Muller (oracle.noise); the loss changes
of leave-one-out come from oracle.head_delta_loss, those of the antithetic
pairs from the log-sum-exp of the perturbed logits written out here.
"""
import numpy as np


def _lse(z):
    m = z.max(axis=1, keepdims=True)
    return m[:, 0] + np.log(np.exp(z - m).sum(axis=1))


def head_estimate_leave_one_out(z, targets, x, sigma, K, seed, layer, draw0=0, token0=0):
    from . import ghat, head_delta_loss, outer
    z = np.asarray(z, np.float64)
    T, V = z.shape
    dl = head_delta_loss(z, targets, sigma, K, seed, layer, draw0, token0)  # K x T
    c = np.empty_like(dl)
    for t in range(T):
        total = dl[:, t].sum()
        for i in range(K):
            c[i, t] = -(dl[i, t] - (total - dl[i, t]) / (K - 1))
    g = ghat(c, V, sigma, seed, layer, draw0, token0)
    return {"dl": dl, "c": c, "g": g, "G": outer(g, np.asarray(x, np.float64))}


def head_estimate_antithetic(z, targets, x, sigma, K, seed, layer, draw0=0, token0=0):
    from . import noise, outer
    z = np.asarray(z, np.float64)
    T, V = z.shape
    y = np.asarray(targets, np.int64)
    rows = np.arange(T)
    lse0 = _lse(z)
    acc = np.zeros((T, V), np.float64)
    c = np.empty((K, T), np.float64)
    for i in range(K):
        a = noise(seed, layer, draw0 + i, token0, T, V)
        dl_plus = (_lse(z + sigma * a) - (z[rows, y] + sigma * a[rows, y])) - (lse0 - z[rows, y])
        dl_minus = (_lse(z - sigma * a) - (z[rows, y] - sigma * a[rows, y])) - (lse0 - z[rows, y])
        c[i] = -(dl_plus - dl_minus) / 2.0
        acc += c[i][:, None] * a
    g = -acc / (K * sigma)
    return {"c": c, "g": g, "G": outer(g, np.asarray(x, np.float64))}


def head_estimate_chunked(z, targets, x, sigma, K, seed, layer, chunk, draw0=0, token0=0):
    """The head with one vocabulary chunk perturbed per draw (laoyaoba.com,
    section 机制拆解: each round recomputes the cross-entropy of a small chunk of
    the vocabulary), read as: chunks of width `chunk` tile the vocabulary, draw
    j perturbs chunk j mod (V/chunk), the loss change is the full-row cross
    entropy with only that chunk's logits moved, each chunk's draws are centred
    by their own mean, and each chunk's columns of g average over its draws."""
    from . import noise, outer
    z = np.asarray(z, np.float64)
    T, V = z.shape
    nch = V // chunk
    Kc = K // nch
    y = np.asarray(targets, np.int64)
    rows = np.arange(T)
    lse0 = _lse(z)
    g = np.zeros((T, V), np.float64)
    for c in range(nch):
        cols = slice(c * chunk, (c + 1) * chunk)
        dls, noises = [], []
        for k in range(Kc):
            j = c + k * nch  # the draw's index within the call
            a = noise(seed, layer, draw0 + j, token0, T, V)
            zp = z.copy()
            zp[:, cols] += sigma * a[:, cols]
            dls.append((_lse(zp) - zp[rows, y]) - (lse0 - z[rows, y]))
            noises.append(a[:, cols])
        dl = np.stack(dls)                  # Kc x T
        cc = -(dl - dl.mean(axis=0))
        for k in range(Kc):
            g[:, cols] += cc[k][:, None] * noises[k]
        g[:, cols] *= -1.0 / (Kc * sigma)
    return {"g": g, "G": outer(g, np.asarray(x, np.float64))}


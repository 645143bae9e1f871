"""fp64 CPU oracle of the Dust virtual-population gradient estimator.

TEST INFRASTRUCTURE ONLY: tests/, __graft_entry__.smoke() and the CPU-baseline
leg of bench.py are the only callers.  The CUDA library never imports, links or
runs anything here, and nothing here uses the CUDA library.

The arithmetic lives in dust_oracle.c (plain loops, double precision).  This
module marshals numpy arrays and chains the steps in the order the method
states them (hn.213312.xyz Dust translation, §2.2 credit assignment):

    noise a  ->  per-token loss change  ->  centred decrease c  ->
    reward r_t = sum_{s>=t} gamma^(s-t) c_s  ->  g_t = -(1/(K sigma)) sum_i r a
    ->  G_W = sum_t g_t x_t^T   (embedding: scatter-add of g_t into row id_t)

The two dense contractions of the interior re-forward (Delta h W2^T and
Delta e W_head^T) use numpy's float64 matmul as a library step; everything else
is the C loops.  What consumes the estimate (the optimiser step, the exact head
gradient it is compared with) is in optim.py; the head estimator with the
leave-one-out and antithetic baselines in baselines.py; the value projection
inside attention, the gate, the queries and the keys, scored by the
attention-output error, in attention.py.
"""
import ctypes
import os

import numpy as np

from . import build as _build
from .attention import (attn_forward, attn_gate_delta_loss, attn_gate_estimate,  # noqa: F401
                        attn_qk_delta_loss, attn_qk_estimate, attn_value_delta_loss,
                        attn_value_estimate)
from .baselines import (head_estimate_antithetic, head_estimate_chunked,  # noqa: F401
                        head_estimate_leave_one_out)
from .optim import (adam_step, es_estimate, es_noise, head_backprop,  # noqa: F401
                    head_grad_rows, sgd_step)

_lib = None

_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_u32p = np.ctypeslib.ndpointer(dtype=np.uint32, flags="C_CONTIGUOUS")
_I64 = ctypes.c_int64
_U32 = ctypes.c_uint32
_U64 = ctypes.c_uint64
_D = ctypes.c_double


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        sig = {
            "orc_philox_batch": [_u32p, _I64, _U32, _U32, _u32p],
            "orc_noise_words": [_U64, _U32, _U32, _I64, _I64, _I64, _u32p],
            "orc_noise_normals": [_U64, _U32, _U32, _I64, _I64, _I64, _f64p],
            "orc_head_delta_loss": [_f64p, _i32p, _I64, _I64, _D, _U64, _U32, _U32, _I64, _I64,
                                    _f64p],
            "orc_center": [_f64p, _I64, _I64, _f64p],
            "orc_reward_literal": [_f64p, _I64, _I64, _I64, _D, _f64p],
            "orc_reward_recurrence": [_f64p, _I64, _I64, _I64, _D, _f64p],
            "orc_ghat": [_f64p, _I64, _I64, _I64, _D, _U64, _U32, _U32, _I64, _f64p],
            "orc_outer": [_f64p, _f64p, _I64, _I64, _I64, _f64p],
            "orc_embed_scatter": [_f64p, _i32p, _I64, _I64, _I64, _i64p, _f64p],
            "orc_gelu": [_f64p, _I64, _f64p],
            "orc_interior_dh": [_f32p, _I64, _I64, _D, _U64, _U32, _U32, _I64, _f64p],
            "orc_ema": [_f64p, _I64, _I64, _I64, _D, _f64p],
            "orc_ce_delta": [_f64p, _f64p, _i32p, _I64, _I64, _f64p],
        }
        for name, args in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = None
        L.orc_uniform.argtypes = [_U32]
        L.orc_uniform.restype = _D
        _lib = L
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- noise ----
def philox(counters, key):
    """Philox4x32-10 of each counter (n x 4 uint32) under key (k0, k1)."""
    ctr = _c(counters, np.uint32).reshape(-1, 4)
    out = np.empty_like(ctr)
    lib().orc_philox_batch(ctr, ctr.shape[0], int(key[0]) & 0xFFFFFFFF,
                           int(key[1]) & 0xFFFFFFFF, out)
    return out


def uniform(word):
    return lib().orc_uniform(int(word))


def box_muller(words):
    """Normals of Philox words taken in pairs (n x 2 uint32, even word first),
    fp64: rho = sqrt(-2 ln u(w_even)), theta = 2 pi u(w_odd), the pair
    (rho cos theta, rho sin theta); u(w) = ((w >> 9) + 0.5) 2^-23 (Box & Muller,
    1958, with the uniform map of the noise).  The same map as the C oracle's
    token normals, applied to any words (tests feed it chosen ones)."""
    w = _c(words, np.uint32).reshape(-1, 2).astype(np.float64)
    u = (np.floor(w / 512.0) + 0.5) * 2.0 ** -23
    rho = np.sqrt(-2.0 * np.log(u[:, 0]))
    theta = 2.0 * np.pi * u[:, 1]
    return np.stack([rho * np.cos(theta), rho * np.sin(theta)], axis=1)


def noise_words(seed, layer, draw, token0, ntok, nchan):
    """Raw Philox words, ntok x nchan: word c%4 of block (c/4, token, draw, layer)."""
    out = np.empty((ntok, nchan), np.uint32)
    lib().orc_noise_words(seed, layer, draw, token0, ntok, nchan, out)
    return out


def noise(seed, layer, draw, token0, ntok, nchan):
    """Standard normals a_{draw,t}[c], ntok x nchan, fp64."""
    out = np.empty((ntok, nchan), np.float64)
    lib().orc_noise_normals(seed, layer, draw, token0, ntok, nchan, out)
    return out


# -------------------------------------------------------- method steps ----
def head_delta_loss(z, targets, sigma, K, seed, layer, draw0=0, token0=0):
    """K x T: CE(z_t + sigma a_{i,t}) - CE(z_t) on the cached logits (widened to fp64)."""
    z = _c(z, np.float64)
    T, V = z.shape
    dl = np.empty((K, T), np.float64)
    lib().orc_head_delta_loss(z, _c(targets, np.int32), T, V, sigma, seed, layer, draw0,
                              token0, K, dl)
    return dl


def center(dl):
    dl = _c(dl, np.float64)
    K, T = dl.shape
    c = np.empty_like(dl)
    lib().orc_center(dl, K, T, c)
    return c


def reward(c, gamma, seq_len, literal=False):
    c = _c(c, np.float64)
    K, T = c.shape
    assert T % seq_len == 0
    r = np.empty_like(c)
    fn = lib().orc_reward_literal if literal else lib().orc_reward_recurrence
    fn(c, K, T, seq_len, gamma, r)
    return r


def ghat(r, C, sigma, seed, layer, draw0=0, token0=0):
    r = _c(r, np.float64)
    K, T = r.shape
    g = np.empty((T, C), np.float64)
    lib().orc_ghat(r, K, T, C, sigma, seed, layer, draw0, token0, g)
    return g


def outer(g, x):
    """G[c][k] = sum_t g[t][c] x[t][k] by plain loops."""
    g = _c(g, np.float64)
    x = _c(x, np.float64)
    T, C = g.shape
    d = x.shape[1]
    G = np.empty((C, d), np.float64)
    lib().orc_outer(g, x, T, C, d, G)
    return G


def embed_scatter(g, ids, V):
    """(perm, G_E): stable order of (id, t) and the per-row sums of g."""
    g = _c(g, np.float64)
    T, d = g.shape
    perm = np.empty(T, np.int64)
    GE = np.empty((V, d), np.float64)
    lib().orc_embed_scatter(g, _c(ids, np.int32), T, d, V, perm, GE)
    return perm, GE


def gelu(u):
    u = _c(u, np.float64)
    out = np.empty_like(u)
    lib().orc_gelu(u.reshape(-1), u.size, out.reshape(-1))
    return out


def interior_dh(y1, sigma, seed, layer, draw, token0=0):
    y1 = _c(y1, np.float32)
    T, C = y1.shape
    dh = np.empty((T, C), np.float64)
    lib().orc_interior_dh(y1, T, C, sigma, seed, layer, draw, token0, dh)
    return dh


def ema(u, seq_len, lam):
    u = _c(u, np.float64)
    T, n = u.shape
    e = np.empty_like(u)
    lib().orc_ema(u, T, n, seq_len, lam, e)
    return e


def ce_delta(z, dz, targets):
    z = _c(z, np.float64)
    T, V = z.shape
    dl = np.empty(T, np.float64)
    lib().orc_ce_delta(z, _c(dz, np.float64), _c(targets, np.int32), T, V, dl)
    return dl


def interior_delta_loss(y1, W2, W_head, z_clean, targets, seq_len, lam, sigma, K, seed, layer,
                        draw0=0, token0=0):
    """K x T loss changes of the interior layer, re-running only the downstream.

    Per draw: dh = GELU(y1 + sigma a) - GELU(y1); du = dh W2^T; de = EMA(du);
    dz = de W_head^T; dl = CE(z_clean + dz) - CE(z_clean).  The perturbed
    logits are z_clean + dz because W2, the EMA and W_head are linear.
    """
    W2d = np.asarray(W2, np.float64)
    WHd = np.asarray(W_head, np.float64)
    T = y1.shape[0]
    dl = np.empty((K, T), np.float64)
    for i in range(K):
        dh = interior_dh(y1, sigma, seed, layer, draw0 + i, token0)
        du = dh @ W2d.T
        de = ema(du, seq_len, lam)
        dz = de @ WHd.T
        dl[i] = ce_delta(z_clean, dz, targets)
    return dl


# -------------------------------------------------------- whole paths ----
def head_estimate(z, targets, x, sigma, K, seed, layer, draw0=0, token0=0):
    """LM-head estimator (gamma = 0).  Returns dict(dl, c, g, G)."""
    T, V = np.shape(z)
    dl = head_delta_loss(z, targets, sigma, K, seed, layer, draw0, token0)
    c = center(dl)
    r = reward(c, 0.0, T)
    g = ghat(r, V, sigma, seed, layer, draw0, token0)
    G = outer(g, np.asarray(x, np.float64))
    return {"dl": dl, "c": c, "r": r, "g": g, "G": G}


def linear_estimate(x, y1, W2, lam, W_head, z_clean, targets, seq_len, sigma, gamma, K, seed,
                    layer, draw0=0, token0=0):
    """Interior linear layer estimator.  Returns dict(dl, c, r, g, G)."""
    y1 = np.asarray(y1, np.float32)
    C = y1.shape[1]
    dl = interior_delta_loss(y1, W2, W_head, z_clean, targets, seq_len, lam, sigma, K, seed,
                             layer, draw0, token0)
    c = center(dl)
    r = reward(c, gamma, seq_len)
    g = ghat(r, C, sigma, seed, layer, draw0, token0)
    G = outer(g, np.asarray(x, np.float64))
    return {"dl": dl, "c": c, "r": r, "g": g, "G": G}

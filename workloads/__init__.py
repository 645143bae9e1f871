"""Seeded synthetic inputs for the Dust estimator workloads.

This module only draws inputs and runs the clean (unperturbed) forward that
both the CUDA library and the CPU oracle receive as cached activations.  It
holds none of the estimator's arithmetic: no noise, no loss change, no reward,
no error estimate and no outer product.

The pages train an 8-layer, 512-wide GPT on FineWeb with a 4096-token BPE
vocabulary and batches of 8 x 2048 tokens (linlog.top article, experimental
setup; hn.213312.xyz Dust translation §3.1).  FineWeb is not used: token ids
and targets are drawn from a Zipf(1.1) law over the vocabulary, which stands
in for natural-text token frequencies, at the pages' batch shape.

Every array is a numpy array.  Values documented as bf16 are rounded to bf16
(round to nearest even) and returned as float32 arrays holding those exact
values; `as_bf16` marks which ones.
"""
import functools
import math

import numpy as np
import torch

# Data seeds per tensor role.
SEED_X, SEED_WHEAD, SEED_TARGETS, SEED_W1, SEED_W2, SEED_IDS, SEED_GHAT = 11, 12, 13, 14, 15, 16, 17
NOISE_SEED = 1234          # Philox seed of every workload
LAYER_HEAD, LAYER_INTERIOR = 0, 1


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def bf16_round(a):
    """Round float32 values to bf16 (nearest even); return them as float32."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def normal(seed, shape, std=1.0, bf16=False):
    a = (_rng(seed).standard_normal(shape) * std).astype(np.float32)
    return bf16_round(a) if bf16 else a


def zipf_ids(seed, n, vocab, s=1.1):
    """n ids with P(k) proportional to (k+1)^-s, k in [0, vocab), by inverse CDF."""
    p = np.arange(1, vocab + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(p)
    cdf /= cdf[-1]
    u = _rng(seed).random(n)
    return np.minimum(np.searchsorted(cdf, u, side="right"), vocab - 1).astype(np.int32)


def uniform_ids(seed, n, vocab):
    return _rng(seed).integers(0, vocab, n).astype(np.int32)


def _mm64(a, b_t, device):
    """a @ b_t.T in float64 (clean forward only)."""
    A = torch.from_numpy(np.ascontiguousarray(a, np.float64)).to(device)
    B = torch.from_numpy(np.ascontiguousarray(b_t, np.float64)).to(device)
    return A @ B.T


def _to_np32(t):
    return t.to(torch.float32).cpu().numpy()


# ------------------------------------------------------------ LM head ----
@functools.lru_cache(maxsize=8)
def head_workload(T, d, V, seq_len, x_bf16, zipf, device="cpu"):
    """Clean LM-head inputs: x (T x d), W_head (V x d), cached logits z = x W^T
    (fp32, computed in fp64 and rounded), targets (T)."""
    x = normal(SEED_X, (T, d), 1.0, x_bf16)
    W = normal(SEED_WHEAD, (V, d), 1.0 / math.sqrt(d), x_bf16)
    z = _to_np32(_mm64(x, W, device))
    y = zipf_ids(SEED_TARGETS, T, V) if zipf else uniform_ids(SEED_TARGETS, T, V)
    return {"x": x, "W": W, "z": z, "targets": y, "T": T, "d": d, "V": V,
            "seq_len": seq_len, "x_bf16": x_bf16}


HEAD_TINY = dict(T=256, d=64, V=512, seq_len=256, x_bf16=False, zipf=False)
HEAD_BATCH = dict(T=16384, d=512, V=4096, seq_len=2048, x_bf16=True, zipf=True)
HEAD_SCALE = dict(T=16384, d=1536, V=4096, seq_len=2048, x_bf16=True, zipf=True)

HEAD_PARAMS = {
    "head_tiny": dict(HEAD_TINY, sigma=0.05, K=64),
    "head_batch": dict(HEAD_BATCH, sigma=0.05, K=64),
    "head_scale": dict(HEAD_SCALE, sigma=0.05, K=4096),
    # the batch shape with antithetic pairs: 32 noise draws, 64 evaluations
    "head_batch_antithetic": dict(HEAD_BATCH, sigma=0.05, K=32, baseline=2),
    # one vocabulary chunk of 512 perturbed per draw: 512 draws cost the
    # element work of 64 full-vocabulary draws
    "head_batch_chunked": dict(HEAD_BATCH, sigma=0.05, K=512, chunk=512),
}
HEAD_SWEEP_K = (64, 256, 1024, 4096, 16384)


# ------------------------------------------------------ interior layer ----
def _ema_seq(u, seq_len, lam):
    """Causal per-sequence EMA of the clean forward, float64 torch."""
    T = u.shape[0]
    e = torch.empty_like(u)
    v = u.view(T // seq_len, seq_len, -1)
    ev = e.view(T // seq_len, seq_len, -1)
    prev = torch.zeros_like(v[:, 0])
    for t in range(seq_len):
        prev = lam * prev + (1.0 - lam) * v[:, t]
        ev[:, t] = prev
    return e


@functools.lru_cache(maxsize=4)
def interior_workload(T, d_in, C, d_model, V, seq_len, lam=0.9, device="cpu"):
    """Interior layer y1 = x W1^T (perturbed) with the fixed downstream
    GELU -> W2 -> causal EMA -> W_head -> CE.  Cached clean activations y1 and
    z_clean are fp32 (computed in fp64 and rounded)."""
    x = normal(SEED_X, (T, d_in), 1.0, True)
    W1 = normal(SEED_W1, (C, d_in), 1.0 / math.sqrt(d_in), True)
    W2 = normal(SEED_W2, (d_model, C), 1.0 / math.sqrt(C), True)
    WH = normal(SEED_WHEAD, (V, d_model), 1.0 / math.sqrt(d_model), True)
    y1_64 = _mm64(x, W1, device)
    y1 = _to_np32(y1_64)
    y1r = torch.from_numpy(y1).to(device).to(torch.float64)
    h0 = torch.nn.functional.gelu(y1r)                      # exact-erf GELU
    u0 = h0 @ torch.from_numpy(W2.astype(np.float64)).to(device).T
    e0 = _ema_seq(u0, seq_len, lam)
    z = _to_np32(e0 @ torch.from_numpy(WH.astype(np.float64)).to(device).T)
    y = zipf_ids(SEED_TARGETS, T, V)
    return {"x": x, "W1": W1, "W2": W2, "W_head": WH, "y1": y1, "z_clean": z, "targets": y,
            "T": T, "d_in": d_in, "C": C, "d_model": d_model, "V": V, "seq_len": seq_len,
            "lam": lam}


INTERIOR_BASE = dict(T=16384, d_in=512, C=2048, d_model=512, V=4096, seq_len=2048)
INTERIOR_SCALE = dict(T=16384, d_in=1536, C=6144, d_model=1536, V=4096, seq_len=2048)
INTERIOR_PARAMS = {
    "interior": dict(INTERIOR_BASE, sigma=0.02, gamma=0.95, K=256),
    "interior_scale": dict(INTERIOR_SCALE, sigma=0.02, gamma=0.95, K=256),
}


# ------------------------------------------------------------ embedding ----
@functools.lru_cache(maxsize=2)
def embed_workload(T=16384, d=1536, V=4096):
    """Synthetic error estimates g (T x d fp32, N(0,1)) and Zipf(1.1) ids."""
    g = normal(SEED_GHAT, (T, d), 1.0, False)
    ids = zipf_ids(SEED_IDS, T, V)
    return {"g": g, "ids": ids, "T": T, "d": d, "V": V}

"""Single-batch tuning by the cosine between the estimate and backprop.

The pages tune hyperparameters either by a grid search on the loss or by
maximising, on one batch, the cosine between the estimated gradient and
backprop's (Dust translation §2.3); the same cosine, measured against the
population size, follows cos(K) = c_max / sqrt(1 + c / K) (§4.2).  Both sides
of the cosine come from the library: the estimate from dust_head_estimate, the
exact gradient from dust_head_backprop.  The cosine itself is one fp64 dot
product on the device.
"""
import math

import torch

from . import head_backprop, head_estimate


def cosine(a, b):
    a = a.double().reshape(-1)
    b = b.double().reshape(-1)
    return float(torch.dot(a, b) / (torch.linalg.vector_norm(a) * torch.linalg.vector_norm(b)))


def head_cosine(logits, targets, x, sigma, K, seed, G_bp=None, draw0=0):
    """cos(estimated G_W, exact G_W) for one batch of the LM head."""
    if G_bp is None:
        _, G_bp, _ = head_backprop(logits, targets, x)
    _, G, _ = head_estimate(logits, targets, x, sigma, K, seed, draw0=draw0, want_g=False)
    return cosine(G, G_bp)


def head_sigma_sweep(logits, targets, x, sigmas, K, seed):
    """[(sigma, cosine)] over a grid of noise scales, and the sigma with the
    largest cosine (the single-batch tuning rule)."""
    _, G_bp, _ = head_backprop(logits, targets, x)
    rows = [(s, head_cosine(logits, targets, x, s, K, seed, G_bp=G_bp)) for s in sigmas]
    best = max(rows, key=lambda r: r[1])[0]
    return rows, best


def population_law(K, c, c_max=1.0):
    """The cosine law the pages fit against the population size."""
    return c_max / math.sqrt(1.0 + c / K)

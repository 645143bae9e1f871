"""Pins of the oracle's interior-layer estimator (CPU only).

- Each downstream step against an independent library routine: GELU against
  torch's exact-erf GELU, the causal EMA against scipy's IIR filter, the loss
  change against torch's float64 cross-entropy.
- Delta form: z_clean + W_head EMA(W2 dh) equals a full float64 re-forward of
  the perturbed activations (the only reason the oracle may start from the
  cached clean logits; laoyaoba.com 机制拆解 and hn.213312.xyz §2.3 say only the
  part after the perturbed layer is re-run).
- Reward: literal double sum equals the backward recurrence; segments never
  mix.
- gamma reductions in expectation (hn.213312.xyz §2.2): with gamma = 1 the
  estimate's mean is ((K-1)/K) times the backprop gradient of the sequence's
  summed loss with respect to the perturbed output; with gamma = 0.95 it is the
  gamma-discounted sum of per-token gradients.  Both references come from torch
  autograd in float64.
"""
import math

import numpy as np
import pytest
import scipy.signal
import torch

from conftest import rel_l2


def _interior_tiny(T=32, seq_len=16, d_in=6, C=16, dm=8, V=16, lam=0.9, seed=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d_in))
    W1 = rng.standard_normal((C, d_in)) / math.sqrt(d_in)
    W2 = rng.standard_normal((dm, C)) / math.sqrt(C)
    WH = rng.standard_normal((V, dm)) * 2 / math.sqrt(dm)
    y = rng.integers(0, V, T).astype(np.int32)
    y1 = (x @ W1.T).astype(np.float32)
    return dict(x=x, W1=W1, W2=W2, WH=WH, y=y, y1=y1, T=T, seq_len=seq_len, C=C, dm=dm, V=V,
                lam=lam)


def _forward_torch(y1, W2, WH, seq_len, lam):
    """Full float64 forward from y1 with torch ops: logits T x V."""
    h = torch.nn.functional.gelu(y1)
    u = h @ W2.T
    T = u.shape[0]
    es = []
    prev = None
    for t in range(T):
        if t % seq_len == 0:
            prev = torch.zeros_like(u[0])
        prev = lam * prev + (1 - lam) * u[t]
        es.append(prev)
    return torch.stack(es) @ WH.T


def test_gelu_matches_torch(orc):
    u = np.linspace(-12, 12, 20001)
    ref = torch.nn.functional.gelu(torch.tensor(u), approximate="none").numpy()
    np.testing.assert_allclose(orc.gelu(u), ref, rtol=1e-10, atol=1e-15)
    # GELU(u) - GELU(-u) = u
    np.testing.assert_allclose(orc.gelu(u) - orc.gelu(-u), u, atol=1e-13)


def test_ema_matches_iir_filter(orc):
    rng = np.random.default_rng(1)
    u = rng.standard_normal((60, 5))
    e = orc.ema(u, 20, 0.9)
    for s in range(3):
        ref = scipy.signal.lfilter([0.1], [1.0, -0.9], u[20 * s:20 * (s + 1)], axis=0)
        np.testing.assert_allclose(e[20 * s:20 * (s + 1)], ref, rtol=1e-13, atol=1e-15)


def test_ce_delta_matches_torch(orc):
    rng = np.random.default_rng(2)
    z = rng.standard_normal((7, 11)) * 3
    dz = rng.standard_normal((7, 11)) * 0.01
    y = rng.integers(0, 11, 7).astype(np.int32)
    yt = torch.tensor(y, dtype=torch.long)
    ref = (torch.nn.functional.cross_entropy(torch.tensor(z + dz), yt, reduction="none")
           - torch.nn.functional.cross_entropy(torch.tensor(z), yt, reduction="none"))
    np.testing.assert_allclose(orc.ce_delta(z, dz, y), ref.numpy(), rtol=1e-10, atol=1e-14)


def test_interior_dh(orc):
    w = _interior_tiny()
    dh = orc.interior_dh(w["y1"], 0.02, 5, 1, 3, token0=0)
    a = orc.noise(5, 1, 3, 0, w["T"], w["C"])
    y1 = torch.tensor(w["y1"].astype(np.float64))
    ref = (torch.nn.functional.gelu(y1 + 0.02 * torch.tensor(a))
           - torch.nn.functional.gelu(y1)).numpy()
    np.testing.assert_allclose(dh, ref, rtol=1e-12, atol=1e-16)


def test_delta_form_equals_full_reforward(orc):
    w = _interior_tiny()
    y1 = torch.tensor(w["y1"].astype(np.float64))
    W2 = torch.tensor(w["W2"])
    WH = torch.tensor(w["WH"])
    z_clean = _forward_torch(y1, W2, WH, w["seq_len"], w["lam"])
    yt = torch.tensor(w["y"], dtype=torch.long)
    ce0 = torch.nn.functional.cross_entropy(z_clean, yt, reduction="none")
    sigma, seed, K = 0.02, 9, 4
    dl = orc.interior_delta_loss(w["y1"], w["W2"], w["WH"], z_clean.numpy(), w["y"],
                                 w["seq_len"], w["lam"], sigma, K, seed, 1)
    for i in range(K):
        a = torch.tensor(orc.noise(seed, 1, i, 0, w["T"], w["C"]))
        zp = _forward_torch(y1 + sigma * a, W2, WH, w["seq_len"], w["lam"])
        ref = torch.nn.functional.cross_entropy(zp, yt, reduction="none") - ce0
        np.testing.assert_allclose(dl[i], ref.numpy(), rtol=1e-9, atol=1e-13)


@pytest.mark.parametrize("gamma", [0.0, 0.5, 0.95, 1.0])
def test_reward_literal_equals_recurrence(orc, gamma):
    c = np.random.default_rng(3).standard_normal((4, 30))
    r1 = orc.reward(c, gamma, 10, literal=True)
    r2 = orc.reward(c, gamma, 10)
    np.testing.assert_allclose(r1, r2, rtol=1e-12, atol=1e-13)
    # the last token of each sequence keeps only its own decrease
    np.testing.assert_array_equal(r2[:, 9::10], c[:, 9::10])


def test_reward_segments_do_not_mix(orc):
    c = np.zeros((1, 20))
    c[0, 10] = 1.0               # first token of sequence 2
    r = orc.reward(c, 0.9, 10)
    assert np.all(r[0, :10] == 0)
    assert r[0, 10] == 1.0


def _expected_grad(w, gamma):
    """sum_{s>=t, same seq} gamma^(s-t) d loss_s / d y1_t by autograd, T x C."""
    y1 = torch.tensor(w["y1"].astype(np.float64), requires_grad=True)
    z = _forward_torch(y1, torch.tensor(w["W2"]), torch.tensor(w["WH"]), w["seq_len"], w["lam"])
    ce = torch.nn.functional.cross_entropy(z, torch.tensor(w["y"], dtype=torch.long),
                                           reduction="none")
    T = w["T"]
    G = np.zeros((T, w["C"]))
    for s in range(T):
        gs, = torch.autograd.grad(ce[s], y1, retain_graph=True)
        gs = gs.numpy()
        start = (s // w["seq_len"]) * w["seq_len"]
        for t in range(start, s + 1):
            G[t] += gamma ** (s - t) * gs[t]
    return G


@pytest.mark.parametrize("gamma", [1.0, 0.95])
def test_gamma_reduction_in_expectation(orc, gamma):
    w = _interior_tiny()
    y1 = torch.tensor(w["y1"].astype(np.float64))
    z_clean = _forward_torch(y1, torch.tensor(w["W2"]), torch.tensor(w["WH"]), w["seq_len"],
                             w["lam"]).numpy()
    K = 40000
    out = orc.linear_estimate(w["x"], w["y1"], w["W2"], w["lam"], w["WH"], z_clean, w["y"],
                              w["seq_len"], 0.01, gamma, K, 2024, 1)
    ref = (K - 1) / K * _expected_grad(w, gamma)
    cos = float(np.sum(out["g"] * ref) / np.linalg.norm(out["g"]) / np.linalg.norm(ref))
    scale = float(np.sum(out["g"] * ref) / np.sum(ref * ref))
    assert cos >= 0.97, cos
    assert abs(scale - 1) < 0.05, scale

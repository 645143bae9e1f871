"""The optimiser steps and the exact head gradient on the GPU against the
fp64 oracle, and the estimate driving a short training loop."""
import numpy as np
import pytest
import torch

import workloads as W
from conftest import parity, rel_l2, to_dev

pytestmark = pytest.mark.gpu


def _state(n, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(n).astype(np.float32), rng.standard_normal(n).astype(np.float32),
            (0.1 * rng.standard_normal(n)).astype(np.float32),
            np.abs(0.01 * rng.standard_normal(n)).astype(np.float32))


def _err(a, ref):
    """Largest error over the largest magnitude, and rel-L2: the larger."""
    a = a.cpu().numpy().astype(np.float64)
    return max(float(np.max(np.abs(a - ref)) / np.max(np.abs(ref))), rel_l2(a, ref))


@pytest.mark.parametrize("n,offset", [(1_000_003, 0), (4099, 1), (4, 0), (0, 0)])
def test_sgd_matches_oracle(dust, orc, n, offset):
    """Three steps, with weight decay; offset 1 shifts every array off 16-byte
    alignment (scalar path); n = 0 is a no-op."""
    Wn, Gn, bn, _ = _state(n + offset, 5)
    Wd, Gd, bd = to_dev(Wn), to_dev(Gn), to_dev(bn)
    Wv, Gv, bv = Wd[offset:], Gd[offset:], bd[offset:]
    wbf = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    rW, rb = Wn[offset:].astype(np.float64), bn[offset:].astype(np.float64)
    lr, mu, wd = (float(np.float32(h)) for h in (0.05, 0.9, 1e-2))  # as the kernel sees them
    for _ in range(3):
        dust.sgd_step(Wv, Gv, bv, lr, momentum=mu, weight_decay=wd, W_bf16=wbf)
        rW, rb = orc.sgd_step(rW, Gn[offset:], rb, lr, mu, wd)
    torch.cuda.synchronize()
    if n == 0:
        return
    # fp32 steps against fp64 ones: a few roundings of operands of size ~1, so
    # the error is measured against the arrays' scale (elements where the
    # update cancels W have no relative accuracy to keep).
    e, eb = _err(Wv, rW), _err(bv, rb)
    assert e <= 2e-6 and eb <= 2e-6, (e, eb)
    np.testing.assert_array_equal(wbf.cpu().float().numpy(),
                                  Wv.cpu().to(torch.bfloat16).float().numpy())
    parity(W=e, momentum=eb)


@pytest.mark.parametrize("n,offset,wd", [(1_000_003, 0, 0.0), (4099, 3, 0.1)])
def test_adam_matches_oracle(dust, orc, n, offset, wd):
    Wn, Gn, mn, vn = _state(n + offset, 6)
    Wd, Gd, md, vd = to_dev(Wn), to_dev(Gn), to_dev(mn), to_dev(vn)
    Wv, Gv, mv, vv = Wd[offset:], Gd[offset:], md[offset:], vd[offset:]
    rW, rm, rv = (a[offset:].astype(np.float64) for a in (Wn, mn, vn))
    # the kernel receives its hyper-parameters as fp32: the oracle gets the same
    # values (1 - 0.999 differs by 1.3e-5 between the fp32 and fp64 betas)
    lr, b1, b2, eps, wdf = (float(np.float32(h)) for h in (1e-3, 0.9, 0.999, 1e-8, wd))
    for t in range(1, 4):
        dust.adam_step(Wv, Gv, mv, vv, t, lr, beta1=b1, beta2=b2, eps=eps, weight_decay=wdf)
        rW, rm, rv = orc.adam_step(rW, Gn[offset:], rm, rv, t, lr, b1, b2, eps, wdf)
    torch.cuda.synchronize()
    errs = [_err(a, b) for a, b in ((Wv, rW), (mv, rm), (vv, rv))]
    assert max(errs) <= 2e-6, errs
    parity(W=errs[0], m=errs[1], v=errs[2])


@pytest.mark.parametrize("T,V,d,bf16_x", [(256, 512, 64, False), (300, 4100, 40, True),
                                          (16384, 4096, 512, True)])
def test_head_backprop_matches_oracle(dust, orc, T, V, d, bf16_x):
    wl = W.head_workload(T, d, V, min(T, 2048), bf16_x, True)
    x = to_dev(wl["x"], torch.bfloat16) if bf16_x else to_dev(wl["x"])
    g, G, ws = dust.head_backprop(to_dev(wl["z"]), to_dev(wl["targets"]), x, want_g=True)
    torch.cuda.synchronize()
    assert dust.workspace_status(ws) == 0
    rows = slice(0, min(T, 512))
    ref = orc.head_backprop(wl["z"][rows], wl["targets"][rows], wl["x"][rows])
    eg = rel_l2(g[rows].cpu().numpy(), ref["g"])
    assert eg <= 1e-6, eg
    # G_W: bf16 operands, fp32 accumulation, against the fp64 product of the
    # rounded operands (all rows) and against the oracle (sampled rows' sizes).
    gb = torch.from_numpy(W.bf16_round(g.cpu().numpy())).cuda().double()
    xb = torch.from_numpy(W.bf16_round(np.asarray(wl["x"], np.float32))).cuda().double()
    eG = rel_l2(G.cpu().numpy(), (gb.T @ xb).cpu().numpy())
    assert eG <= 1e-4, eG
    if T <= 512:
        eO = rel_l2(G.cpu().numpy(), ref["G"])
        assert eO <= 5e-3, eO
    parity(g=eg, G_W_vs_g_x=eG)


def test_head_backprop_bad_target_sets_status(dust):
    z = torch.randn(4, 16, device="cuda")
    y = torch.tensor([0, 3, 99, 2], dtype=torch.int32, device="cuda")
    _, _, ws = dust.head_backprop(z, y, torch.randn(4, 8, device="cuda"))
    torch.cuda.synchronize()
    assert dust.workspace_status(ws) == 6


def _ce(z, y):
    return float(torch.nn.functional.cross_entropy(z.double(), y.long()))


@pytest.mark.parametrize("opt", ["sgd", "adam"])
def test_estimate_trains_a_head(dust, opt):
    """Closing the loop on synthetic data: a student head W fits a teacher's
    labels using only the estimator's gradient.  Each step: logits = x W^T
    on the tensor cores (the library's bf16 GEMM, with the bf16 copy of W that
    the optimiser writes), the head estimate, one optimiser step.  From ln V
    the loss must fall by 4x (the same loop on the fp64 oracle reaches 0.011
    with SGD and 0.26 with Adam after 60 steps)."""
    torch.manual_seed(0)
    T, d, V, K = 2048, 64, 256, 64
    x = torch.randn(T, d, device="cuda")
    teacher = torch.randn(V, d, device="cuda") * 0.6
    y = torch.argmax(x @ teacher.T, dim=1).to(torch.int32)
    Wt = torch.zeros(V, d, device="cuda")
    Wb = Wt.to(torch.bfloat16)
    xb = x.to(torch.bfloat16)
    m = torch.zeros_like(Wt)
    v = torch.zeros_like(Wt)
    losses = []
    for step in range(1, 61):
        z = dust.gemm_bf16(xb, False, Wb, False, T, V, d)
        losses.append(_ce(z, y))
        _, G, _ = dust.head_estimate(z, y, xb, 0.05, K, 1234, draw0=K * step, want_g=False)
        if opt == "sgd":
            dust.sgd_step(Wt, G, m, lr=2e-3, momentum=0.9, W_bf16=Wb)
        else:
            dust.adam_step(Wt, G, m, v, step, lr=2e-2, W_bf16=Wb)
    torch.cuda.synchronize()
    assert losses[0] == pytest.approx(np.log(V), rel=1e-3)
    assert losses[-1] < 0.25 * losses[0], losses[::10]


def test_tuning_cosine_rises_with_population_and_sweep_picks_best(dust):
    from activation_perturbation_es_noise_b300 import tuning
    wl = W.head_workload(256, 64, 512, 256, False, False)
    z, y, x = to_dev(wl["z"]), to_dev(wl["targets"]), to_dev(wl["x"])
    cos = [tuning.head_cosine(z, y, x, 0.05, K, 1234) for K in (64, 1024, 16384)]
    assert cos[0] < cos[1] < cos[2] and cos[2] > 0.95, cos
    rows, best = tuning.head_sigma_sweep(z, y, x, [0.01, 0.05, 0.5, 3.0], 1024, 1234)
    assert best == max(rows, key=lambda r: r[1])[0]
    # far too large a sigma leaves the linear regime: the cosine drops
    assert dict(rows)[3.0] < dict(rows)[0.05], rows
    parity(cos_K64=cos[0], cos_K1024=cos[1], cos_K16384=cos[2])


def test_es_perturb_and_estimate_match_oracle(dust, orc):
    n, K, sigma = 37, 24, 0.05
    theta = torch.randn(n, generator=torch.Generator().manual_seed(2))
    th = dust.es_perturb(theta.cuda(), sigma, K, 1234, layer=9, draw0=4)
    torch.cuda.synchronize()
    eps = orc.es_noise(n, K, 1234, 9, 4)
    want = theta.double().numpy()[None] + float(np.float32(sigma)) * eps
    assert np.abs(th.cpu().numpy() - want).max() <= 1e-6
    w = torch.randn(n, generator=torch.Generator().manual_seed(3))
    losses = (th.cpu().double() @ w.double()).float() + torch.linspace(0, 1e-3, K)
    g = dust.es_estimate(losses.cuda(), n, sigma, 1234, layer=9, draw0=4)
    torch.cuda.synchronize()
    ref = orc.es_estimate(losses.numpy(), n, float(np.float32(sigma)), 1234, 9, 4)
    e = rel_l2(g.cpu().numpy(), ref)
    assert e <= 1e-4, e  # fp32 normals (within 5e-6) and sums, as for g elsewhere
    parity(g_es=e)

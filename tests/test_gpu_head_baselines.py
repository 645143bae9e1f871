"""The head estimator with the leave-one-out and antithetic baselines on the
GPU against the fp64 oracle (oracle/baselines.py)."""
import numpy as np
import pytest
import torch

import workloads as W
from conftest import parity, rel_l2, to_dev

pytestmark = pytest.mark.gpu

G_TOL, GW_TOL = 1e-4, 5e-3


def _inputs(T, d, V, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d)).astype(np.float32)
    Wh = (rng.standard_normal((V, d)) / np.sqrt(d)).astype(np.float32)
    z = (x.astype(np.float64) @ Wh.T.astype(np.float64)).astype(np.float32)
    y = rng.integers(0, V, T).astype(np.int32)
    return x, z, y


# one-warp CTAs (V <= 1024); 256-thread CTAs; 160-thread CTAs with absent warp
# slots and the draw-chunk split (T < 1184) with its finalize kernel; tiny.
@pytest.mark.parametrize("T,d,V,K", [(256, 64, 512, 64), (64, 512, 4096, 8),
                                     (19, 16, 4100, 48), (5, 8, 7, 2)])
@pytest.mark.parametrize("baseline", [1, 2])
def test_head_baselines_match_oracle(dust, orc, T, d, V, K, baseline):
    x, z, y = _inputs(T, d, V, seed=T + V + baseline)
    g, G, ws = dust.head_estimate(to_dev(z), to_dev(y), to_dev(x), 0.05, K, 1234, 0, 3, 11,
                                  baseline=baseline)
    torch.cuda.synchronize()
    assert dust.workspace_status(ws) == 0
    fn = orc.head_estimate_leave_one_out if baseline == 1 else orc.head_estimate_antithetic
    ref = fn(z, y, x, 0.05, K, 1234, 0, 3, 11)
    eg, eG = rel_l2(g.cpu().numpy(), ref["g"]), rel_l2(G.cpu().numpy(), ref["G"])
    assert eg <= G_TOL and eG <= GW_TOL, (eg, eG)
    parity(g=eg, G_W=eG)


def test_head_antithetic_batch_shape_sampled(dust, orc):
    """The 16384 x 4096 batch with 32 antithetic pairs, as the bench times it:
    g of sampled token ranges against the oracle."""
    p = W.HEAD_PARAMS["head_batch_antithetic"]
    wl = W.head_workload(p["T"], p["d"], p["V"], p["seq_len"], p["x_bf16"], p["zipf"])
    g, G, ws = dust.head_estimate(to_dev(wl["z"]), to_dev(wl["targets"]),
                                  to_dev(wl["x"], torch.bfloat16), p["sigma"], p["K"],
                                  W.NOISE_SEED, baseline=2)
    torch.cuda.synchronize()
    assert dust.workspace_status(ws) == 0
    g = g.cpu().numpy()
    worst = 0.0
    for a in (0, 9000, 16384 - 16):
        sl = slice(a, a + 16)
        ref = orc.head_estimate_antithetic(wl["z"][sl], wl["targets"][sl], wl["x"][sl],
                                           p["sigma"], p["K"], W.NOISE_SEED, 0, 0, a)
        worst = max(worst, rel_l2(g[sl], ref["g"]))
    assert worst <= G_TOL, worst
    parity(g_sampled=worst)


def test_unknown_baseline_rejected(dust):
    z = torch.zeros(4, 8, device="cuda")
    with pytest.raises(dust.DustError):
        dust.head_estimate(z, torch.zeros(4, dtype=torch.int32, device="cuda"),
                           torch.zeros(4, 4, device="cuda"), 0.05, 4, 1, baseline=7)


# one-warp CTAs at several block counts, 160-thread CTAs (a single chunk of
# 4100 columns, absent warp slots), and the draw-split path with its finalize
@pytest.mark.parametrize("T,d,V,K,chunk", [(256, 64, 512, 64, 128), (64, 512, 4096, 16, 1024),
                                           (19, 16, 4100, 40, 820), (7, 16, 4100, 4, 4100),
                                           (5, 8, 64, 128, 16)])
def test_head_chunked_matches_oracle(dust, orc, T, d, V, K, chunk):
    x, z, y = _inputs(T, d, V, seed=T + V + chunk)
    g, G, ws = dust.head_estimate_chunked(to_dev(z), to_dev(y), to_dev(x), 0.05, K, 1234, chunk,
                                          draw0=3, token0=11)
    torch.cuda.synchronize()
    assert dust.workspace_status(ws) == 0
    ref = orc.head_estimate_chunked(z, y, x, 0.05, K, 1234, 0, chunk, 3, 11)
    eg, eG = rel_l2(g.cpu().numpy(), ref["g"]), rel_l2(G.cpu().numpy(), ref["G"])
    assert eg <= G_TOL and eG <= GW_TOL, (eg, eG)
    parity(g=eg, G_W=eG)


def test_head_chunked_with_one_chunk_equals_the_head(dust):
    x, z, y = _inputs(64, 32, 512, seed=9)
    g1, G1, _ = dust.head_estimate_chunked(to_dev(z), to_dev(y), to_dev(x), 0.05, 8, 7, 512)
    g2, G2, _ = dust.head_estimate(to_dev(z), to_dev(y), to_dev(x), 0.05, 8, 7)
    torch.cuda.synchronize()
    # the same arithmetic up to the softmax's normaliser (full-row lse here)
    assert rel_l2(g1.cpu().numpy(), g2.cpu().numpy()) <= 1e-5


def test_head_chunked_rejects_bad_shapes(dust):
    L = dust.lib()
    assert L.dust_head_chunked_workspace(16, 512, 8, 8, 100) == 0  # does not divide V
    assert L.dust_head_chunked_workspace(16, 512, 8, 6, 128) == 0  # 4 chunks do not divide K
    assert L.dust_head_chunked_workspace(16, 512, 8, 4, 128) == 0  # 1 draw per chunk
    assert L.dust_head_chunked_workspace(16, 512, 8, 8, 128) > 0

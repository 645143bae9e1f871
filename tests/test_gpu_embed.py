"""Embedding scatter-add: CUDA path against the oracle (GPU), through both
sorts: the counting pass (at most 8190 ids and 64 chunks of 1024 tokens) and
the LSD radix sort (everything else).

perm is bit-exact (the stable order of the ids is unique); G_E within
rel-L2 1e-5 (fp32 sums in a fixed order against float64).
"""
import numpy as np
import pytest
import torch

import workloads as W
from conftest import rel_l2, to_dev, parity

pytestmark = pytest.mark.gpu


def _run(dust, g, ids, V):
    G, perm, ws = dust.embed_scatter(to_dev(g), to_dev(ids), V)
    torch.cuda.synchronize()
    st = dust.workspace_status(ws)
    return G.cpu().numpy(), perm.cpu().numpy(), st


@pytest.mark.parametrize("T,d,V,kind", [
    (1000, 7, 50, "uniform"),
    (4096, 64, 4096, "zipf"),
    (3000, 33, 300, "same"),      # every token has the same id: one long run
    (1, 4, 1, "uniform"),
    (2500, 16, 70000, "uniform"), # three radix passes
    (65536, 8, 8190, "uniform"),  # the counting pass at its limits: 64 chunks, 8190 ids
    (70000, 8, 300, "zipf"),      # 69 chunks: the radix sort with few ids
    (5000, 8, 8191, "uniform"),   # one id more than the counting pass takes
])
def test_embed_shapes(dust, orc, T, d, V, kind):
    rng = np.random.default_rng(T + d)
    g = rng.standard_normal((T, d)).astype(np.float32)
    if kind == "zipf":
        ids = W.zipf_ids(3, T, V)
    elif kind == "same":
        ids = np.full(T, V - 1, np.int32)
    else:
        ids = rng.integers(0, V, T).astype(np.int32)
    G, perm, st = _run(dust, g, ids, V)
    assert st == 0
    ref_perm, ref_G = orc.embed_scatter(g, ids, V)
    np.testing.assert_array_equal(perm, ref_perm)
    e = rel_l2(G, ref_G)
    assert e <= 1e-5
    parity(G_E=e)


def test_embed_scale_config(dust, orc):
    """The scale workload: g 16384 x 1536 fp32, Zipf(1.1) ids over 4096 rows."""
    wl = W.embed_workload()
    G, perm, st = _run(dust, wl["g"], wl["ids"], wl["V"])
    assert st == 0
    ref_perm, ref_G = orc.embed_scatter(wl["g"], wl["ids"], wl["V"])
    np.testing.assert_array_equal(perm, ref_perm)
    assert rel_l2(G, ref_G) <= 1e-5
    G2, perm2, _ = _run(dust, wl["g"], wl["ids"], wl["V"])
    np.testing.assert_array_equal(G, G2)


def test_embed_empty(dust):
    g = torch.empty((0, 8), device="cuda")
    ids = torch.empty(0, dtype=torch.int32, device="cuda")
    G, perm, ws = dust.embed_scatter(g, ids, 10)
    torch.cuda.synchronize()
    assert G.abs().sum().item() == 0


def test_embed_bad_id_sets_status(dust):
    g = np.ones((10, 4), np.float32)
    ids = np.arange(10, dtype=np.int32)
    ids[3] = 99
    G, perm, st = _run(dust, g, ids, 10)
    assert st == 6
    assert G[3].sum() == 0 and G[4].sum() == 4


def test_embed_bad_id_sets_status_radix(dust):
    """The same through the radix sort (more ids than the counting pass takes)."""
    g = np.ones((10, 4), np.float32)
    ids = np.arange(10, dtype=np.int32) * 900
    ids[3] = 9999
    G, perm, st = _run(dust, g, ids, 9000)
    assert st == 6
    assert G[2700].sum() == 0 and G[3600].sum() == 4
    assert perm[-1] == 3  # the bad id sorts last


def test_embed_without_perm_output(dust):
    """perm_out = NULL gives the same rows as the call that returns it."""
    rng = np.random.default_rng(4)
    g = rng.standard_normal((700, 12)).astype(np.float32)
    ids = W.zipf_ids(2, 700, 90)
    G1, _, _ = dust.embed_scatter(to_dev(g), to_dev(ids), 90, want_perm=False)
    G2, _, _ = dust.embed_scatter(to_dev(g), to_dev(ids), 90)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(G1.cpu().numpy(), G2.cpu().numpy())

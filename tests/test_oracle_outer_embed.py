"""Pins of the oracle's outer product and embedding scatter-add (CPU only).

hn.213312.xyz Dust translation §2.2: the weight gradient is the outer product
sum_t g_t x_t^T, and with one-hot embedding inputs that outer product is a
scatter-add.  The loops are checked against numpy's float64 matmul (outer
product, and the dense one-hot product for the scatter) and the token order
against numpy's stable argsort.
"""
import numpy as np
import pytest

from conftest import rel_l2


def test_outer_matches_matmul(orc):
    rng = np.random.default_rng(0)
    g = rng.standard_normal((300, 37))
    x = rng.standard_normal((300, 11))
    G = orc.outer(g, x)
    ref = g.T @ x
    assert rel_l2(G, ref) < 1e-13
    assert G.shape == (37, 11)


def test_outer_single_token_is_rank_one(orc):
    g = np.arange(5.0)[None, :]
    x = np.array([[2.0, -1.0, 0.5]])
    np.testing.assert_array_equal(orc.outer(g, x), np.outer(g[0], x[0]))


@pytest.mark.parametrize("T,V,d", [(1000, 50, 7), (257, 4096, 3), (64, 8, 16)])
def test_scatter_equals_onehot_product(orc, T, V, d):
    import workloads
    rng = np.random.default_rng(T)
    g = rng.standard_normal((T, d))
    ids = workloads.zipf_ids(T, T, V)
    perm, GE = orc.embed_scatter(g, ids, V)
    np.testing.assert_array_equal(perm, np.argsort(ids, kind="stable"))
    onehot = np.zeros((T, V))
    onehot[np.arange(T), ids] = 1.0
    ref = onehot.T @ g
    assert rel_l2(GE, ref) < 1e-13
    absent = np.setdiff1d(np.arange(V), ids)
    assert np.all(GE[absent] == 0)


def test_scatter_order_is_ascending_t(orc):
    """Within a row the sum runs in ascending t: a cancelling sequence shows it."""
    g = np.array([[1e16], [1.0], [-1e16], [1.0]])
    ids = np.array([3, 3, 3, 3], np.int32)
    perm, GE = orc.embed_scatter(g, ids, 5)
    np.testing.assert_array_equal(perm, [0, 1, 2, 3])
    assert GE[3, 0] == ((1e16 + 1.0) - 1e16) + 1.0


def test_scatter_empty(orc):
    perm, GE = orc.embed_scatter(np.zeros((0, 4)), np.zeros(0, np.int32), 6)
    assert perm.size == 0 and np.all(GE == 0) and GE.shape == (6, 4)


def test_zipf_ids_shape_of_law():
    import workloads
    ids = workloads.zipf_ids(16, 200000, 4096)
    share0 = np.mean(ids == 0)
    p = np.arange(1, 4097) ** -1.1
    assert abs(share0 - 1 / p.sum()) < 0.005
    assert ids.min() >= 0 and ids.max() < 4096

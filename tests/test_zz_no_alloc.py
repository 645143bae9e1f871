"""The allocation-free embedding entry point (GPU).

dust_embed_scatter_static serves callers that cannot allocate device memory
where they need the embedding gradient -- for example code running under a
host framework that owns every device allocation, or a hook that runs while
the caller's memory pool is locked -- so it takes no workspace and uses a
fixed scratch array inside the library instead.

It is called here through the C ABI and must give exactly what the
workspace-taking dust_embed_scatter gives (same kernels, same fixed summation
order; checked against the tolerance the embedding tests use and bitwise), on
two calls in a row, which also shows that a call does not depend on what the
previous call left in the shared scratch.  The file sorts last so that a run
stopping at the first failure has run every other test first.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from conftest import rel_l2

pytestmark = pytest.mark.gpu


def _static_call(dust, g, ids, V):
    T, d = g.shape
    G = torch.empty((V, d), dtype=torch.float32, device="cuda")
    perm = torch.empty(T, dtype=torch.int32, device="cuda")
    st = dust.lib().dust_embed_scatter_static(
        ctypes.c_void_p(g.data_ptr()), ctypes.c_void_p(ids.data_ptr()), T, d, V,
        ctypes.c_void_p(G.data_ptr()), ctypes.c_void_p(perm.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, dust.STATUS_NAMES.get(st, st)
    torch.cuda.synchronize()
    return G.cpu().numpy(), perm.cpu().numpy()


@pytest.mark.parametrize("T,d,V,seed", [(16384, 1536, 4096, 16), (3000, 40, 700, 3)])
def test_static_scratch_matches_workspace_entry_point(dust, T, d, V, seed):
    rng = np.random.default_rng(seed)
    g = torch.from_numpy(rng.standard_normal((T, d)).astype(np.float32)).cuda()
    ids = torch.from_numpy(W.zipf_ids(seed, T, V)).cuda()
    G_ref, perm_ref, _ = dust.embed_scatter(g, ids, V)
    torch.cuda.synchronize()
    G_ref, perm_ref = G_ref.cpu().numpy(), perm_ref.cpu().numpy()
    for _ in range(2):
        G, perm = _static_call(dust, g, ids, V)
        np.testing.assert_array_equal(perm, perm_ref)
        assert rel_l2(G, G_ref) <= 1e-5
        np.testing.assert_array_equal(G, G_ref)


def test_static_scratch_rejects_oversized(dust):
    """A workspace need beyond the 32 MiB scratch is refused before any launch."""
    T, d, V = 16384, 4096, 4096
    st = dust.lib().dust_embed_scatter_static(
        ctypes.c_void_p(256), ctypes.c_void_p(256), T, d, V, ctypes.c_void_p(256), None,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 2  # DUST_ERR_UNSUPPORTED

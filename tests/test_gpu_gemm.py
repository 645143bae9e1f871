"""The tcgen05 GEMM test hook against a float64 matmul of the same bf16 values (GPU).

bf16 products are exact in fp32; only the fp32 accumulation order differs, so
the bound is a few fp32 ulps of the sum of |products|.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _ref(A, a_mn, B, b_mn):
    A64 = A.float().cpu().numpy().astype(np.float64)
    B64 = B.float().cpu().numpy().astype(np.float64)
    Am = A64.T if a_mn else A64  # M x K
    Bn = B64.T if b_mn else B64  # N x K
    return Am @ Bn.T, np.abs(Am) @ np.abs(Bn).T


@pytest.mark.parametrize("a_mn,b_mn", [(False, False), (True, True), (True, False), (False, True)])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (300, 200, 333), (1024, 512, 2048), (64, 8, 16)])
def test_gemm_majorness(dust, a_mn, b_mn, M, N, K):
    g = torch.Generator(device="cuda").manual_seed(M * 7 + N * 3 + K)
    # MN-major storage: K rows of M (N) elements, row stride padded to 8.
    def mk(rows, cols):
        ld = (cols + 7) // 8 * 8
        t = torch.randn((rows, ld), generator=g, device="cuda").to(torch.bfloat16)
        t[:, cols:] = 0
        return t, ld
    A, lda = mk(K, M) if a_mn else mk(M, K)
    B, ldb = mk(K, N) if b_mn else mk(N, K)
    Av = A[:, :M] if a_mn else A[:, :K]
    Bv = B[:, :N] if b_mn else B[:, :K]
    G = dust.gemm_bf16(A, a_mn, B, b_mn, M, N, K)
    ref, mag = _ref(Av, a_mn, Bv, b_mn)
    err = np.abs(G.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= 4e-7 * K ** 0.5 * mag + 1e-30), float((err / (mag + 1e-30)).max())

"""The CUDA noise regenerator against the oracle's own Philox (GPU).

Words must match bit for bit; normals within 5e-6 absolute: the kernels' fp32
Box-Muller (own logarithm to about 1e-7 relative, hardware sin/cos with about
4e-7 absolute error on (-pi, pi)) against the oracle's float64 one, at radii
up to sqrt(48 ln 2) = 5.77.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

CASES = [
    # seed, layer, draw, token0, ntok, nchan
    (1234, 0, 0, 0, 64, 512),
    (1234, 1, 255, 16000, 17, 2048),
    (0xDEADBEEF12345678, 7, 65535, 123456, 9, 33),
    (0, 0, 4095, 0, 3, 5),
    (0xFFFFFFFFFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF, 2**32 - 4, 4, 1),
]


@pytest.mark.parametrize("seed,layer,draw,token0,ntok,nchan", CASES)
def test_words_bit_exact(dust, orc, seed, layer, draw, token0, ntok, nchan):
    w, a = dust.philox_fill(seed, layer, draw, token0, ntok, nchan)
    got = w.cpu().numpy().view(np.uint32)
    ref = orc.noise_words(seed, layer, draw, token0, ntok, nchan)
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("seed,layer,draw,token0,ntok,nchan", CASES)
def test_normals_close(dust, orc, seed, layer, draw, token0, ntok, nchan):
    w, a = dust.philox_fill(seed, layer, draw, token0, ntok, nchan)
    ref = orc.noise(seed, layer, draw, token0, ntok, nchan)
    np.testing.assert_allclose(a.cpu().numpy().astype(np.float64), ref, rtol=0, atol=5e-6)


def test_large_fill_statistics(dust):
    """A million normals: mean, variance and the bound |a| <= sqrt(48 ln 2)."""
    _, a = dust.philox_fill(1234, 0, 3, 0, 1024, 1024)
    a = a.cpu().numpy().astype(np.float64)
    assert abs(a.mean()) < 5e-3
    assert abs(a.var() - 1.0) < 5e-3
    assert np.abs(a).max() <= np.sqrt(48 * np.log(2)) + 1e-5

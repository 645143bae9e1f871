"""Pins of the oracle's counter-based noise (CPU only).

Philox4x32-10 is pinned against an implementation the oracle does not share:
cuRAND's host-side PHILOX4_32_10 generator, called through its public C API and
compared by output only.  Black-box runs of that generator show that output
block b of a stream with word offset o is Philox4x32-10 of the 128-bit counter
whose low 64 bits are B // 65536 and whose third word is B % 65536, where
B = o / 4 + b, under the key (seed low word, seed high word).  This exercises
counter words 0-2, both key words, every round and all four output words; the
fourth counter word is compared against cuRAND's device API, run as a black
box on the GPU, in tests/test_gpu_curand_device.py.

The uniform map and Box-Muller step are pinned by exactness and by their
distribution: moments, a Kolmogorov-Smirnov test against N(0, 1), channel
independence and the bound |a| <= sqrt(2 * 24 ln 2).
"""
import ctypes
import ctypes.util
import math
import os

import numpy as np
import pytest
from scipy import stats


def _curand():
    for name in ("libcurand.so.10", "libcurand.so", "/usr/local/cuda/lib64/libcurand.so.10",
                 "/usr/local/cuda/lib64/libcurand.so"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    return None


CURAND = _curand()
CURAND_RNG_PSEUDO_PHILOX4_32_10 = 161


def curand_host_words(seed, offset_words, n_words):
    L = CURAND
    gen = ctypes.c_void_p()
    assert L.curandCreateGeneratorHost(ctypes.byref(gen), CURAND_RNG_PSEUDO_PHILOX4_32_10) == 0
    try:
        assert L.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        assert L.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(offset_words)) == 0
        out = np.zeros(n_words, np.uint32)
        assert L.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p),
                                ctypes.c_size_t(n_words)) == 0
    finally:
        L.curandDestroyGenerator(gen)
    return out.reshape(-1, 4)


def _counter_of(block):
    lo = block // 65536
    return [lo & 0xFFFFFFFF, (lo >> 32) & 0xFFFFFFFF, block % 65536, 0]


SEEDS = [1234, 0, 0xDEADBEEF12345678, 0xFFFFFFFFFFFFFFFF, 0x00000001FFFFFFFF]
OFFSET_BLOCKS = [0, 3, 65535, 65536 * 7 + 11, 65536 * (2**32 - 1) + 5, 65536 * 2**32 + 9,
                 65536 * 0x123456789A + 40000]


@pytest.mark.skipif(CURAND is None, reason="cuRAND host library not found")
@pytest.mark.parametrize("seed", SEEDS)
def test_philox_matches_curand_host(orc, seed):
    key = (seed & 0xFFFFFFFF, seed >> 32)
    for ob in OFFSET_BLOCKS:
        nblk = 64
        ref = curand_host_words(seed, 4 * ob, 4 * nblk)
        ctrs = np.array([_counter_of(ob + b) for b in range(nblk)], np.uint32)
        got = orc.philox(ctrs, key)
        np.testing.assert_array_equal(got, ref, err_msg=f"seed={seed:#x} offset block {ob}")


@pytest.mark.skipif(CURAND is None, reason="cuRAND host library not found")
def test_philox_long_stream(orc):
    """65536 consecutive blocks (the third counter word sweeps its range)."""
    seed = 0x9E3779B97F4A7C15
    ref = curand_host_words(seed, 0, 4 * 65536 * 2)
    blocks = np.arange(65536 * 2)
    ctrs = np.stack([blocks // 65536, np.zeros_like(blocks), blocks % 65536,
                     np.zeros_like(blocks)], 1).astype(np.uint32)
    got = orc.philox(ctrs, (seed & 0xFFFFFFFF, seed >> 32))
    np.testing.assert_array_equal(got, ref)


def test_noise_words_layout(orc):
    """noise_words puts word c%4 of block (c/4, token, draw, layer) at channel c."""
    seed, layer, draw, t0 = 0xABCDEF0123, 3, 17, 1000
    w = orc.noise_words(seed, layer, draw, t0, 5, 10)
    for t in range(5):
        ctrs = np.array([[j, t0 + t, draw, layer] for j in range(3)], np.uint32)
        blk = orc.philox(ctrs, (seed & 0xFFFFFFFF, seed >> 32)).reshape(-1)
        np.testing.assert_array_equal(w[t], blk[:10])


def test_layer_word_changes_stream(orc):
    a = orc.noise_words(7, 0, 0, 0, 4, 16)
    b = orc.noise_words(7, 1, 0, 0, 4, 16)
    c = orc.noise_words(7, 0, 1, 0, 4, 16)
    d = orc.noise_words(7, 0, 0, 1, 4, 16)
    assert not np.any(a == b) and not np.any(a == c)
    np.testing.assert_array_equal(a[1:], d[:3])   # token word = global token index


def test_uniform_map_exact(orc):
    """u(w) = ((w >> 9) + 0.5) 2^-23 lies in [2^-24, 1 - 2^-24] and is an fp32 value."""
    words = np.concatenate([np.array([0, 1, 511, 512, 0xFFFFFFFF, 0xFFFFFE00, 0x80000000],
                                     np.uint64),
                            np.random.default_rng(0).integers(0, 2**32, 20000, np.uint64)])
    for w in words:
        u = orc.uniform(int(w))
        assert 2.0**-24 <= u <= 1 - 2.0**-24
        assert float(np.float32(u)) == u
        assert u == ((int(w) >> 9) + 0.5) / 2**23
    assert orc.uniform(0) == 2.0**-24
    assert orc.uniform(0xFFFFFFFF) == 1 - 2.0**-24


def test_normals_distribution(orc):
    a = orc.noise(1234, 0, 0, 0, 2000, 1000).reshape(-1)   # 2e6 normals
    n = a.size
    assert abs(a.mean()) < 5 / math.sqrt(n)
    assert abs(a.var() - 1) < 5 * math.sqrt(2 / n)
    assert abs(stats.skew(a)) < 5 * math.sqrt(6 / n)
    assert abs(stats.kurtosis(a)) < 5 * math.sqrt(24 / n)
    assert stats.kstest(a, "norm").pvalue > 1e-4
    assert np.abs(a).max() <= math.sqrt(2 * 24 * math.log(2)) + 1e-12


def test_normals_channels_independent(orc):
    a = orc.noise(99, 2, 5, 0, 40000, 8)
    corr = np.corrcoef(a.T)
    off = corr[~np.eye(8, dtype=bool)]
    assert np.abs(off).max() < 5 / math.sqrt(40000)
    # each channel slot (position within a Philox block) is N(0, 1) on its own
    for q in range(8):
        assert stats.kstest(a[:, q], "norm").pvalue > 1e-4


def test_normals_draws_independent(orc):
    a0 = orc.noise(99, 1, 0, 0, 200, 512).reshape(-1)
    a1 = orc.noise(99, 1, 1, 0, 200, 512).reshape(-1)
    assert abs(np.corrcoef(a0, a1)[0, 1]) < 5 / math.sqrt(a0.size)


def test_ragged_channel_count(orc):
    """A channel count not divisible by 4 keeps the leading channels unchanged."""
    full = orc.noise(5, 0, 3, 7, 3, 12)
    part = orc.noise(5, 0, 3, 7, 3, 10)
    np.testing.assert_array_equal(full[:, :10], part)


def test_box_muller_on_words_matches_counter_normals(orc):
    """oracle.box_muller (the map on given words) equals the C oracle's normals
    of the same counters: two implementations of one map, written apart."""
    seed, layer, draw, t0, ntok, nchan = 0xABCDEF0123, 2, 9, 77, 40, 64
    w = orc.noise_words(seed, layer, draw, t0, ntok, nchan)
    a = orc.noise(seed, layer, draw, t0, ntok, nchan)
    got = orc.box_muller(w.reshape(-1, 2)).reshape(ntok, nchan)
    np.testing.assert_allclose(got, a, rtol=0, atol=1e-12)

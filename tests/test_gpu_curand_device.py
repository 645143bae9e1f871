"""The oracle's Philox against cuRAND's device-API Philox4_32_10 (GPU, run as
a black box from tests/c/curand_device_philox.cu): with subsequence
draw + layer * 2^32 and offset 4 (j + token * 2^32), the generator's first
four words are Philox4x32-10 of the counter (j, token, draw, layer) under the
key (seed low word, seed high word).  Nonzero layers exercise the fourth
counter word, which the host-API comparison (tests/test_oracle_philox.py)
cannot reach."""
import os
import subprocess

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
REC = np.dtype([("seed", "<u8"), ("layer", "<u4"), ("draw", "<u4"), ("token", "<u4"),
                ("j", "<u4")])


def test_fourth_counter_word_against_curand_device(orc, tmp_path):
    rng = np.random.default_rng(3)
    n = 4096
    rec = np.zeros(n, REC)
    rec["seed"] = rng.integers(0, 2**63, n, dtype=np.uint64) * np.uint64(2) + \
        rng.integers(0, 2, n, dtype=np.uint64)
    rec["layer"] = np.concatenate([[0, 1, 7, 0xFFFFFFFF, 0x80000000],
                                   rng.integers(0, 2**32, n - 5, dtype=np.uint64)]).astype(np.uint32)
    rec["draw"] = rng.integers(0, 2**32, n, dtype=np.uint64).astype(np.uint32)
    rec["token"] = rng.integers(0, 2**30, n, dtype=np.uint64).astype(np.uint32)
    rec["j"] = rng.integers(0, 2**32, n, dtype=np.uint64).astype(np.uint32)
    exe = tmp_path / "curand_device_philox"
    subprocess.run(["nvcc", "-O2", "-gencode", "arch=compute_103a,code=sm_103a",
                    os.path.join(ROOT, "tests", "c", "curand_device_philox.cu"), "-o", str(exe)],
                   check=True)
    rpath, wpath = tmp_path / "rec.bin", tmp_path / "words.bin"
    rec.tofile(rpath)
    r = subprocess.run([str(exe), str(rpath), str(wpath)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    got = np.fromfile(wpath, dtype=np.uint32).reshape(n, 4)
    for k in range(n):
        s = int(rec["seed"][k])
        ctr = np.array([[rec["j"][k], rec["token"][k], rec["draw"][k], rec["layer"][k]]], np.uint32)
        ref = orc.philox(ctr, (s & 0xFFFFFFFF, s >> 32))[0]
        np.testing.assert_array_equal(got[k], ref, err_msg="record %d" % k)

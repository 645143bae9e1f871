"""The C ABI from a plain C program (tests/c/abi_head.c): cudaMalloc'd
buffers, workspace queries, status codes and the status read-back, with no
Python or torch on its side.  Its results must equal, bit for bit, the same
calls made through the Python binding on the same inputs."""
import os
import subprocess

import numpy as np
import pytest
import torch

import activation_perturbation_es_noise_b300 as dust_pkg

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
T, V, D = 300, 1000, 24


def _hval(i, salt):
    x = (np.asarray(i, np.uint64) * np.uint64(2654435761)) & np.uint64(0xFFFFFFFF)
    x = x ^ ((np.uint64(salt) * np.uint64(2246822519)) & np.uint64(0xFFFFFFFF))
    x ^= x >> np.uint64(15)
    x = (x * np.uint64(2246822519)) & np.uint64(0xFFFFFFFF)
    x ^= x >> np.uint64(13)
    return (x >> np.uint64(8)).astype(np.float32) / np.float32(8388608.0) - np.float32(1.0)


def test_c_program_matches_the_binding(dust, tmp_path):
    exe = tmp_path / "abi_head"
    pkg = os.path.dirname(dust_pkg.LIB_PATH)
    subprocess.run(["nvcc", "-O2", os.path.join(ROOT, "tests", "c", "abi_head.c"), "-o", str(exe),
                    "-L" + pkg, "-ldust", "-Xlinker", "-rpath," + pkg], check=True)
    out = tmp_path / "out.bin"
    r = subprocess.run([str(exe), str(out)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    res = np.fromfile(out, dtype=np.float32)
    G_c, GE_c = res[:V * D].reshape(V, D), res[V * D:].reshape(V, D)

    z = np.float32(3.0) * _hval(np.arange(T * V), 1).reshape(T, V)
    x = _hval(np.arange(T * D), 2).reshape(T, D)
    h = _hval(np.arange(T), 3)
    y = ((h * np.float32(0.5) * np.float32(V) + np.float32(V)).astype(np.uint32) % V).astype(np.int32)
    zt, xt, yt = (torch.from_numpy(a).cuda() for a in (z, x, y))
    _, G, _ = dust.head_estimate(zt, yt, xt, 0.05, 16, 1234, want_g=False)
    GE, _, _ = dust.embed_scatter(xt, yt, V)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(G_c, G.cpu().numpy())
    np.testing.assert_array_equal(GE_c, GE.cpu().numpy())

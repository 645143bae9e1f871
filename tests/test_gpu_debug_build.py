"""The bounds-checked debug build (libdust_debug.so): every computed global
index of the CUDA-core code is checked against its buffer's extent, an index
out of range skips its access and records the source file and line.

The index check is shown to work on its own (a check that addresses nothing),
then the parity tests of every entry point run again in a child process
against the debug library; conftest fails any of them after which a checked
index was out of range, so a pass means the oracle parity holds and no
checked access left its buffer.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Parity and edge-case tests of each entry point at the oracle's small and
# ragged sizes (the full-size and statistics tests are left to the release run).
FILES = ["test_gpu_head.py", "test_gpu_head_baselines.py", "test_gpu_interior.py",
         "test_gpu_embed.py", "test_gpu_attention.py", "test_gpu_attention_qk.py",
         "test_gpu_gemm.py", "test_gpu_optim.py", "test_gpu_block.py", "test_gpu_philox.py",
         "test_gpu_failure.py"]
SKIP = ("full or batch_config or scale_config or sweep or config_sequence or large_fill "
        "or every_uniform or trains_a_head or tuning_cosine or antithetic_batch_shape")


def _child_env():
    env = dict(os.environ)
    env["DUST_LIBRARY"] = "debug"
    return env


@pytest.mark.gpu
def test_debug_library_records_an_out_of_range_index():
    if os.environ.get("DUST_LIBRARY") == "debug":
        pytest.skip("runs from the release test session")
    code = r"""
import activation_perturbation_es_noise_b300 as d
assert d.debug_build()
assert d.debug_fault() is None
assert d.debug_check_index(5, 6)
assert d.debug_fault() is None
assert not d.debug_check_index(6, 6)
assert not d.debug_check_index(-1, 6)
f = d.debug_fault()
assert f is not None and f[0] == 10 and f[1] > 0, f
assert d.debug_fault() is None  # reading cleared it
print("ok")
"""
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=_child_env(),
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr


@pytest.mark.gpu
def test_release_library_is_not_the_debug_build(dust):
    if os.environ.get("DUST_LIBRARY") == "debug":
        pytest.skip("runs from the release test session")
    assert not dust.debug_build()
    assert dust.debug_check_index(7, 6)  # the release check is the constant true
    assert dust.debug_fault() is None


@pytest.mark.gpu
def test_parity_tests_pass_under_the_debug_build():
    if os.environ.get("DUST_LIBRARY") == "debug":
        pytest.skip("runs from the release test session")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-k", "not (%s)" % SKIP,
           "-p", "no:cacheprovider"] + [os.path.join("tests", f) for f in FILES]
    r = subprocess.run(cmd, cwd=ROOT, env=_child_env(), capture_output=True, text=True,
                       timeout=1500)
    tail = "\n".join((r.stdout + r.stderr).splitlines()[-30:])
    assert r.returncode == 0, tail
    assert " passed" in tail and "error" not in tail.lower(), tail

"""Build the engine's shared libraries in the package directory: libdust.so
and its bounds-checked twin libdust_debug.so (-DDUST_DEBUG).

Every .cu under csrc/ is compiled for sm_103a only (B300) and linked with the
static CUDA runtime, so the library needs nothing but the NVIDIA driver at run
time.  Run from anywhere:  python -m activation_perturbation_es_noise_b300.build
"""
import concurrent.futures
import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(os.path.dirname(HERE), "_build")
LIB = os.path.join(HERE, "libdust.so")
LIB_DEBUG = os.path.join(HERE, "libdust_debug.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr", "-diag-suppress", "177"]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh")) +
                               glob.glob(os.path.join(CSRC, "*.h")) +
                               [os.path.join(os.path.dirname(HERE), "include", "dust.h")])


def _stale(lib):
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _deps() + [os.path.abspath(__file__)])


def _compile(src, verbose, build_dir, extra):
    obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
    cmd = ([NVCC] + ARCH + FLAGS + extra + (["-Xptxas", "-v"] if verbose else []) +
           ["-c", src, "-o", obj])
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, r.stdout, r.stderr))
    return obj, r.stderr


def _link(lib, build_dir, extra, verbose):
    os.makedirs(build_dir, exist_ok=True)
    srcs = _sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose, build_dir, extra), srcs))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    objs = [o for o, _ in results]
    tmp = lib + ".tmp"
    cmd = [NVCC] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, lib)


def build(force=False, verbose=False):
    """Compile csrc/*.cu into libdust.so and the bounds-checked libdust_debug.so
    (-DDUST_DEBUG); returns the release library's path."""
    if force or _stale(LIB):
        _link(LIB, BUILD, [], verbose)
    if force or _stale(LIB_DEBUG):
        _link(LIB_DEBUG, os.path.join(BUILD, "debug"), ["-DDUST_DEBUG"], verbose)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

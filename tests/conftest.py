import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: long CPU test")


def parity(**errors):
    """Prints the measured errors of a parity check on one line (shown with
    pytest -s), so that a run reports the margins, not only pass/fail."""
    name = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    print("PARITY %s %s" % (name, " ".join("%s=%.3e" % kv for kv in errors.items())))


def rel_l2(a, b):
    import numpy as np
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.lib()
    return oracle


@pytest.fixture(scope="session")
def dust():
    """The engine's Python binding with libdust.so loaded (GPU tests only)."""
    import torch
    import activation_perturbation_es_noise_b300 as d
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected without a CUDA device")
    d.lib()
    return d


def to_dev(a, dtype=None):
    import numpy as np
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


@pytest.fixture(autouse=True)
def _debug_build_faults(request):
    """Under DUST_LIBRARY=debug (the bounds-checked library) every GPU test
    also fails if a checked index went out of range while it ran."""
    yield
    if os.environ.get("DUST_LIBRARY") == "debug" and request.node.get_closest_marker("gpu"):
        import activation_perturbation_es_noise_b300 as d
        if d._lib is not None:
            fault = d.debug_fault()
            assert fault is None, "index out of range in csrc file id %d, line %d" % fault

"""Failure detection on the GPU without a fault (GPU).

Every wait inside the library's kernels is bounded: when it runs out the kernel
records DUST_ERR_TIMEOUT in the workspace status word and returns, and the
context stays usable.  The check here waits on a barrier that nothing sets,
with a 1 ms limit.  Device-side range errors are covered in the head and
embedding tests; host-side argument errors in test_abi.py.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(dust):
    assert dust.wait_selftest(1_000_000) == 5  # DUST_ERR_TIMEOUT
    # the context is still usable: a normal call afterwards succeeds
    w, a = dust.philox_fill(1234, 0, 0, 0, 4, 8)
    torch.cuda.synchronize()
    assert torch.isfinite(a).all()


def test_wait_selftest_rejects_bad_limits(dust):
    with pytest.raises(dust.DustError):
        dust.wait_selftest(0)

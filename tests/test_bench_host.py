"""Host-side logic of bench.py's timing rules (no GPU): how each workload keeps
a step's inputs out of L2."""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402


def _wl(nbytes, **kw):
    return dict({"host": {"a": np.zeros(nbytes // 4, np.float32)}}, **kw)


def test_large_inputs_need_no_flush():
    wl = _wl(bench.L2_BYTES + 4096)
    assert bench.l2_mode(wl) == "large"
    assert "no flush" in bench.l2_label(wl)


def test_small_inputs_are_flushed():
    wl = _wl(1 << 20)
    assert bench.l2_mode(wl) == "flush"
    assert "flushed" in bench.l2_label(wl)


def test_rotated_inputs_exceed_l2():
    wl = _wl(100 << 20, rotate=3)
    assert bench.l2_mode(wl) == "rotate"
    assert 3 * bench.input_bytes(wl) > bench.L2_BYTES
    assert "3 input sets" in bench.l2_label(wl)


def test_embedding_workload_rotates_past_l2():
    import workloads as W
    e = W.embed_workload()
    wl = {"host": {"g": e["g"], "ids": e["ids"]}, "rotate": 3}
    assert bench.input_bytes(wl) < bench.L2_BYTES  # one set alone would stay in L2
    assert bench.l2_mode(wl) == "rotate"
    assert wl["rotate"] * bench.input_bytes(wl) > 2 * bench.L2_BYTES

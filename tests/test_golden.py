"""The oracle still reproduces its committed micro fixtures (CPU only)."""
import json
import os

import numpy as np

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(HERE, name + ".json")) as f:
        return json.load(f)


def test_micro_philox(orc):
    g = _load("micro_philox")
    ctrs = np.array(g["counters"], np.uint32)
    for key, words in zip(g["keys"], g["words"]):
        np.testing.assert_array_equal(orc.philox(ctrs, key), np.array(words, np.uint32))


def test_micro_head(orc):
    g = _load("micro_head")
    out = orc.head_estimate(np.array(g["z"], np.float32), np.array(g["targets"], np.int32),
                            np.array(g["x"], np.float32), g["sigma"], g["K"], g["seed"],
                            g["layer"])
    for k in ("dl", "g", "G"):
        np.testing.assert_allclose(out[k], np.array(g[k]), rtol=1e-12, atol=1e-15)


def test_micro_interior(orc):
    g = _load("micro_interior")
    f32 = lambda k: np.array(g[k], np.float32)
    out = orc.linear_estimate(f32("x"), f32("y1"), f32("W2"), g["lam"], f32("W_head"),
                              f32("z_clean"), np.array(g["targets"], np.int32), g["seq_len"],
                              g["sigma"], g["gamma"], g["K"], g["seed"], g["layer"])
    for k in ("dl", "g", "G"):
        np.testing.assert_allclose(out[k], np.array(g[k]), rtol=1e-11, atol=1e-15)

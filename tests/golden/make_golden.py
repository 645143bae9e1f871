"""Write the oracle's outputs on micro cases to tests/golden/*.json.

These fixtures are regression anchors for the oracle itself: they are written
by this script, which calls only oracle/, and a later change of the oracle's
arithmetic shows up as a mismatch.  The pages print no worked numeric example
of the estimator (hn.213312.xyz Dust translation §2.2 gives the formulas only),
so no fixture here comes from the pages.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import math
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402


def micro_head():
    rng = np.random.default_rng(20261202)
    T, V, d = 4, 8, 3
    x = rng.standard_normal((T, d)).astype(np.float32)
    z = rng.standard_normal((T, V)).astype(np.float32)
    y = rng.integers(0, V, T).astype(np.int32)
    out = oracle.head_estimate(z, y, x, 0.05, 6, 1234, 0)
    return {"T": T, "V": V, "d": d, "sigma": 0.05, "K": 6, "seed": 1234, "layer": 0,
            "x": x.tolist(), "z": z.tolist(), "targets": y.tolist(),
            "dl": out["dl"].tolist(), "g": out["g"].tolist(), "G": out["G"].tolist()}


def micro_philox():
    ctrs = np.array([[0, 0, 0, 0], [1, 2, 3, 4], [0xFFFFFFFF] * 4, [7, 1000, 63, 1]], np.uint32)
    keys = [(1234, 0), (0xDEADBEEF, 0x12345678)]
    return {"counters": ctrs.tolist(), "keys": keys,
            "words": [oracle.philox(ctrs, k).tolist() for k in keys]}


def micro_interior():
    rng = np.random.default_rng(7)
    T, seq_len, C, dm, V, d_in = 8, 4, 8, 4, 8, 3
    x = rng.standard_normal((T, d_in)).astype(np.float32)
    y1 = rng.standard_normal((T, C)).astype(np.float32)
    W2 = (rng.standard_normal((dm, C)) / math.sqrt(C)).astype(np.float32)
    WH = (rng.standard_normal((V, dm)) / math.sqrt(dm)).astype(np.float32)
    z = rng.standard_normal((T, V)).astype(np.float32)
    y = rng.integers(0, V, T).astype(np.int32)
    out = oracle.linear_estimate(x, y1, W2, 0.9, WH, z, y, seq_len, 0.02, 0.95, 5, 99, 1)
    return {"T": T, "seq_len": seq_len, "C": C, "d_model": dm, "V": V, "d_in": d_in,
            "lam": 0.9, "sigma": 0.02, "gamma": 0.95, "K": 5, "seed": 99, "layer": 1,
            "x": x.tolist(), "y1": y1.tolist(), "W2": W2.tolist(), "W_head": WH.tolist(),
            "z_clean": z.tolist(), "targets": y.tolist(),
            "dl": out["dl"].tolist(), "g": out["g"].tolist(), "G": out["G"].tolist()}


if __name__ == "__main__":
    for name, fn in [("micro_head", micro_head), ("micro_philox", micro_philox),
                     ("micro_interior", micro_interior)]:
        with open(os.path.join(HERE, name + ".json"), "w") as f:
            json.dump(fn(), f, indent=0)
        print("wrote", name)

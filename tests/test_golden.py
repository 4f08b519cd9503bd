"""The frozen worked example (tests/golden/worked_example.json).

Its closed-form entries are checked against the mathematics directly: the
first output has pre-activation exactly 1 (1/16 + 1/2*1 - 1/4*(-1) + 1/8*1/2 +
1*1/8), so it is SiLU(1); channels with zero input give SiLU(bias); the state
written is the last three raw inputs (FlashInfer causal_conv1d_fn, conv_state)
with position 3 untouched.  The whole fixture is then a regression pin of the
oracle.
"""
import json
import math
import os

import numpy as np

from tests.golden import make_golden

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _silu(z):
    return z / (1.0 + math.exp(-z))


def test_golden_closed_forms():
    doc = json.load(open(os.path.join(HERE, "worked_example.json")))["results"]
    assert doc["out_c0"][0] == _silu(1.0)
    assert all(v == _silu(1.0 / 16) for v in doc["out_c1"])
    assert doc["state_c0"] == [0.5, 0.625, 0.75, 7.0]
    # dbias with dy = 1 is the sum of SiLU'(z) over the six tokens
    hist = [1.0, -1.0, 0.5] + [(t + 1) / 8.0 for t in range(6)]
    w = [0.5, -0.25, 0.125, 1.0]
    zs = [1.0 / 16 + sum(w[k] * hist[j + k] for k in range(4)) for j in range(6)]
    dsilu = [1 / (1 + math.exp(-z)) * (1 + z * (1 - 1 / (1 + math.exp(-z)))) for z in zs]
    assert math.isclose(doc["dbias_c0"], sum(dsilu), rel_tol=1e-13)


def test_golden_regression():
    doc = json.load(open(os.path.join(HERE, "worked_example.json")))["results"]
    now = make_golden.run(make_golden.example())
    for k, v in doc.items():
        np.testing.assert_allclose(np.asarray(now[k]), np.asarray(v), rtol=1e-14, atol=0)

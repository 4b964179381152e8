"""The oracle still reproduces its committed fixture on the tiny workload."""
import json
import math
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))

import make_golden  # noqa: E402


def test_tiny_layer_fixture():
    with open(os.path.join(HERE, "golden", "oracle_tiny_layer.json")) as f:
        want = json.load(f)
    got = make_golden.compute()
    for key in ("out_sum", "out_abs_sum", "y13_abs_sum"):  # float sums: summation order may vary
        assert math.isclose(got.pop(key), want.pop(key), rel_tol=1e-12)
    assert got == want


def test_tiny_shard_fixture():
    with open(os.path.join(HERE, "golden", "oracle_tiny_shard.json")) as f:
        want = json.load(f)
    got = make_golden.compute_shard()
    for key in ("out_sum", "out_abs_sum"):
        assert math.isclose(got.pop(key), want.pop(key), rel_tol=1e-12)
    assert got == want

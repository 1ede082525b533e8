"""Regression of the oracle against its own committed fixture on the tiny
workload (tests/golden/tiny_oracle.json, written by make_golden.py).  This
guards the oracle against accidental change, e.g. between the x86 host and
the Arm GPU host; its correctness is pinned by test_oracle_pins.py."""
import json
import os

import numpy as np

from tests.golden.make_golden import compute

HERE = os.path.dirname(os.path.abspath(__file__))


def test_tiny_matches_fixture():
    with open(os.path.join(HERE, "golden", "tiny_oracle.json")) as f:
        want = json.load(f)
    got = compute()
    assert got["state_indices"] == want["state_indices"]
    np.testing.assert_allclose([float.fromhex(x) for x in got["out_sample"]],
                               [float.fromhex(x) for x in want["out_sample"]], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose([float.fromhex(x) for x in got["states_sample"]],
                               [float.fromhex(x) for x in want["states_sample"]], rtol=1e-12, atol=1e-15)
    assert abs(got["out_bf16_sum"] - want["out_bf16_sum"]) <= 4
    np.testing.assert_allclose(float.fromhex(got["pool_written_f32_sum"]),
                               float.fromhex(want["pool_written_f32_sum"]), rtol=1e-9)

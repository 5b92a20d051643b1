"""Regression pin: the oracle still reproduces its stored values on the tiny decode workload.

The fixture was written by tests/golden/make_golden.py, which calls only the oracle and the
seeded generator.  A change to either shows up here first.
"""

import json
import os

import numpy as np

from tests.golden.make_golden import tiny_decode

HERE = os.path.dirname(os.path.abspath(__file__))


def test_tiny_decode_golden():
    with open(os.path.join(HERE, "golden", "tiny_decode_oracle.json")) as f:
        gold = json.load(f)
    now = tiny_decode()
    assert now["input_sha256"] == gold["input_sha256"], "seeded generator changed"
    assert now["q_rot_bits"] == gold["q_rot_bits"]
    assert now["k_cache_sha256"] == gold["k_cache_sha256"]
    assert now["v_cache_sha256"] == gold["v_cache_sha256"]
    assert np.max(np.abs(np.array(now["out"]) - np.array(gold["out"]))) < 1e-14

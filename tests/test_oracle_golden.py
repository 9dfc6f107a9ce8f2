"""The oracle still reproduces its frozen small-case outputs (regression guard)."""
import json
import os

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))

import sys  # noqa: E402
sys.path.insert(0, os.path.join(HERE, "golden"))
import make_golden  # noqa: E402

with open(os.path.join(HERE, "golden", "oracle_small_cases.json")) as f:
    _CASES = json.load(f)["cases"]


@pytest.mark.parametrize("case", _CASES, ids=lambda c: c["name"])
def test_oracle_reproduces_frozen_outputs(case):
    assert make_golden.compute(case) == case["expected"]

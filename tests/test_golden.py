"""Regression of the oracle against its stored small cases.

The fixtures were written by tests/golden/make_golden.py from the oracle; the
inputs are closed-form patterns.  A change of the oracle's arithmetic shows up
here and must cite the passage (or its reading) that justifies it.
"""
import json
import os

import numpy as np
import pytest

from oracle import muon_step

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
CASES = json.load(open(os.path.join(HERE, "oracle_small_cases.json")))["cases"]


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_oracle_matches_stored_case(case):
    a, b, c = case["coeffs"]
    out = muon_step(np.array(case["W"]), np.array(case["G"]),
                    np.array(case["M"]), lr=case["lr"], beta=case["beta"],
                    nesterov=case["nesterov"], ns_steps=case["ns_steps"],
                    a=a, b=b, c=c, mode=case["mode"], nb=case["nb"],
                    eps=case["eps"])
    for k, key in (("W", "W_new"), ("M", "M_new"), ("O", "O")):
        assert np.allclose(out[k], np.array(case[key]), rtol=0, atol=1e-13)

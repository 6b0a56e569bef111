"""Oracle regression against the fixture written by tests/golden/make_golden.py."""
import json
import math
import os

import numpy as np

from tests.golden.make_golden import build

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_oracle_matches_stored_regression_values():
    with open(os.path.join(HERE, "oracle_regression.json")) as f:
        stored = json.load(f)
    now = build()
    for key, val in stored.items():
        if key == "inputs":
            continue
        if "bits" in key or "codes" in key or "ids" in key:
            assert now[key] == val, key
        else:
            # Same platform family: libm may differ in the last ulp, nothing more.
            np.testing.assert_allclose(now[key], val, rtol=1e-13, atol=1e-300, err_msg=key)
    assert not math.isnan(sum(stored["score_t1_c60_70"][:9]))

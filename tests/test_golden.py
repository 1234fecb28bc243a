"""The oracle still reproduces the stored fixtures written by tests/golden/make_golden.py."""
import json
import os

import numpy as np
import pytest

from tests.golden.make_golden import CASES, golden

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.mark.parametrize("name", sorted(CASES))
def test_oracle_matches_stored_fixture(name):
    with open(os.path.join(HERE, name + ".json")) as f:
        stored = json.load(f)
    now = golden(CASES[name])
    assert now["blob_sha256"] == stored["blob_sha256"]
    assert [s[:2] for s in now["y_samples"]] == [s[:2] for s in stored["y_samples"]]
    got = [float.fromhex(s[2]) for s in now["y_samples"]] + [float.fromhex(v) for v in now["y_row_abs_sums"]]
    want = [float.fromhex(s[2]) for s in stored["y_samples"]] + [float.fromhex(v) for v in stored["y_row_abs_sums"]]
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=0)

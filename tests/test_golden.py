"""The oracle still computes the stored results of tests/golden/oracle_regression.json."""
import json
import os

import numpy as np

from tests.golden.make_golden import OUT, compute


def test_oracle_matches_stored_results():
    stored = json.load(open(OUT))
    now = compute()
    assert set(stored) == set(now)
    for name, ref in stored.items():
        got = now[name]
        assert got["n"] == ref["n"] and got["positions"] == ref["positions"], name
        for key in ("sum", "sumsq"):
            assert np.isclose(got[key], ref[key], rtol=1e-10, atol=1e-10), (name, key)
        assert np.allclose(got["samples"], ref["samples"], rtol=1e-10, atol=1e-12), name

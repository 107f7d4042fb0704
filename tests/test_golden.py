"""The oracle against its stored outputs (tests/golden/oracle_small.json, written by
tests/golden/make_golden.py from the oracle alone): a guard against silent changes to the
oracle's arithmetic.  Its independent pins are tests/test_oracle*.py."""
import json
import os
import sys

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))
import make_golden  # noqa: E402

with open(os.path.join(HERE, "golden", "oracle_small.json")) as f:
    GOLDEN = json.load(f)


@pytest.mark.parametrize("i", range(len(make_golden.CASES)))
def test_oracle_reproduces_its_stored_outputs(i):
    c = make_golden.CASES[i]
    got = make_golden.run_case(*c, seed=500 + i)
    want = GOLDEN[c[0]]
    assert np.array_equal(np.isfinite(got["lse"]), np.asarray(want["lse_finite"]))
    for k in ("O", "lse", "dQ", "dK", "dV", "dbias", "ddense"):
        g = np.where(np.isfinite(got[k]), got[k], 0.0)
        assert np.allclose(g, np.asarray(want[k]), atol=1e-13, rtol=1e-12), k

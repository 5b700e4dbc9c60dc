"""The oracle on hand-worked examples (tests/golden/worked_examples.json):
each stored spectrum is a closed form derived by hand, evaluated here in
50-digit arithmetic, never a solver's output.  CPU only."""
import json
import os

import numpy as np
import pytest

import oracle
from tests import helpers as H

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "worked_examples.json")
with open(GOLDEN) as fh:
    DATA = json.load(fh)


def _eval(expr):
    import mpmath as mp
    mp.mp.dps = 50
    return float(mp.mpf(eval(expr, {"sqrt": mp.sqrt, "__builtins__": {}})))


@pytest.mark.parametrize("dt", [np.float32, np.float64])
@pytest.mark.parametrize("case", DATA["cases"], ids=lambda c: c["name"])
def test_worked_spectra(case, dt):
    d = np.array([case["d"]], dtype=dt)
    e = np.array([case["e"]], dtype=dt)
    n = d.shape[1]
    want = np.array([_eval(x) for x in case["lam"]])
    r = oracle.steqr(d, e, jobz=True)
    assert r.info[0] == 0
    tn = float(H.norm1(d, e)[0])
    assert np.max(np.abs(r.lam[0].astype(np.float64) - want)) <= H.lam_tol(n, dt, tn)
    res, orth = H.residual_orth(d, e, r.lam, r.Q)
    assert res[0] <= 64 * n * H.eps_of(dt) * tn and orth[0] <= 64 * n * H.eps_of(dt)


@pytest.mark.parametrize("dt", [np.float32, np.float64])
@pytest.mark.parametrize("case", DATA["leaf_cases"], ids=lambda c: c["name"])
def test_worked_leaf_tear(case, dt):
    d = np.array([case["d"]], dtype=dt)
    e = np.array([case["e"]], dtype=dt)
    r = oracle.stedc_leaves(d, e, case["leaf"], jobz=True)
    assert np.array_equal(r.d_torn[0], np.array(case["d_torn"], dtype=dt))   # integers: exact
    want = np.array([_eval(x) for x in case["lam"]])
    for s, m in zip(r.starts, r.sizes):
        tn = float(H.norm1(r.d_torn[:, s:s + m], e[:, s:s + m - 1])[0])
        got = r.lam[0, s:s + m].astype(np.float64)
        assert np.max(np.abs(got - want[s:s + m])) <= H.lam_tol(m, dt, tn)

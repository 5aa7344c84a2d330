"""Stored oracle values (tests/golden/, written by tests/golden/make_golden.py) still hold."""
import json
import os

import numpy as np

import oracle
from exact_io_aware_34_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "n256_d64_oracle.json")


def test_n256_golden():
    g = json.load(open(GOLDEN))
    w = inputs.workload("n256_d64")
    q, k, v, scale = inputs.make_inputs(w)
    assert inputs.sha256_of(q, k, v) == g["inputs_sha256"]
    Q, K, V = (x.float().numpy().astype(np.float64) for x in (q, k, v))
    O, L = oracle.attention(Q, K, V, scale)
    np.testing.assert_allclose(L[0, 0], g["lse"], rtol=0, atol=1e-12)
    for r, row in g["o_rows"].items():
        np.testing.assert_allclose(O[0, 0, int(r)], row, rtol=0, atol=1e-13)
    assert abs(O.sum() - g["o_sum"]) < 1e-9
    assert abs(np.abs(O).sum() - g["o_abs_sum"]) < 1e-9

"""Drift guard: the oracle still reproduces its own committed summary of the
tiny fp32 workload (written by tests/golden/make_golden.py, oracle only)."""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))

import make_golden  # noqa: E402


def test_tiny_golden_summary():
    with open(os.path.join(HERE, "golden", "tiny_fp32_oracle.json")) as f:
        want = json.load(f)
    got = make_golden.compute()
    assert got["ce_argmax"] == want["ce_argmax"]
    for key in ("Y_l2", "Y_sum", "dX_l2", "lse_sum", "ce_loss", "ce_dX_l2", "ce_dW_l2"):
        np.testing.assert_allclose(got[key], want[key], rtol=1e-12, err_msg=key)
    for k, v in want["grad_l2"].items():
        np.testing.assert_allclose(got["grad_l2"][k], v, rtol=1e-12, err_msg=k)

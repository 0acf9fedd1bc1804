"""Regression fixture: the oracle still reproduces the values it stored.

The pages print no worked example, so this fixture is written by
tests/golden/make_golden.py (oracle only); it guards the oracle against silent
changes, while tests/oracle_pins.py pins its correctness.
"""
import json
import os

import numpy as np

from oracle import attn_oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "tiny_gqa_s4_d4.json")


def test_golden_fixture():
    g = json.load(open(GOLDEN))
    inp = {k: np.array(v) for k, v in g["inputs"].items()}
    for name, causal in (("full", False), ("causal", True)):
        r = attn_oracle.mha_backward(inp["q"], inp["k"], inp["v"], inp["do"], g["scale"], causal)
        for key, val in g["cases"][name].items():
            np.testing.assert_allclose(np.asarray(r[key]), np.array(val), rtol=1e-12, atol=1e-13)

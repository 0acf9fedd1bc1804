"""Writes the stored oracle outputs under tests/golden/ (calls only oracle/).

Run from the repository root:  python tests/golden/make_golden.py
The inputs are small exact binary fractions listed in the file itself, so the
fixture does not depend on any random generator.
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle import attn_oracle  # noqa: E402


def tiny_inputs():
    # B=1, Sq=Sk=4, Hq=2, Hk=1 (one GQA group of two query heads), D=4
    idx = np.arange(1 * 4 * 2 * 4).reshape(1, 4, 2, 4)
    q = ((idx * 7) % 11 - 5) / 4.0
    do = ((idx * 5) % 9 - 4) / 8.0
    kidx = np.arange(1 * 4 * 1 * 4).reshape(1, 4, 1, 4)
    k = ((kidx * 3) % 7 - 3) / 4.0
    v = ((kidx * 11) % 13 - 6) / 4.0
    return q, k, v, do


def main():
    q, k, v, do = tiny_inputs()
    out = {"inputs": {"q": q.tolist(), "k": k.tolist(), "v": v.tolist(), "do": do.tolist()},
           "scale": 0.5, "cases": {}}
    for causal in (False, True):
        r = attn_oracle.mha_backward(q, k, v, do, 0.5, causal)
        out["cases"]["causal" if causal else "full"] = {
            key: np.asarray(r[key]).tolist() for key in ("O", "LSE", "Delta", "dQ", "dK", "dV")}
    path = os.path.join(ROOT, "tests", "golden", "tiny_gqa_s4_d4.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()

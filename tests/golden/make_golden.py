"""Writes the oracle regression fixture ``oracle_t37_c16.json``.

Calls only ``oracle/`` (and NumPy's seeded generator for the inputs).  Run
from the repository root:  python tests/golden/make_golden.py
The fixture pins the oracle against accidental change; its values are the
oracle's own, so it is a regression guard, not an independent pin.
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402


def main():
    rng = np.random.default_rng(2024)
    B, T, Hk, Hv, Dk, Dv = 1, 37, 1, 2, 8, 6
    q = rng.standard_normal((B, T, Hk, Dk))
    k = rng.standard_normal((B, T, Hk, Dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, Hv, Dv))
    g = rng.uniform(0.5, 1.0, (B, T, Hv))
    beta = rng.uniform(0.0, 1.0, (B, T, Hv))
    s0 = rng.standard_normal((B, Hv, Dv, Dk)) * 0.3
    y, s = oracle.gdn_sequential(q, k, v, g, beta, s0)
    fx = {"written_by": "tests/golden/make_golden.py (oracle.gdn_sequential)",
          "shape": {"B": B, "T": T, "Hk": Hk, "Hv": Hv, "Dk": Dk, "Dv": Dv},
          "inputs": {"q": q.tolist(), "k": k.tolist(), "v": v.tolist(),
                     "g": g.tolist(), "beta": beta.tolist(), "s0": s0.tolist()},
          "y": y.tolist(), "s": s.tolist()}
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)),
                           "oracle_t37_c16.json"), "w") as f:
        json.dump(fx, f)


if __name__ == "__main__":
    main()

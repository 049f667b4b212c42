"""Writes the oracle regression fixtures in this folder.

Every stored value is produced here by the float64 oracle alone; inputs are
deterministic closed-form patterns (no random generator), so the fixture can
be re-derived on any machine:  python tests/golden/make_golden.py
The pages ("Advancing Emerging Optimizers for Accelerated LLM Training" and
its summaries) print no worked example, so no value here is the pages' own.
"""
import json
import math
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

from oracle import muon_step  # noqa: E402

COEFFS = (3.4445, -4.7750, 2.0315)


def pattern(rows, cols, k):
    return np.array([[math.sin(0.37 * (i + 1) * k + 0.11 * (j + 1) * (k + 2))
                      for j in range(cols)] for i in range(rows)])


def case(name, rows, cols, mode="full", nb=1, nesterov=True):
    W = 0.02 * pattern(rows, cols, 1)
    G = pattern(rows, cols, 2)
    M = 0.5 * pattern(rows, cols, 3)
    out = muon_step(W, G, M, lr=0.02, beta=0.95, nesterov=nesterov,
                    ns_steps=5, a=COEFFS[0], b=COEFFS[1], c=COEFFS[2],
                    mode=mode, nb=nb)
    return {"name": name, "rows": rows, "cols": cols, "mode": mode, "nb": nb,
            "nesterov": nesterov, "lr": 0.02, "beta": 0.95, "ns_steps": 5,
            "coeffs": list(COEFFS), "eps": 1e-7,
            "W": W.tolist(), "G": G.tolist(), "M": M.tolist(),
            "W_new": out["W"].tolist(), "M_new": out["M"].tolist(),
            "O": out["O"].tolist()}


def main():
    cases = [case("wide_8x16", 8, 16), case("tall_16x8", 16, 8),
             case("square_8x8_plain", 8, 8, nesterov=False),
             case("blockwise_8x16_nb2", 8, 16, mode="blockwise", nb=2)]
    with open(os.path.join(HERE, "oracle_small_cases.json"), "w") as f:
        json.dump({"source": "oracle/muon_ref.py via make_golden.py",
                   "cases": cases}, f, indent=0)


if __name__ == "__main__":
    main()

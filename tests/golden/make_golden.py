"""Writes tests/golden/tiny_step.json: a tiny Muon step computed by the oracle.

The inputs are small seeded values rounded to bfloat16 (so they are exact in
every storage type the library accepts); the expected outputs come from the
fp64 oracle in oracle/ and nothing else. Run from the repository root:
    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))
from oracle import muon_ref as ref  # noqa: E402

SHAPES = [(3, 5), (6, 2), (4, 4), (1, 7)]
HYPER = dict(lr=0.02, mu=0.95, nesterov=True, ns_steps=5, coeffs=list(ref.DEFAULT_COEFFS), eps=1e-7)


def main():
    rng = np.random.default_rng(20261202)
    cases = []
    for r, c in SHAPES:
        W = ref.round_to_dtype(rng.standard_normal((r, c)), "bf16")
        G = ref.round_to_dtype(rng.standard_normal((r, c)), "bf16")
        M = ref.round_to_dtype(0.5 * rng.standard_normal((r, c)), "bf16")
        W2, M2, X = ref.muon_step(W, G, M, lr=HYPER["lr"], mu=HYPER["mu"], nesterov=HYPER["nesterov"],
                                  ns_steps=HYPER["ns_steps"], coeffs=tuple(HYPER["coeffs"]), eps=HYPER["eps"])
        cases.append({"shape": [r, c], "W": W.tolist(), "G": G.tolist(), "M": M.tolist(),
                      "W_new": W2.tolist(), "M_new": M2.tolist(), "X": X.tolist()})
    out = {
        "source": "fp64 oracle (oracle/muon_ref.py) via tests/golden/make_golden.py; inputs seeded, bf16-exact",
        "hyper": HYPER,
        "cases": cases,
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_step.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()

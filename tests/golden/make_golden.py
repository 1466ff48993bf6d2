"""Writes tests/golden/oracle_seeded.json: a regression fixture of the oracle.

It calls only ``oracle`` (the fp64 CPU attention) on small inputs drawn from a
seeded numpy generator, and stores the first 64 values and the sums of O and
LSE.  It pins nothing by itself; it detects unintended edits to the oracle.
Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import sys
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parents[2]

CASES = [
    {"name": "sq_nc", "Nq": 40, "Nk": 40, "d": 16, "scale": 0.25, "causal": False, "seed": 7},
    {"name": "sq_causal", "Nq": 40, "Nk": 40, "d": 16, "scale": 0.25, "causal": True, "seed": 8},
    {"name": "rect_causal", "Nq": 23, "Nk": 57, "d": 8, "scale": 0.35, "causal": True, "seed": 9},
]


def case_inputs(case):
    g = np.random.default_rng(case["seed"])
    Q = g.standard_normal((case["Nq"], case["d"])).astype(np.float32)
    K = g.standard_normal((case["Nk"], case["d"])).astype(np.float32)
    V = g.standard_normal((case["Nk"], case["d"])).astype(np.float32)
    return Q, K, V


def main():
    sys.path.insert(0, str(ROOT))
    import oracle
    out = []
    for case in CASES:
        Q, K, V = case_inputs(case)
        O, L = oracle.attention(Q, K, V, case["scale"], case["causal"])
        c = dict(case)
        c["O_head"] = O.reshape(-1)[:64].tolist()
        c["LSE_head"] = L.reshape(-1)[:64].tolist()
        c["O_sum"] = float(O.sum())
        c["LSE_sum"] = float(L.sum())
        out.append(c)
    path = Path(__file__).resolve().parent / "oracle_seeded.json"
    path.write_text(json.dumps({"about": __doc__.strip().splitlines()[0], "cases": out}, indent=1))
    print("wrote", path)


if __name__ == "__main__":
    main()

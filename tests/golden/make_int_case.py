"""Writes int_case.json: a small exact-integer problem and the oracle's answer.

Calls only the oracle. The inputs are small integers, so every intermediate
value is exact in double, in f32 and, for |values| < 256, in bf16 too; GPU
tests can therefore demand bit-exact agreement on this case.

    python tests/golden/make_int_case.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
import oracle  # noqa: E402


def main():
    rng = np.random.default_rng(20261202)
    B, T, C, OC = 1, 5, 8, 16
    BT = B * T
    r = lambda *s: rng.integers(-2, 3, size=s).astype(np.float64)  # noqa: E731
    case = dict(dout=r(BT, OC), inp=r(BT, C), weight=r(OC, C), dinp_init=r(BT, C),
                dweight_init=r(OC, C))
    dinp, dweight, dbias = oracle.get("st").matmul_backward(
        case["dout"], case["inp"], case["weight"], "f64", case["dinp_init"], case["dweight_init"])
    doc = {"cite": "oracle output (matmul_backward_cpu semantics) for small-integer inputs; "
                   "written by tests/golden/make_int_case.py",
           "B": B, "T": T, "C": C, "OC": OC,
           "inputs": {k: v.astype(int).tolist() for k, v in case.items()},
           "expected": {"dinp": dinp.astype(int).tolist(), "dweight": dweight.astype(int).tolist(),
                        "dbias": dbias.astype(int).tolist()}}
    assert np.all(np.abs(dinp) < 256) and np.all(np.abs(dweight) < 256)
    with open(os.path.join(HERE, "int_case.json"), "w") as f:
        json.dump(doc, f, indent=1)


if __name__ == "__main__":
    main()

"""Golden fixtures: the page's own test configuration and an exact-integer case."""
import json
import os

import numpy as np

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_mlp_fc_layer_is_the_pages_test_shape():
    g = load("matmul_backward_main_config.json")
    fc = synth.WORKLOADS["mlp"].layers[0]
    assert (fc.B, fc.T, fc.C, fc.OC) == (g["B"], g["T"], g["C"], g["OC"])
    assert g["OC"] == 4 * g["C"]


def test_int_case_reproduced_by_oracle():
    g = load("int_case.json")
    x = {k: np.array(v, dtype=np.float64) for k, v in g["inputs"].items()}
    dinp, dweight, dbias = oracle.get("st").matmul_backward(
        x["dout"], x["inp"], x["weight"], "f64", x["dinp_init"], x["dweight_init"])
    assert np.array_equal(dinp, g["expected"]["dinp"])
    assert np.array_equal(dweight, g["expected"]["dweight"])
    assert np.array_equal(dbias, g["expected"]["dbias"])
    # and, independently of the oracle, against exact integer matmul
    assert np.array_equal(dinp, x["dinp_init"] + x["dout"] @ x["weight"])
    assert np.array_equal(dweight, x["dweight_init"] + x["dout"].T @ x["inp"])

"""Pins of the oracle to facts that do not come from the oracle itself.

Each ``pin_*`` takes a loaded oracle build and raises AssertionError when the
build disagrees with what the mathematics fixes. ``test_oracle_pins.py`` runs
them on the real builds; ``test_oracle_mutants.py`` runs them on builds with a
planted mistake and requires every mistake to be caught by at least one pin.

The reference computation (llm.c dev/cuda/matmul_backward.cu,
``matmul_backward_cpu``) is the gradient of the forward linear layer
``out = inp @ weight^T + bias`` (the forward call quoted in that file's
``matmul_backward1`` comment) contracted with ``dout``:
L(inp, weight, bias) = sum_{bt,o} dout[bt,o] * out[bt,o]. The pins derive the
expected gradients from that forward scalar, not from the backward formula.
"""
from __future__ import annotations

import itertools
from fractions import Fraction

import numpy as np

import synth

# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------


def _int_case(rng, BT, C, OC, lo=-3, hi=3, init=True):
    """Small-integer inputs as float64 (every sum stays exact in double)."""
    r = lambda *s: rng.integers(lo, hi + 1, size=s).astype(np.float64)  # noqa: E731
    case = dict(dout=r(BT, OC), inp=r(BT, C), weight=r(OC, C), bias=r(OC))
    case["dinp_init"] = r(BT, C) if init else np.zeros((BT, C))
    case["dweight_init"] = r(OC, C) if init else np.zeros((OC, C))
    return case


def _forward_loss_exact(dout, inp, weight, bias):
    """L = sum_{bt,o} dout[bt,o] * (sum_i inp[bt,i]*weight[o,i] + bias[o]) in exact
    rational arithmetic (inputs are small integers or dyadic rationals)."""
    BT, OC = dout.shape
    C = inp.shape[1]
    F = lambda x: Fraction(float(x))  # noqa: E731
    total = Fraction(0)
    for bt in range(BT):
        for o in range(OC):
            out = F(bias[o])
            for i in range(C):
                out += F(inp[bt, i]) * F(weight[o, i])
            total += F(dout[bt, o]) * out
    return total


def _forward_loss_f64(dout, inp, weight, bias):
    return float(np.sum(dout * (inp @ weight.T + bias[None, :])))


def _run_full(orc, case, bias=True):
    return orc.matmul_backward(case["dout"], case["inp"], case["weight"], "f64",
                               case["dinp_init"], case["dweight_init"], bias=bias)


# ---------------------------------------------------------------------------
# pins
# ---------------------------------------------------------------------------


def pin_exact_unit_differences(orc):
    """Brute force on tiny integer problems. L is affine in each single
    coordinate, so L(x + e_k) - L(x) is exactly dL/dx_k; with integer inputs
    every value is an exact integer and the comparison is exact equality."""
    rng = np.random.default_rng(1234)
    # the last shape is square in (BT, C) so that a transposed index would stay in bounds
    for (BT, C, OC) in [(2, 3, 4), (4, 4, 4), (6, 5, 3), (4, 4, 3)]:
        case = _int_case(rng, BT, C, OC)
        dinp, dweight, dbias = _run_full(orc, case)
        args = [case["dout"], case["inp"], case["weight"], case["bias"]]
        L0 = _forward_loss_exact(*args)
        for name, idx_shape, got in (("inp", (BT, C), dinp - case["dinp_init"]),
                                     ("weight", (OC, C), dweight - case["dweight_init"]),
                                     ("bias", (OC,), dbias)):
            pos = {"inp": 1, "weight": 2, "bias": 3}[name]
            for k in itertools.product(*[range(s) for s in idx_shape]):
                bumped = [a.copy() for a in args]
                bumped[pos][k] += 1.0
                want = _forward_loss_exact(*bumped) - L0
                assert want.denominator == 1
                assert got[k] == float(want), (name, k, got[k], want)


def pin_central_differences(orc):
    """Central finite differences of the float64 forward scalar at the tiny
    workload's shape and distributions (B=2, T=64, C=64, OC=192), on random
    coordinates. L is affine in each coordinate, so the difference quotient is
    the gradient up to the rounding of L, which bounds the tolerance."""
    rng = np.random.default_rng(7)
    BT, C, OC = 128, 64, 192
    dout = rng.standard_normal((BT, OC))
    inp = rng.standard_normal((BT, C))
    weight = 0.02 * rng.standard_normal((OC, C))
    bias = 0.02 * rng.standard_normal(OC)
    dinp0 = 0.01 * rng.standard_normal((BT, C))
    dw0 = 0.01 * rng.standard_normal((OC, C))
    dinp, dweight, dbias = orc.matmul_backward(dout, inp, weight, "f64", dinp0, dw0)
    h = 2.0 ** -10
    # rounding of L: about eps * sum |terms|
    scale = np.sum(np.abs(dout) * (np.abs(inp) @ np.abs(weight).T + np.abs(bias)))
    tol = 64 * np.finfo(np.float64).eps * scale / h
    for name, arr, grad in (("inp", inp, dinp - dinp0), ("weight", weight, dweight - dw0),
                            ("bias", bias, dbias)):
        for _ in range(32):
            k = tuple(int(rng.integers(0, s)) for s in arr.shape)
            old = arr[k]
            arr[k] = old + h
            lp = _forward_loss_f64(dout, inp, weight, bias)
            arr[k] = old - h
            lm = _forward_loss_f64(dout, inp, weight, bias)
            arr[k] = old
            fd = (lp - lm) / (2 * h)
            assert abs(fd - grad[k]) <= tol, (name, k, fd, grad[k], tol)


def pin_library_matmul(orc):
    """The three results reduce to library routines: numpy float64 matmul and
    column sums (a different summation order, so a 1e-12 relative bound)."""
    rng = np.random.default_rng(11)
    for (BT, C, OC) in [(128, 64, 192), (33, 17, 40), (1, 8, 8)]:
        dout = rng.standard_normal((BT, OC))
        inp = rng.standard_normal((BT, C))
        weight = rng.standard_normal((OC, C))
        dinp0 = rng.standard_normal((BT, C))
        dw0 = rng.standard_normal((OC, C))
        dinp, dweight, dbias = orc.matmul_backward(dout, inp, weight, "f64", dinp0, dw0)
        for got, want in ((dinp, dinp0 + dout @ weight), (dweight, dw0 + dout.T @ inp),
                          (dbias, dout.sum(axis=0))):
            err = np.max(np.abs(got - want) / (np.abs(want) + 1.0))
            assert err < 1e-12, err


def pin_colsum_invariant(orc):
    """dbias is the column sum of dout: equal, bit for bit on integer data, to
    dout^T times a ones vector, and its total equals the sum of all of dout."""
    rng = np.random.default_rng(5)
    case = _int_case(rng, 37, 8, 24, lo=-9, hi=9)
    _, _, dbias = _run_full(orc, case)
    ones = np.ones(case["dout"].shape[0])
    assert np.array_equal(dbias, case["dout"].T @ ones)
    assert dbias.sum() == case["dout"].sum()


def pin_adjoint_identities(orc):
    """<dinp - dinp0, X> = <dout, X weight^T> and <dweight - dw0, Y> = <dout, inp Y^T>
    for random X, Y: catches transposed or permuted operands."""
    rng = np.random.default_rng(99)
    BT, C, OC = 48, 24, 40
    dout, inp, weight = (rng.standard_normal(s) for s in ((BT, OC), (BT, C), (OC, C)))
    dinp0, dw0 = rng.standard_normal((BT, C)), rng.standard_normal((OC, C))
    dinp, dweight, _ = orc.matmul_backward(dout, inp, weight, "f64", dinp0, dw0)
    X, Y = rng.standard_normal((BT, C)), rng.standard_normal((OC, C))
    lhs1, rhs1 = np.sum((dinp - dinp0) * X), np.sum(dout * (X @ weight.T))
    lhs2, rhs2 = np.sum((dweight - dw0) * Y), np.sum(dout * (inp @ Y.T))
    assert abs(lhs1 - rhs1) <= 1e-10 * (abs(rhs1) + 1)
    assert abs(lhs2 - rhs2) <= 1e-10 * (abs(rhs2) + 1)


def pin_special_cases(orc):
    """Identity weight, one-hot dout and zero dout have closed-form results."""
    rng = np.random.default_rng(3)
    BT, C = 10, 6
    # weight = I (C == OC): dinp = dinp0 + dout
    dout = rng.standard_normal((BT, C))
    inp = rng.standard_normal((BT, C))
    dinp0 = rng.standard_normal((BT, C))
    dinp, _, _ = orc.matmul_backward(dout, inp, np.eye(C), "f64", dinp0, np.zeros((C, C)))
    assert np.array_equal(dinp, dinp0 + dout)
    # one-hot dout at (bt0, o0)
    OC, bt0, o0 = 7, 3, 5
    dout = np.zeros((BT, OC))
    dout[bt0, o0] = 1.0
    weight = rng.standard_normal((OC, C))
    dinp0 = rng.standard_normal((BT, C))
    dw0 = rng.standard_normal((OC, C))
    dinp, dweight, dbias = orc.matmul_backward(dout, inp, weight, "f64", dinp0, dw0)
    want_dw = dw0.copy()
    want_dw[o0] += inp[bt0]
    want_dinp = dinp0.copy()
    want_dinp[bt0] += weight[o0]
    assert np.array_equal(dweight, want_dw)
    assert np.array_equal(dinp, want_dinp)
    assert np.array_equal(dbias, np.eye(OC)[o0])
    # dout = 0: outputs equal their initial values, dbias = 0
    dinp, dweight, dbias = orc.matmul_backward(np.zeros((BT, OC)), inp, weight, "f64", dinp0, dw0)
    assert np.array_equal(dinp, dinp0) and np.array_equal(dweight, dw0)
    assert np.array_equal(dbias, np.zeros(OC))


def pin_double_accumulation(orc):
    """Sums with cancellation that single precision cannot carry: the exact
    integer results require the double accumulation the oracle promises."""
    big = 2.0 ** 27
    dout = np.array([[big, 1.0], [1.0, -big], [-big, 1.0]])  # column sums: 1, 2 - 2^27
    inp = np.array([[1.0], [1.0], [1.0]])
    weight = np.array([[1.0], [1.0]])
    _, dweight, dbias = orc.matmul_backward(dout, inp, weight, "f64", np.zeros((3, 1)),
                                            np.zeros((2, 1)))
    assert dbias[0] == 1.0 and dbias[1] == 2.0 - big, dbias
    assert dweight[0, 0] == 1.0 and dweight[1, 0] == 2.0 - big


def pin_storage_types(orc):
    """bf16 and f32 inputs are read at their exact values: the typed oracle
    equals the float64 oracle run on the exactly converted values."""
    rng = np.random.default_rng(21)
    BT, C, OC = 20, 16, 24
    for dtype in ("bf16", "f32"):
        arrs = {k: synth.normal(s, dtype, 0, 40 + j, 0.0, 1.0)
                for j, (k, s) in enumerate((("dout", (BT, OC)), ("inp", (BT, C)),
                                            ("weight", (OC, C)), ("dinp_init", (BT, C)),
                                            ("dweight_init", (OC, C))))}
        got = orc.matmul_backward(arrs["dout"], arrs["inp"], arrs["weight"], dtype,
                                  arrs["dinp_init"], arrs["dweight_init"])
        f = {k: synth.to_f64(v, dtype) for k, v in arrs.items()}
        want = orc.matmul_backward(f["dout"], f["inp"], f["weight"], "f64", f["dinp_init"],
                                   f["dweight_init"])
        for g, w in zip(got, want):
            assert np.array_equal(g, w)
    del rng


def pin_subset_rows(orc):
    """Row-subset mode returns exactly the rows of the full computation."""
    rng = np.random.default_rng(8)
    BT, C, OC = 40, 12, 30
    dout, inp, weight = (rng.standard_normal(s) for s in ((BT, OC), (BT, C), (OC, C)))
    dinp0, dw0 = rng.standard_normal((BT, C)), rng.standard_normal((OC, C))
    dinp, dweight, dbias = orc.matmul_backward(dout, inp, weight, "f64", dinp0, dw0)
    rows_bt = np.array([0, 7, 39, 7])
    rows_o = np.array([29, 0, 13])
    assert np.array_equal(orc.dinp_rows(dout, weight, "f64", rows_bt, dinp0), dinp[rows_bt])
    dw_rows, db_rows = orc.dweight_rows(dout, inp, "f64", rows_o, dw0)
    assert np.array_equal(dw_rows, dweight[rows_o]) and np.array_equal(db_rows, dbias[rows_o])


def pin_null_bias(orc):
    """Skipping the bias (a NULL dbias) changes nothing else."""
    rng = np.random.default_rng(4)
    case = _int_case(rng, 9, 5, 6)
    a = _run_full(orc, case, bias=True)
    b = _run_full(orc, case, bias=False)
    assert b[2] is None
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def pin_empty_dims(orc):
    """Degenerate sizes: BT = 0 gives dbias = 0 (the empty sum) and leaves
    dweight at its initial value; C = 0 still gives dbias = column sums."""
    rng = np.random.default_rng(6)
    OC, C = 5, 3
    dw0 = rng.standard_normal((OC, C))
    dinp, dweight, dbias = orc.matmul_backward(np.zeros((0, OC)), np.zeros((0, C)),
                                               rng.standard_normal((OC, C)), "f64",
                                               np.zeros((0, C)), dw0)
    assert dinp.shape == (0, C) and np.array_equal(dweight, dw0)
    assert np.array_equal(dbias, np.zeros(OC))
    dout = rng.integers(-4, 5, size=(6, OC)).astype(np.float64)
    _, _, dbias = orc.matmul_backward(dout, np.zeros((6, 0)), np.zeros((OC, 0)), "f64",
                                      np.zeros((6, 0)), np.zeros((OC, 0)))
    assert np.array_equal(dbias, dout.sum(axis=0))


def pin_forward_exact_integers(orc):
    """The forward on small integer inputs against exact Python integer sums,
    with and without the bias, on shapes that include a square weight."""
    rng = np.random.default_rng(31)
    for (BT, C, OC) in [(3, 4, 5), (4, 4, 4), (2, 7, 3)]:
        inp = rng.integers(-3, 4, size=(BT, C)).astype(np.float64)
        w = rng.integers(-3, 4, size=(OC, C)).astype(np.float64)
        b = rng.integers(-3, 4, size=OC).astype(np.float64)
        got_b = orc.forward_rows(inp, w, "f64", bias=b)
        got_n = orc.forward_rows(inp, w, "f64")
        for bt in range(BT):
            for o in range(OC):
                exact = sum(int(inp[bt, i]) * int(w[o, i]) for i in range(C))
                assert got_n[bt, o] == exact
                assert got_b[bt, o] == exact + int(b[o])


def pin_forward_library_and_adjoint(orc):
    """The forward equals numpy's float64 inp @ W^T + b, and is the adjoint of
    the (separately pinned) backward into inp: <dout, inp W^T> = <dout W, inp>."""
    rng = np.random.default_rng(32)
    BT, C, OC = 40, 24, 56
    inp, w = rng.standard_normal((BT, C)), rng.standard_normal((OC, C))
    b, dout = rng.standard_normal(OC), rng.standard_normal((BT, OC))
    out = orc.forward_rows(inp, w, "f64", bias=b)
    want = inp @ w.T + b
    assert np.max(np.abs(out - want) / (np.abs(want) + 1)) < 1e-12
    dinp = orc.dinp_rows(dout, w, "f64")
    lhs, rhs = np.sum(dout * (out - b)), np.sum(dinp * inp)
    assert abs(lhs - rhs) <= 1e-10 * (abs(rhs) + 1)
    rows = np.array([0, 5, 39])
    assert np.array_equal(orc.forward_rows(inp, w, "f64", rows, b), out[rows])


ALL_PINS = [pin_exact_unit_differences, pin_central_differences, pin_library_matmul,
            pin_colsum_invariant, pin_adjoint_identities, pin_special_cases,
            pin_double_accumulation, pin_storage_types, pin_subset_rows, pin_null_bias,
            pin_empty_dims, pin_forward_exact_integers, pin_forward_library_and_adjoint]

# The LayerNorm backward's pins live beside these; the mutant test runs them all.
from oracle_pins_ln import LN_PINS  # noqa: E402

ALL_PINS = ALL_PINS + LN_PINS
from oracle_pins_enc import ENC_PINS  # noqa: E402

ALL_PINS = ALL_PINS + ENC_PINS
from oracle_pins_sr import SR_PINS  # noqa: E402

ALL_PINS = ALL_PINS + SR_PINS

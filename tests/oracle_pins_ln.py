"""Pins of the LayerNorm-backward oracle to facts that do not come from it.

The reference computation (llm.c dev/cuda/layernorm_backward.cu,
``layernorm_backward_cpu``) is the gradient of the layer norm of each row
(``layernorm_forward_cpu`` of the same file) contracted with ``dout``:
L(inp, weight, bias) = sum_{bt,i} dout[bt,i] * out[bt,i]. The pins take the
expected gradients from torch's own LayerNorm in float64 (a library routine,
differentiated by autograd), from central differences of L, and from
properties the mathematics fixes; none retypes the backward formula.
"""
from __future__ import annotations

import numpy as np

EPS = 1e-5


def _case(rng, BT=6, C=40, scale=None):
    """Rows with different offsets and spreads (so mean and rstd matter)."""
    scale = rng.uniform(0.3, 3.0, size=(BT, 1)) if scale is None else scale
    x = rng.normal(size=(BT, C)) * scale + rng.uniform(-2, 2, size=(BT, 1))
    return dict(inp=x, weight=rng.normal(1.0, 0.5, size=C), bias=rng.normal(size=C),
                dout=rng.normal(size=(BT, C)))


def _stats(x):
    """Row mean and reciprocal standard deviation (population variance), numpy."""
    return x.mean(axis=1), 1.0 / np.sqrt(x.var(axis=1) + EPS)


def _torch_reference(c):
    import torch

    x = torch.tensor(c["inp"], dtype=torch.float64, requires_grad=True)
    w = torch.tensor(c["weight"], dtype=torch.float64, requires_grad=True)
    b = torch.tensor(c["bias"], dtype=torch.float64, requires_grad=True)
    out = torch.nn.functional.layer_norm(x, (x.shape[1],), w, b, eps=EPS)
    (out * torch.tensor(c["dout"], dtype=torch.float64)).sum().backward()
    return out.detach().numpy(), x.grad.numpy(), w.grad.numpy(), b.grad.numpy()


def pin_ln_torch_library(orc):
    """Forward values and all three gradients equal torch's float64 LayerNorm
    and its autograd gradients (statistics from numpy, not from the oracle)."""
    rng = np.random.default_rng(11)
    for C in (1, 2, 7, 40):
        c = _case(rng, BT=5, C=C)
        t_out, t_dx, t_dw, t_db = _torch_reference(c)
        out, mean, rstd = orc.layernorm_forward(c["inp"], c["weight"], c["bias"], "f64")
        assert np.allclose(out, t_out, rtol=1e-12, atol=1e-12)
        m, s = _stats(c["inp"])
        assert np.allclose(mean, m, rtol=1e-13, atol=1e-13) and np.allclose(rstd, s, rtol=1e-12)
        dx = orc.layernorm_dinp_rows(c["dout"], c["inp"], c["weight"], m, s, "f64")
        dw, db = orc.layernorm_params(c["dout"], c["inp"], m, s, "f64")
        tol = 1e-11 * (1 + np.abs(t_dx).max())
        assert np.abs(dx - t_dx).max() <= tol, np.abs(dx - t_dx).max()
        assert np.allclose(dw, t_dw, rtol=1e-11, atol=1e-11)
        assert np.allclose(db, t_db, rtol=1e-12, atol=1e-12)


def pin_ln_central_differences(orc):
    """d L / d inp by central differences through the forward (L is smooth in
    inp; h = 1e-5 leaves an O(h^2) error), and d L / d weight, d L / d bias
    (L is affine in them, so the quotient is exact up to rounding)."""
    rng = np.random.default_rng(12)
    c = _case(rng, BT=4, C=24)
    x, w, b, d = c["inp"], c["weight"], c["bias"], c["dout"]

    def L(x_, w_, b_):
        out, _, _ = orc.layernorm_forward(x_, w_, b_, "f64")
        return float(np.sum(d * out))

    _, mean, rstd = orc.layernorm_forward(x, w, b, "f64")
    dx = orc.layernorm_dinp_rows(d, x, w, mean, rstd, "f64")
    dw, db = orc.layernorm_params(d, x, mean, rstd, "f64")
    h = 1e-5
    for _ in range(24):
        r, i = int(rng.integers(4)), int(rng.integers(24))
        xp, xm = x.copy(), x.copy()
        xp[r, i] += h
        xm[r, i] -= h
        fd = (L(xp, w, b) - L(xm, w, b)) / (2 * h)
        assert abs(fd - dx[r, i]) <= 1e-6 * (1 + abs(dx[r, i])), (r, i, fd, dx[r, i])
    for i in range(24):
        wp, wm = w.copy(), w.copy()
        wp[i] += h
        wm[i] -= h
        assert abs((L(x, wp, b) - L(x, wm, b)) / (2 * h) - dw[i]) <= 1e-7 * (1 + abs(dw[i]))
        bp, bm = b.copy(), b.copy()
        bp[i] += h
        bm[i] -= h
        assert abs((L(x, w, bp) - L(x, w, bm)) / (2 * h) - db[i]) <= 1e-7 * (1 + abs(db[i]))


def pin_ln_shift_invariance(orc):
    """Adding a constant to a row leaves the layer norm unchanged, so each row
    of the input gradient sums to zero (with exact statistics); holds for any
    weight and dout, and with fp32 statistics up to their rounding."""
    rng = np.random.default_rng(13)
    c = _case(rng, BT=8, C=33)
    m, s = _stats(c["inp"])
    dx = orc.layernorm_dinp_rows(c["dout"], c["inp"], c["weight"], m, s, "f64")
    scale = np.abs(dx).sum(axis=1)
    assert np.all(np.abs(dx.sum(axis=1)) <= 1e-12 * scale)
    dx32 = orc.layernorm_dinp_rows(c["dout"], c["inp"], c["weight"], m.astype(np.float32),
                                   s.astype(np.float32), "f64")
    assert np.all(np.abs(dx32.sum(axis=1)) <= 1e-5 * scale)


def pin_ln_exact_bias_and_zero_cases(orc):
    """Integer dout: dbias is its exact column sum; weight = 0 gives no input
    gradient; dout = 0 gives no gradient at all; C = 1 has n = 0 and no input
    gradient."""
    rng = np.random.default_rng(14)
    c = _case(rng, BT=7, C=9)
    d = rng.integers(-4, 5, size=(7, 9)).astype(np.float64)
    m, s = _stats(c["inp"])
    _, db = orc.layernorm_params(d, c["inp"], m, s, "f64")
    assert np.array_equal(db, d.sum(axis=0))
    dx0 = orc.layernorm_dinp_rows(d, c["inp"], np.zeros(9), m, s, "f64")
    assert np.array_equal(dx0, np.zeros_like(dx0))
    z = np.zeros_like(d)
    dxz = orc.layernorm_dinp_rows(z, c["inp"], c["weight"], m, s, "f64")
    dwz, dbz = orc.layernorm_params(z, c["inp"], m, s, "f64")
    assert not dxz.any() and not dwz.any() and not dbz.any()
    x1 = c["inp"][:, :1].copy()
    m1, s1 = _stats(x1)
    dx1 = orc.layernorm_dinp_rows(d[:, :1].copy(), x1, c["weight"][:1].copy(), m1, s1, "f64")
    assert np.array_equal(dx1, np.zeros_like(dx1))


def pin_ln_accumulation(orc):
    """The three gradients are added to the initial values (the CPU reference
    accumulates): result(init) - result(0) equals init to rounding, element by
    element, for dinp, dweight and dbias."""
    rng = np.random.default_rng(15)
    c = _case(rng, BT=5, C=16)
    m, s = _stats(c["inp"])
    di, wi, bi = rng.normal(size=(5, 16)), rng.normal(size=16), rng.normal(size=16)
    a = orc.layernorm_dinp_rows(c["dout"], c["inp"], c["weight"], m, s, "f64", dinp_init=di)
    a0 = orc.layernorm_dinp_rows(c["dout"], c["inp"], c["weight"], m, s, "f64")
    w, b = orc.layernorm_params(c["dout"], c["inp"], m, s, "f64", dweight_init=wi, dbias_init=bi)
    w0, b0 = orc.layernorm_params(c["dout"], c["inp"], m, s, "f64")
    for got, base, init in ((a, a0, di), (w, w0, wi), (b, b0, bi)):
        assert np.allclose(got - base, init, rtol=0, atol=1e-13 * (1 + np.abs(base).max()))


def pin_ln_storage_types(orc):
    """fp32 and bf16 inputs give exactly the result of their decoded values in
    float64 (decoded here by bit manipulation, not by the oracle)."""
    rng = np.random.default_rng(16)
    c = _case(rng, BT=4, C=24)
    m, s = _stats(c["inp"])
    m32, s32 = m.astype(np.float32), s.astype(np.float32)
    for dtype in ("f32", "bf16"):
        enc, dec = {}, {}
        for k in ("inp", "weight", "dout"):
            f = c[k].astype(np.float32)
            if dtype == "bf16":
                bits = f.view(np.uint32).astype(np.uint64)
                enc[k] = ((bits + 0x7FFF + ((bits >> 16) & 1)) >> 16).astype(np.uint16)
                dec[k] = (enc[k].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            else:
                enc[k] = f
                dec[k] = f.astype(np.float64)
        got = orc.layernorm_dinp_rows(enc["dout"], enc["inp"], enc["weight"], m32, s32, dtype)
        want = orc.layernorm_dinp_rows(dec["dout"], dec["inp"], dec["weight"], m32, s32, "f64")
        assert np.array_equal(got, want)
        gw, gb = orc.layernorm_params(enc["dout"], enc["inp"], m32, s32, dtype)
        ww, wb = orc.layernorm_params(dec["dout"], dec["inp"], m32, s32, "f64")
        assert np.array_equal(gw, ww) and np.array_equal(gb, wb)


def pin_ln_subset_rows(orc):
    """Selected rows equal the same rows of the full result."""
    rng = np.random.default_rng(17)
    c = _case(rng, BT=9, C=12)
    m, s = _stats(c["inp"])
    full = orc.layernorm_dinp_rows(c["dout"], c["inp"], c["weight"], m, s, "f64")
    rows = np.array([8, 0, 3])
    part = orc.layernorm_dinp_rows(c["dout"], c["inp"], c["weight"], m, s, "f64", rows=rows)
    assert np.array_equal(part, full[rows])


LN_PINS = [pin_ln_torch_library, pin_ln_central_differences, pin_ln_shift_invariance,
           pin_ln_exact_bias_and_zero_cases, pin_ln_accumulation, pin_ln_storage_types,
           pin_ln_subset_rows]

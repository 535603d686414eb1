"""Pins of the encoder-backward oracle to facts that do not come from it.

The reference computation (llm.c llmc/encoder.cuh: the encoder forward adds
row inp[b,t] of wte and row t of wpe; its backward sends each output row's
gradient to both) is a sparse product: dwte = onehot(inp)^T . dout and
dwpe = the sum of dout over the batch. The pins build those from numpy (a
dense one-hot matrix and a library matmul, a reshape and sum) and from
properties the mathematics fixes; none retypes the oracle's loops.
"""
from __future__ import annotations

import numpy as np
import pytest


def _onehot(inp, V):
    m = np.zeros((V, inp.size))
    m[inp, np.arange(inp.size)] = 1.0
    return m


def pin_enc_exact_integers(orc):
    """Integer dout: dwte = onehot^T . dout and dwpe = sum over b, exactly."""
    rng = np.random.default_rng(21)
    for B, T, C, V in ((2, 3, 4, 5), (3, 7, 8, 11), (1, 1, 2, 3)):
        d = rng.integers(-3, 4, size=(B * T, C)).astype(np.float64)
        inp = rng.integers(0, V, size=B * T).astype(np.int32)
        dwte, dwpe = orc.encoder_backward(d, inp, B, T, V, "f64")
        assert np.array_equal(dwte, _onehot(inp, V) @ d)
        assert np.array_equal(dwpe, d.reshape(B, T, C).sum(axis=0))


def pin_enc_conservation(orc):
    """Every dout row lands in exactly one dwte row and one dwpe row: the
    column totals of both increments equal those of dout."""
    rng = np.random.default_rng(22)
    B, T, C, V = 4, 9, 6, 13
    d = rng.normal(size=(B * T, C))
    inp = rng.integers(0, V, size=B * T).astype(np.int32)
    dwte, dwpe = orc.encoder_backward(d, inp, B, T, V, "f64")
    tot = d.sum(axis=0)
    assert np.allclose(dwte.sum(axis=0), tot, rtol=1e-12, atol=1e-12)
    assert np.allclose(dwpe.sum(axis=0), tot, rtol=1e-12, atol=1e-12)


def pin_enc_single_token_and_unused_rows(orc):
    """All positions carry token k: dwte row k is the sum of all rows and every
    other row stays at its initial value."""
    rng = np.random.default_rng(23)
    B, T, C, V = 2, 5, 3, 6
    d = rng.normal(size=(B * T, C))
    init = rng.normal(size=(V, C))
    inp = np.full(B * T, 4, dtype=np.int32)
    dwte, _ = orc.encoder_backward(d, inp, B, T, V, "f64", dwte_init=init)
    others = [i for i in range(V) if i != 4]
    assert np.array_equal(dwte[others], init[others])
    assert np.allclose(dwte[4], init[4] + d.sum(axis=0), rtol=1e-13, atol=1e-13)


def pin_enc_position_permutation(orc):
    """dwte depends only on the multiset of (token, row) pairs: permuting the
    positions (rows move with their tokens) leaves it unchanged up to rounding."""
    rng = np.random.default_rng(24)
    B, T, C, V = 3, 8, 5, 7
    d = rng.normal(size=(B * T, C))
    inp = rng.integers(0, V, size=B * T).astype(np.int32)
    perm = rng.permutation(B * T)
    a, _ = orc.encoder_backward(d, inp, B, T, V, "f64")
    b, _ = orc.encoder_backward(np.ascontiguousarray(d[perm]), np.ascontiguousarray(inp[perm]), B, T, V, "f64")
    assert np.allclose(a, b, rtol=1e-13, atol=1e-13)


def pin_enc_accumulation(orc):
    """Both gradients are added to their initial values."""
    rng = np.random.default_rng(25)
    B, T, C, V = 2, 4, 3, 5
    d = rng.normal(size=(B * T, C))
    inp = rng.integers(0, V, size=B * T).astype(np.int32)
    wi, pi = rng.normal(size=(V, C)), rng.normal(size=(T, C))
    a = orc.encoder_backward(d, inp, B, T, V, "f64", dwte_init=wi, dwpe_init=pi)
    z = orc.encoder_backward(d, inp, B, T, V, "f64")
    assert np.allclose(a[0] - z[0], wi, rtol=0, atol=1e-13)
    assert np.allclose(a[1] - z[1], pi, rtol=0, atol=1e-13)


def pin_enc_storage_types_and_bad_ids(orc):
    """bf16 / fp32 dout give the result of their decoded values (decoded here
    by bit manipulation); a token id outside [0, V) is refused."""
    rng = np.random.default_rng(26)
    B, T, C, V = 2, 3, 8, 4
    f = rng.normal(size=(B * T, C)).astype(np.float32)
    bits = f.view(np.uint32).astype(np.uint64)
    bf = ((bits + 0x7FFF + ((bits >> 16) & 1)) >> 16).astype(np.uint16)
    dec = (bf.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    inp = rng.integers(0, V, size=B * T).astype(np.int32)
    for dt, arr, ref in (("f32", f, f.astype(np.float64)), ("bf16", bf, dec)):
        got = orc.encoder_backward(arr, inp, B, T, V, dt)
        want = orc.encoder_backward(np.ascontiguousarray(ref), inp, B, T, V, "f64")
        assert np.array_equal(got[0], want[0]) and np.array_equal(got[1], want[1])
    bad = inp.copy()
    bad[3] = V
    with pytest.raises(ValueError):
        orc.encoder_backward(dec, bad, B, T, V, "f64")


ENC_PINS = [pin_enc_exact_integers, pin_enc_conservation, pin_enc_single_token_and_unused_rows,
            pin_enc_position_permutation, pin_enc_accumulation, pin_enc_storage_types_and_bad_ids]

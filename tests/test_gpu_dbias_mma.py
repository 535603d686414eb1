"""dbias by MMA (MMBWD_DBIAS=ones): the column sums of dout formed by one more
pair MMA per K step against a tile of ones, dbias = dout^T . 1, instead of
the bias warps.

dinp and dweight come from the same MMAs either way, so they must agree bit
for bit with the default path. dbias: on integer problems every partial sum
is exact in fp32, so it must agree bit for bit too (rounded once, to nearest
or stochastically); on normal inputs it is checked against the oracle.
"""
import numpy as np
import pytest

import linear_layer_gemms_gb300 as mm
import oracle
import synth
from gpu_helpers import TOL, scaled_error, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    mm.load()
    yield


def _int_inputs(B, T, C, OC, seed):
    rng = np.random.default_rng(seed)
    bits = lambda a: (a.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)  # noqa: E731
    r = lambda *s: rng.integers(-2, 3, size=s)  # noqa: E731
    BT = B * T
    return {"dout": bits(r(BT, OC)), "inp": bits(r(BT, C)), "weight": bits(r(OC, C)),
            "dinp": bits(np.zeros((BT, C))), "dweight": bits(np.zeros((OC, C))), "dbias": bits(np.full(OC, 7.0))}


def _run(monkeypatch, x, B, T, C, OC, ones, sr=None, bias=True):
    import torch

    if ones:
        monkeypatch.setenv("MMBWD_DBIAS", "ones")
    else:
        monkeypatch.delenv("MMBWD_DBIAS", raising=False)
    g = {k: to_dev(v, "bf16") for k, v in x.items()}
    args = (g["dinp"], g["dweight"], g["dbias"] if bias else None, g["dout"], g["inp"], g["weight"], B, T, C, OC,
            mm.BF16)
    rc = mm.mmbwd_run_sr(*args, sr) if sr is not None else mm.mmbwd_run(*args)
    assert rc == mm.OK, mm.strerror(rc)
    torch.cuda.synchronize()
    assert mm.mmbwd_device_status()[0] == mm.OK
    return {k: g[k].view(torch.int16).cpu().numpy() for k in ("dinp", "dweight", "dbias")}


SHAPES = [(1, 300, 264, 392), (2, 257, 520, 776), (1, 64, 64, 128), (8, 1024, 768, 768)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("splits", ["0", "3"])
@pytest.mark.parametrize("tile_n", [None, "256,128"])
def test_integer_problems_bit_exact(monkeypatch, shape, splits, tile_n):
    B, T, C, OC = shape
    monkeypatch.setenv("MMBWD_SPLITK", splits)
    if tile_n:
        monkeypatch.setenv("MMBWD_TILE_N", tile_n)
    else:
        monkeypatch.delenv("MMBWD_TILE_N", raising=False)
    x = _int_inputs(B, T, C, OC, seed=sum(shape))
    warps, ones = _run(monkeypatch, x, B, T, C, OC, False), _run(monkeypatch, x, B, T, C, OC, True)
    for k in ("dinp", "dweight", "dbias"):
        assert np.array_equal(warps[k], ones[k]), k
    # and the exact column sums, rounded once
    want = synth.bf16_bits_to_f64(x["dout"]).sum(axis=0)
    got = synth.bf16_bits_to_f64(ones["dbias"].view(np.uint16))
    assert np.array_equal(got, synth.bf16_bits_to_f64(_rne_bits(want)))


def _rne_bits(v):
    f = v.astype(np.float32).view(np.uint32).astype(np.uint64)
    f = (f + 0x7FFF + ((f >> 16) & 1)) >> 16
    return f.astype(np.uint16)


def test_integer_problem_stochastic_rounding(monkeypatch):
    B, T, C, OC = 1, 600, 264, 392
    monkeypatch.setenv("MMBWD_SPLITK", "2")
    x = _int_inputs(B, T, C, OC, seed=5)
    warps, ones = (_run(monkeypatch, x, B, T, C, OC, o, sr=77) for o in (False, True))
    for k in ("dinp", "dweight", "dbias"):
        assert np.array_equal(warps[k], ones[k]), k


@pytest.mark.parametrize("spec", ["mlp:0", "mlp:1", "attn_proj"])
def test_gpt2_layers_against_the_oracle(monkeypatch, spec):
    monkeypatch.delenv("MMBWD_SPLITK", raising=False)
    monkeypatch.delenv("MMBWD_TILE_N", raising=False)
    wl, _, i = spec.partition(":")
    layer = synth.WORKLOADS[wl].layers[int(i or 0)]
    x = synth.make_inputs(layer, seed=0)
    warps = _run(monkeypatch, x, layer.B, layer.T, layer.C, layer.OC, False)
    ones = _run(monkeypatch, x, layer.B, layer.T, layer.C, layer.OC, True)
    for k in ("dinp", "dweight"):
        assert np.array_equal(warps[k], ones[k]), k
    empty = np.zeros((layer.BT, 0), dtype=np.uint16)
    _, ref = oracle.get("omp").dweight_rows(x["dout"], empty, "bf16", None, None, bias=True)
    got = synth.bf16_bits_to_f64(ones["dbias"].view(np.uint16))
    assert scaled_error(got, ref) <= TOL["bf16"]


def test_without_bias_the_flag_changes_nothing(monkeypatch):
    B, T, C, OC = 1, 300, 264, 392
    x = _int_inputs(B, T, C, OC, seed=9)
    a = _run(monkeypatch, x, B, T, C, OC, False, bias=False)
    b = _run(monkeypatch, x, B, T, C, OC, True, bias=False)
    for k in ("dinp", "dweight", "dbias"):
        assert np.array_equal(a[k], b[k]), k
    assert np.array_equal(b["dbias"].view(np.uint16), x["dbias"])

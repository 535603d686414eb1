"""The forward out = inp . weight^T + bias through the C ABI against the
oracle's forward, element by element."""
import json
import os

import numpy as np
import pytest

import linear_layer_gemms_gb300 as mm
import oracle
import synth
from gpu_helpers import assert_close, to_dev, to_host

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module", autouse=True)
def lib():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    mm.load()
    yield


def run_fwd(x, BT, C, OC, dtype, bias=True):
    import torch

    g = {k: to_dev(v, dtype) for k, v in x.items()}
    out = to_dev(synth.normal((BT, OC), dtype, 0, 99), dtype)  # garbage: must be overwritten
    rc = mm.mmbwd_forward(out, g["inp"], g["weight"], g["bias"] if bias else None, 1, BT, C, OC,
                          mm.BF16 if dtype == "bf16" else mm.F32)
    assert rc == mm.OK, mm.strerror(rc)
    torch.cuda.synchronize()
    assert mm.mmbwd_device_status()[0] == mm.OK
    return out


def inputs(BT, C, OC, dtype, seed=0):
    return {"inp": synth.normal((BT, C), dtype, seed, 61, 0.0, 1.0),
            "weight": synth.normal((OC, C), dtype, seed, 62, 0.0, 0.02),
            "bias": synth.normal((OC,), dtype, seed, 63, 0.0, 0.02)}


SHAPES = [(1, 8, 8), (200, 136, 200), (300, 392, 1032), (129, 256, 136), (640, 1600, 264)]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("bias", [True, False])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_forward_parity(shape, dtype, bias):
    BT, C, OC = shape
    x = inputs(BT, C, OC, dtype)
    out = run_fwd(x, BT, C, OC, dtype, bias)
    ref = oracle.get("omp").forward_rows(x["inp"], x["weight"], dtype, bias=x["bias"] if bias else None)
    assert_close(to_host(out, dtype), ref, dtype, "out")


@pytest.mark.parametrize("tile_n", ["256,256", "128,128"])
def test_forward_tile_widths(monkeypatch, tile_n):
    BT, C, OC = 600, 520, 776
    monkeypatch.setenv("MMBWD_TILE_N", tile_n)
    x = inputs(BT, C, OC, "bf16", seed=3)
    out = run_fwd(x, BT, C, OC, "bf16")
    ref = oracle.get("omp").forward_rows(x["inp"], x["weight"], "bf16", bias=x["bias"])
    assert_close(to_host(out, "bf16"), ref, "bf16", "out")


def test_forward_two_box_requests(monkeypatch):
    """The two 64-row weight boxes of a stage in one request
    of 128 rows (ragged OC, so the last request reads past the rows); bitwise
    equal to one request per box."""
    BT, C, OC = 600, 520, 776
    monkeypatch.setenv("MMBWD_TILE_N", "256,256")
    x = inputs(BT, C, OC, "bf16", seed=4)
    wide = to_host(run_fwd(x, BT, C, OC, "bf16"), "bf16")
    monkeypatch.setenv("MMBWD_WIDE_MAPS", "0")
    narrow = to_host(run_fwd(x, BT, C, OC, "bf16"), "bf16")
    assert np.array_equal(wide, narrow)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_forward_integer_case_exact(dtype):
    g = json.load(open(os.path.join(GOLDEN, "int_case.json")))
    inp = np.array(g["inputs"]["inp"], dtype=np.float64)
    w = np.array(g["inputs"]["weight"], dtype=np.float64)
    b = np.arange(w.shape[0], dtype=np.float64) - 3
    conv = (lambda a: (a.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)) if dtype == "bf16" \
        else (lambda a: a.astype(np.float32))
    x = {"inp": conv(inp), "weight": conv(w), "bias": conv(b)}
    out = run_fwd(x, inp.shape[0], inp.shape[1], w.shape[0], dtype)
    assert np.array_equal(to_host(out, dtype), inp @ w.T + b)


def test_forward_degenerate_and_deterministic():
    import torch

    # C == 0: out = bias
    BT, OC = 33, 64
    b = to_dev(synth.normal((OC,), "bf16", 0, 64), "bf16")
    out = to_dev(synth.normal((BT, OC), "bf16", 0, 65), "bf16")
    assert mm.mmbwd_forward(out, None, None, b, 1, BT, 0, OC, mm.BF16) == mm.OK
    torch.cuda.synchronize()
    assert torch.equal(out, b.expand(BT, OC))
    # repeated runs are bitwise identical
    BT, C, OC = 1024, 768, 3072
    x = inputs(BT, C, OC, "bf16", seed=4)
    first = run_fwd(x, BT, C, OC, "bf16").cpu()
    for _ in range(5):
        assert torch.equal(run_fwd(x, BT, C, OC, "bf16").cpu(), first)


FULL = [("mlp_fc", 8192, 768, 3072, "bf16"), ("mlp_fc_proj", 8192, 3072, 768, "bf16"),
        ("attn_proj", 8192, 768, 768, "bf16"), ("lm_head", 8192, 768, 50304, "bf16"),
        ("xl_fc_f32", 4096, 1600, 6400, "f32")]


@pytest.mark.parametrize("case", FULL, ids=lambda c: c[0])
def test_forward_full_size(case, monkeypatch):
    """Every element of the forward at the benchmarked sizes, and the same
    bits on a second run."""
    import torch

    monkeypatch.delenv("MMBWD_TILE_N", raising=False)
    monkeypatch.delenv("MMBWD_F32_PATH", raising=False)
    name, BT, C, OC, dt = case
    x = inputs(BT, C, OC, dt, seed=5)
    bias = name != "lm_head"
    out = run_fwd(x, BT, C, OC, dt, bias=bias)
    ref = oracle.get("omp").forward_rows(x["inp"], x["weight"], dt, bias=x["bias"] if bias else None)
    assert_close(to_host(out, dt), ref, dt, name)
    again = run_fwd(x, BT, C, OC, dt, bias=bias)
    assert torch.equal(out.view(torch.int16 if dt == "bf16" else torch.int32),
                       again.view(torch.int16 if dt == "bf16" else torch.int32))


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_forward_fp32_three_products(shape, monkeypatch):
    """fp32 forward through the tensor-core path (operands split into tf32
    high and exact low parts, three products per K step), forced on small and
    ragged shapes; the default takes it for large layers."""
    monkeypatch.setenv("MMBWD_F32_PATH", "x3")
    BT, C, OC = shape
    for bias in (True, False):
        x = inputs(BT, C, OC, "f32")
        out = run_fwd(x, BT, C, OC, "f32", bias)
        ref = oracle.get("omp").forward_rows(x["inp"], x["weight"], "f32", bias=x["bias"] if bias else None)
        assert_close(to_host(out, "f32"), ref, "f32", "out")

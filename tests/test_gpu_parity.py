"""CUDA path against the oracle, element by element, through the C ABI."""
import json
import os

import numpy as np
import pytest

import linear_layer_gemms_gb300 as mm
import oracle
import synth
from gpu_helpers import assert_close, run_gpu, to_dev, to_host

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


def make(B, T, C, OC, dtype, seed=0, init_std=0.01, dout_std=1.0):
    layer = synth.Layer("case", B, T, C, OC, dtype, True, init_std=init_std, dout_std=dout_std,
                        layer=seed)
    return layer, synth.make_inputs(layer, seed=seed)


def check_full(x, B, T, C, OC, dtype, bias=True):
    g = run_gpu(x, B, T, C, OC, dtype, bias=bias)
    ref = oracle.get("omp").matmul_backward(x["dout"], x["inp"], x["weight"], dtype, x["dinp"],
                                            x["dweight"], bias=bias)
    errs = {}
    for name, r in zip(("dinp", "dweight", "dbias"), ref):
        if r is None:
            continue
        errs[name] = assert_close(to_host(g[name], dtype), r, dtype, name)
    if not bias:  # dbias untouched
        assert np.array_equal(to_host(g["dbias"], dtype), synth.to_f64(x["dbias"], dtype))
    return g, errs


def test_wait_timeout_selftest_reports_and_context_survives():
    assert mm.mmbwd_selftest_wait_timeout(20_000_000) == mm.ERR_DEVICE_TIMEOUT
    assert mm.mmbwd_device_status()[0] == mm.OK  # the self-test cleared it
    _, x = make(1, 64, 64, 64, "bf16")
    check_full(x, 1, 64, 64, 64, "bf16")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_integer_case_is_exact(dtype):
    """Small integers: every product and sum is exact in fp32 and the results
    fit bf16 exactly, so the GPU must reproduce the oracle bit for bit."""
    g = json.load(open(os.path.join(GOLDEN, "int_case.json")))
    B, T, C, OC = g["B"], g["T"], g["C"], g["OC"]
    conv = _bf16_bits if dtype == "bf16" \
        else (lambda a: a.astype(np.float32))
    x = {k: conv(np.array(v, dtype=np.float64)) for k, v in g["inputs"].items()}
    x = {"dout": x["dout"], "inp": x["inp"], "weight": x["weight"], "dinp": x["dinp_init"],
         "dweight": x["dweight_init"], "dbias": conv(np.full(OC, 7.0))}
    out = run_gpu(x, B, T, C, OC, dtype)
    for name in ("dinp", "dweight", "dbias"):
        assert np.array_equal(to_host(out[name], dtype), np.array(g["expected"][name], dtype=np.float64)), name


def _bf16_bits(a):
    f = a.astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)  # exact for small integers


SHAPES = [(1, 1, 8, 8), (1, 200, 136, 200), (2, 64, 64, 192), (3, 100, 264, 520),
          (1, 129, 256, 128), (2, 333, 520, 1032), (1, 64, 1600, 136)]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_parity_small_shapes(shape, dtype):
    B, T, C, OC = shape
    _, x = make(B, T, C, OC, dtype)
    check_full(x, B, T, C, OC, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_no_bias_changes_nothing_else(dtype):
    B, T, C, OC = 2, 100, 136, 264
    _, x = make(B, T, C, OC, dtype)
    g1, _ = check_full(x, B, T, C, OC, dtype, bias=True)
    g0, _ = check_full(x, B, T, C, OC, dtype, bias=False)
    for name in ("dinp", "dweight"):
        assert np.array_equal(to_host(g0[name], dtype), to_host(g1[name], dtype))


@pytest.mark.parametrize("splits", [1, 2, 3, 5])
def test_split_reduction_and_schedule(monkeypatch, splits):
    """Forced splits of the dweight reduction and forced (tiny) persistent
    grids: always within tolerance, and for a fixed split count the result is
    bitwise independent of the grid (the schedule never changes the sums)."""
    B, T, C, OC = 1, 1000, 264, 392
    _, x = make(B, T, C, OC, "bf16", dout_std=1e-2)
    monkeypatch.setenv("MMBWD_SPLITK", str(splits))
    kb = -(-B * T // 64)
    want_splits = -(-kb // -(-kb // splits))  # lowered so that no split is empty
    outs = []
    for grid in (0, 2, 6, 14):
        if grid:
            monkeypatch.setenv("MMBWD_GRID", str(grid))
        else:
            monkeypatch.delenv("MMBWD_GRID", raising=False)
        info = mm.mmbwd_plan_info(B, T, C, OC, mm.BF16, 152)
        assert info["splits"] == want_splits
        assert grid == 0 or info["grid"] == grid
        g, _ = check_full(x, B, T, C, OC, "bf16")
        outs.append({k: to_host(g[k], "bf16") for k in ("dinp", "dweight", "dbias")})
    for o in outs[1:]:
        for k in o:
            assert np.array_equal(o[k], outs[0][k]), k


@pytest.mark.parametrize("split_kb", [7, 12])
def test_uneven_split_lengths(monkeypatch, split_kb):
    """Splits of a forced length with a shorter last one (16 k-blocks of B*T:
    7 + 7 + 2, or 12 + 4): within tolerance of the oracle, dbias included, and
    bitwise independent of the grid."""
    B, T, C, OC = 1, 1000, 264, 392
    _, x = make(B, T, C, OC, "bf16", dout_std=1e-2)
    monkeypatch.setenv("MMBWD_SPLIT_KB", str(split_kb))
    kb = -(-B * T // 64)
    outs = []
    for grid in (0, 6):
        if grid:
            monkeypatch.setenv("MMBWD_GRID", str(grid))
        else:
            monkeypatch.delenv("MMBWD_GRID", raising=False)
        info = mm.mmbwd_plan_info(B, T, C, OC, mm.BF16, 152)
        assert info["kb_per_split"] == split_kb and info["splits"] == -(-kb // split_kb)
        g, _ = check_full(x, B, T, C, OC, "bf16")
        outs.append({k: to_host(g[k], "bf16") for k in ("dinp", "dweight", "dbias")})
    for k in outs[0]:
        assert np.array_equal(outs[1][k], outs[0][k]), k


def test_round_robin_schedule_of_many_items():
    """More items than the per-pair table holds (here 3516 dinp tiles and 16
    splits of 3 dweight tiles, 293 k-blocks each): the round-robin schedule,
    every element against the oracle and bitwise repeatable."""
    B, T, C, OC = 1, 300000, 520, 136
    info = mm.mmbwd_plan_info(B, T, C, OC, mm.BF16, 0)
    assert info["table"] == 0 and info["items"] > 3072 and info["splits"] > 1
    _, x = make(B, T, C, OC, "bf16", dout_std=1e-2)
    g, _ = check_full(x, B, T, C, OC, "bf16")
    again = run_gpu(x, B, T, C, OC, "bf16")
    for k in ("dinp", "dweight", "dbias"):
        assert np.array_equal(to_host(g[k], "bf16"), to_host(again[k], "bf16")), k


def test_split_counts_across_launches(monkeypatch):
    """Split launches of different shapes and split counts, with unsplit
    launches between them, sharing the workspace's partial tiles: each gives
    the same bits every time it runs from the same buffers, within tolerance
    of the oracle."""
    shapes = [((1, 1000, 264, 392), 3), ((2, 640, 520, 776), 2), ((1, 1000, 264, 392), 5), ((1, 512, 128, 128), 0)]
    inputs = {s: make(*s[0], "bf16", dout_std=1e-2)[1] for s in shapes}
    first = {}
    for rep in range(3):
        for shape, splits in shapes:
            if splits:
                monkeypatch.setenv("MMBWD_SPLITK", str(splits))
            else:
                monkeypatch.delenv("MMBWD_SPLITK", raising=False)
            B, T, C, OC = shape
            if rep == 0:
                g, _ = check_full(inputs[(shape, splits)], B, T, C, OC, "bf16")
            else:
                g = run_gpu(inputs[(shape, splits)], B, T, C, OC, "bf16")
            out = {k: to_host(g[k], "bf16") for k in ("dinp", "dweight", "dbias")}
            if rep == 0:
                first[(shape, splits)] = out
            else:
                for k in out:
                    assert np.array_equal(out[k], first[(shape, splits)][k]), (shape, splits, k)
    assert mm.mmbwd_device_status()[0] == mm.OK


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_bitwise_deterministic(dtype):
    B, T, C, OC = 4, 256, 768, 1024
    _, x = make(B, T, C, OC, dtype, init_std=0.0, dout_std=1e-2)
    first = None
    for _ in range(10):
        g = run_gpu(x, B, T, C, OC, dtype)
        cur = [g[k].cpu() for k in ("dinp", "dweight", "dbias")]
        if first is None:
            first = cur
        else:
            for a, b in zip(first, cur):
                assert bool((a.view(-1).view(dtype=_int_view(a)) == b.view(-1).view(dtype=_int_view(b))).all())


def _int_view(t):
    import torch

    return torch.int16 if t.dtype == torch.bfloat16 else torch.int32


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_degenerate_sizes(dtype):
    import torch

    # B*T == 0: dbias becomes the empty sum, dweight untouched
    OC, C = 64, 32
    dw = to_dev(synth.normal((OC, C), dtype, 0, 50), dtype)
    dw0 = dw.clone()
    db = to_dev(synth.normal((OC,), dtype, 0, 51), dtype)
    w = to_dev(synth.normal((OC, C), dtype, 0, 52), dtype)
    dt = mm.BF16 if dtype == "bf16" else mm.F32
    assert mm.mmbwd_run(None, dw, db, None, None, w, 0, 16, C, OC, dt) == mm.OK
    torch.cuda.synchronize()
    assert torch.equal(dw, dw0) and bool((db.float() == 0).all())
    # C == 0: dbias is still the column sum of dout
    BT = 50
    dout = synth.normal((BT, OC), dtype, 0, 53)
    db = to_dev(synth.normal((OC,), dtype, 0, 54), dtype)
    assert mm.mmbwd_run(None, None, db, to_dev(dout, dtype), None, None, 1, BT, 0, OC, dt) == mm.OK
    torch.cuda.synchronize()
    ref = synth.to_f64(dout, dtype).sum(axis=0)
    assert_close(to_host(db, dtype), ref, dtype, "dbias C=0")
    # OC == 0: nothing changes
    dinp = to_dev(synth.normal((BT, C), dtype, 0, 55), dtype)
    d0 = dinp.clone()
    inp = to_dev(synth.normal((BT, C), dtype, 0, 56), dtype)
    assert mm.mmbwd_run(dinp, None, None, None, inp, None, 1, BT, C, 0, dt) == mm.OK
    torch.cuda.synchronize()
    assert torch.equal(dinp, d0)
    assert mm.mmbwd_device_status()[0] == mm.OK


def test_workspace_allocation_failure_is_reported(monkeypatch):
    monkeypatch.setenv("MMBWD_SPLITK", "4")
    B, T, C, OC = 1, 2048, 256, 256
    _, x = make(B, T, C, OC, "bf16")
    g = {k: to_dev(v, "bf16") for k, v in x.items()}
    assert mm.mmbwd_release() == mm.OK
    mm.mmbwd_debug_fail_next_alloc(1)
    rc = mm.mmbwd_run(g["dinp"], g["dweight"], g["dbias"], g["dout"], g["inp"], g["weight"], B, T, C,
                      OC, mm.BF16)
    assert rc == mm.ERR_ALLOC
    mm.mmbwd_debug_fail_next_alloc(0)
    check_full(x, B, T, C, OC, "bf16")


def test_workspace_growth_refused_during_capture(monkeypatch):
    import torch

    monkeypatch.setenv("MMBWD_SPLITK", "3")
    B, T, C, OC = 1, 2048, 512, 384
    _, x = make(B, T, C, OC, "bf16")
    g = {k: to_dev(v, "bf16") for k, v in x.items()}
    assert mm.mmbwd_release() == mm.OK
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    rc = None
    with torch.cuda.graph(graph, stream=s):
        rc = mm.mmbwd_run(g["dinp"], g["dweight"], g["dbias"], g["dout"], g["inp"], g["weight"], B, T,
                          C, OC, mm.BF16, s.cuda_stream)
    assert rc == mm.ERR_CAPTURE


@pytest.mark.parametrize("tile_n", ["128,128", "128,256", "256,128", "256,256"])
@pytest.mark.parametrize("splits", [1, 3])
def test_tile_widths(monkeypatch, tile_n, splits):
    """Every tile width of each product, with and without a split dweight
    reduction, on a shape with ragged rows and columns."""
    B, T, C, OC = 2, 300, 392, 520
    monkeypatch.setenv("MMBWD_TILE_N", tile_n)
    monkeypatch.setenv("MMBWD_SPLITK", str(splits))
    info = mm.mmbwd_plan_info(B, T, C, OC, mm.BF16, 152)
    assert f"{info['tile_n_dinp']},{info['tile_n_dweight']}" == tile_n
    _, x = make(B, T, C, OC, "bf16", dout_std=1e-1)
    check_full(x, B, T, C, OC, "bf16")


@pytest.mark.parametrize("tile_n", ["256,256", "128,128"])
@pytest.mark.parametrize("splits", [1, 3])
def test_tile_widths_on_one_pair(monkeypatch, tile_n, splits):
    """Both tile widths, with or without a split dweight reduction, on a ragged
    shape; and the same plan on a grid of one CTA pair, bitwise equal."""
    B, T, C, OC = 3, 300, 392, 1032
    monkeypatch.setenv("MMBWD_TILE_N", tile_n)
    monkeypatch.setenv("MMBWD_SPLITK", str(splits))
    info = mm.mmbwd_plan_info(B, T, C, OC, mm.BF16, 152)
    assert info["pairs_per_cluster"] == 1
    _, x = make(B, T, C, OC, "bf16", dout_std=1e-1)
    g0, _ = check_full(x, B, T, C, OC, "bf16")
    monkeypatch.setenv("MMBWD_GRID", "2")  # every item on one CTA pair
    g1, _ = check_full(x, B, T, C, OC, "bf16")
    for k in ("dinp", "dweight", "dbias"):
        assert np.array_equal(to_host(g0[k], "bf16"), to_host(g1[k], "bf16")), k


@pytest.mark.parametrize("tile_n", ["256,256", "128,128"])
@pytest.mark.parametrize("splits", [1, 3])
def test_two_box_requests(monkeypatch, tile_n, splits):
    """Where an MN-major operand's extent is a multiple of 64, both 64-column
    boxes of a stage may arrive in one three-dimensional TMA request; the last
    column block of C and the last 128 rows of OC (extents 5 and 11 times 64)
    still take the one-box loads. Within tolerance of the oracle, and bitwise
    equal to the run with one request per box."""
    B, T, C, OC = 2, 300, 320, 704
    monkeypatch.setenv("MMBWD_TILE_N", tile_n)
    monkeypatch.setenv("MMBWD_SPLITK", str(splits))
    _, x = make(B, T, C, OC, "bf16", dout_std=1e-1)
    g1, _ = check_full(x, B, T, C, OC, "bf16")
    monkeypatch.setenv("MMBWD_WIDE_MAPS", "0")
    g0, _ = check_full(x, B, T, C, OC, "bf16")
    for k in ("dinp", "dweight", "dbias"):
        assert np.array_equal(to_host(g0[k], "bf16"), to_host(g1[k], "bf16")), k

"""The fp32 path on the tensor cores (three tf32 products per K step, the
operands split in shared memory by the kernel) through the C ABI against the
oracle, element by element: ragged sizes (K not a multiple of the 32-deep
k-block, rows not a multiple of the 256-row tile or of 4, one tile, many
tiles, 64-wide boxes partly outside the tensor), with and without dbias, a
seeded sweep of ragged shapes through both the paired and the two-launch
forms and the forward, run-to-run bitwise determinism, and the choice between
it and the fp32 FMA kernel."""
import numpy as np
import pytest

import linear_layer_gemms_gb300 as mm
import oracle
import synth
from gpu_helpers import assert_close, run_gpu, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    mm.load()
    yield


def inputs(BT, C, OC, seed=0):
    layer = synth.Layer("x3", 1, BT, C, OC, "f32", True, inp_std=1.0, w_std=0.02, dout_std=1.0,
                        init_std=0.01)
    return synth.make_inputs(layer, seed)


# (BT, C, OC): K = OC or BT ragged against 32; BT not a multiple of 4 (the
# transposed operands' rows are padded); one 256 x 128 tile; several tiles;
# both reductions above 2048 (both products in one launch, each with its
# correction accumulator); only the dweight reduction above 2048 (the
# products in two launches).
SHAPES = [(64, 8, 4), (301, 264, 136), (513, 520, 1028), (256, 128, 256), (2048, 768, 768), (2304, 264, 2304),
          (2560, 264, 512), (301, 260, 132), (777, 132, 516)]


@pytest.mark.parametrize("bias", [True, False])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_x3_parity(shape, bias, monkeypatch):
    monkeypatch.setenv("MMBWD_F32_PATH", "x3")
    BT, C, OC = shape
    assert mm.mmbwd_plan_info(1, BT, C, OC, mm.F32)["path"] == 2
    x = inputs(BT, C, OC)
    g = run_gpu(x, 1, BT, C, OC, "f32", bias=bias)
    ref = oracle.get("omp").matmul_backward(x["dout"], x["inp"], x["weight"], "f32", x["dinp"], x["dweight"],
                                            bias=bias)
    assert_close(to_host(g["dinp"], "f32"), ref[0], "f32", "dinp")
    assert_close(to_host(g["dweight"], "f32"), ref[1], "f32", "dweight")
    if bias:
        assert_close(to_host(g["dbias"], "f32"), ref[2], "f32", "dbias")
    else:
        assert np.array_equal(to_host(g["dbias"], "f32"), x["dbias"].astype(np.float64))


@pytest.mark.parametrize("tile_n", ["256", "128"])
def test_x3_paired_launch_tile_widths(tile_n, monkeypatch):
    """Both products in one launch at either tile width: the dinp and dweight
    tiles share the CTA pairs (ragged in every dimension)."""
    monkeypatch.setenv("MMBWD_F32_PATH", "x3")
    monkeypatch.setenv("MMBWD_TILE_N_X3", tile_n)
    BT, C, OC = 777, 392, 520
    info = mm.mmbwd_plan_info(1, BT, C, OC, mm.F32)
    assert info["launches"] == 1 and info["tile_n_dinp"] == int(tile_n) == info["tile_n_dweight"]
    x = inputs(BT, C, OC, seed=7)
    g = run_gpu(x, 1, BT, C, OC, "f32")
    ref = oracle.get("omp").matmul_backward(x["dout"], x["inp"], x["weight"], "f32", x["dinp"], x["dweight"])
    assert_close(to_host(g["dinp"], "f32"), ref[0], "f32", "dinp")
    assert_close(to_host(g["dweight"], "f32"), ref[1], "f32", "dweight")
    assert_close(to_host(g["dbias"], "f32"), ref[2], "f32", "dbias")


def test_x3_deterministic(monkeypatch):
    monkeypatch.setenv("MMBWD_F32_PATH", "x3")
    BT, C, OC = 777, 392, 520
    x = inputs(BT, C, OC, seed=5)
    outs = []
    for _ in range(3):
        g = run_gpu(x, 1, BT, C, OC, "f32")
        outs.append([g[k].cpu().numpy().tobytes() for k in ("dinp", "dweight", "dbias")])
    assert outs[0] == outs[1] == outs[2]


def test_path_choice(monkeypatch):
    monkeypatch.delenv("MMBWD_F32_PATH", raising=False)
    # every shape the tensor-core path takes uses it, from the tiny check to the
    # XL fp32 layers
    assert mm.mmbwd_plan_info(2, 64, 64, 192, mm.F32)["path"] == 2
    assert mm.mmbwd_plan_info(4, 1024, 1600, 6400, mm.F32)["path"] == 2
    # rows of 4 (mod 8) floats stay on the tensor cores; a reduction longer
    # than 8192 falls back to the FMA kernel, even when forced
    assert mm.mmbwd_plan_info(1, 512, 260, 516, mm.F32)["path"] == 2
    monkeypatch.setenv("MMBWD_F32_PATH", "x3")
    assert mm.mmbwd_plan_info(1, 512, 260, 8196, mm.F32)["path"] == 0
    monkeypatch.setenv("MMBWD_F32_PATH", "ffma")
    assert mm.mmbwd_plan_info(4, 1024, 1600, 6400, mm.F32)["path"] == 0


def _sweep(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        BT = int(rng.integers(1, 3200))
        C = 4 * int(rng.integers(1, 280))
        OC = 4 * int(rng.integers(1, 700))
        out.append((BT, C, OC))
    return out


@pytest.mark.parametrize("shape", _sweep(16, 7), ids=lambda s: "x".join(map(str, s)))
def test_x3_ragged_sweep(shape, monkeypatch):
    """Seeded ragged shapes (either reduction above or below the correction
    threshold, so both launch forms occur), forced onto the tensor-core path:
    dinp, dweight and dbias against the oracle, then the forward of the same
    layer against the oracle's forward."""
    monkeypatch.setenv("MMBWD_F32_PATH", "x3")
    BT, C, OC = shape
    assert mm.mmbwd_plan_info(1, BT, C, OC, mm.F32)["path"] == 2
    x = inputs(BT, C, OC, seed=BT + C + OC)
    g = run_gpu(x, 1, BT, C, OC, "f32")
    orc = oracle.get("omp")
    ref = orc.matmul_backward(x["dout"], x["inp"], x["weight"], "f32", x["dinp"], x["dweight"])
    assert_close(to_host(g["dinp"], "f32"), ref[0], "f32", "dinp")
    assert_close(to_host(g["dweight"], "f32"), ref[1], "f32", "dweight")
    assert_close(to_host(g["dbias"], "f32"), ref[2], "f32", "dbias")
    if mm.mmbwd_forward_path(1, BT, C, OC, mm.F32) == 2:
        import torch

        out = torch.empty(BT * OC, dtype=torch.float32, device="cuda")
        bias = torch.from_numpy(x["dbias"].astype(np.float32)).cuda()
        assert mm.mmbwd_forward(out, g["inp"], g["weight"], bias, 1, BT, C, OC, mm.F32) == mm.OK
        torch.cuda.synchronize()
        want = orc.forward_rows(x["inp"], x["weight"], "f32", bias=x["dbias"])
        assert_close(out.cpu().numpy().astype(np.float64).reshape(BT, OC), want, "f32", "forward")

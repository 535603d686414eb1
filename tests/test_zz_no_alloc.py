"""mmbwd_run_static_scratch -- the entry point that allocates nothing.

Some callers cannot allocate device memory: code running inside an allocator
or memory-pool callback (allocating there would re-enter the allocator),
programs held to a device-memory budget fixed at start-up, or runtimes that
forbid cudaMalloc once running because it synchronises the device. For them
this entry point takes the split partials of the bf16 path from a fixed
buffer compiled into the library instead of growing a workspace.

Each test runs both entry points from identical buffers, twice in a row, and
compares the outputs after each call. The file is named so that pytest
collects it last.
"""
import numpy as np
import pytest

import linear_layer_gemms_gb300 as mm
import oracle
import synth
from gpu_helpers import TOL, scaled_error, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    mm.load()
    yield


# (B, T, C, OC, forced splits): a forced 3-way split with ragged tiles, the
# attention-projection shape whose own plan splits dweight, and a small shape
# whose plan needs no scratch at all.
CASES = [(1, 1000, 264, 392, "3"), (8, 1024, 768, 768, ""), (2, 100, 136, 264, "1")]


def _call(fn, t, layer, bias=True):
    return fn(t["dinp"], t["dweight"], t["dbias"] if bias else None, t["dout"], t["inp"], t["weight"], layer.B,
              layer.T, layer.C, layer.OC, mm.BF16 if layer.dtype == "bf16" else mm.F32)


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:4])) + (f"-s{c[4]}" if c[4] else ""))
def test_matches_mmbwd_run_on_two_calls_in_a_row(monkeypatch, case):
    import torch

    B, T, C, OC, splits = case
    if splits:
        monkeypatch.setenv("MMBWD_SPLITK", splits)
    else:
        monkeypatch.delenv("MMBWD_SPLITK", raising=False)
    monkeypatch.delenv("MMBWD_GRID", raising=False)
    layer = synth.Layer("no_alloc", B, T, C, OC, "bf16", True, init_std=0.01, dout_std=1e-2, layer=3)
    x = synth.make_inputs(layer, seed=11)
    info = mm.mmbwd_plan_info(B, T, C, OC, mm.BF16, 0)
    needs_scratch = mm.mmbwd_workspace_bytes(B, T, C, OC, mm.BF16) > 0
    assert needs_scratch == (info["splits"] > 1)
    assert mm.mmbwd_workspace_bytes(B, T, C, OC, mm.BF16) <= mm.STATIC_SCRATCH_BYTES
    ref = {k: to_dev(v, "bf16") for k, v in x.items()}
    got = {k: to_dev(v, "bf16") for k, v in x.items()}
    for call in range(2):
        assert _call(mm.mmbwd_run, ref, layer) == mm.OK
        assert _call(mm.mmbwd_run_static_scratch, got, layer) == mm.OK
        torch.cuda.synchronize()
        assert mm.mmbwd_device_status()[0] == mm.OK
        for name in ("dinp", "dweight", "dbias"):
            a, b = to_host(ref[name], "bf16"), to_host(got[name], "bf16")
            err = scaled_error(b, a)
            assert err <= TOL["bf16"], (call, name, err)
            # same plan and same kernels: the results are in fact identical
            assert np.array_equal(a, b), (call, name)


def test_rejects_a_split_that_does_not_fit_and_enqueues_nothing(monkeypatch):
    import torch

    B, T, C, OC = 1, 1024, 4096, 4096
    monkeypatch.setenv("MMBWD_SPLITK", "4")
    monkeypatch.delenv("MMBWD_GRID", raising=False)
    assert mm.mmbwd_workspace_bytes(B, T, C, OC, mm.BF16) > mm.STATIC_SCRATCH_BYTES
    dev = torch.device("cuda:0")
    t = {"dinp": torch.zeros(B * T, C, dtype=torch.bfloat16, device=dev),
         "dweight": torch.zeros(OC, C, dtype=torch.bfloat16, device=dev),
         "dbias": torch.full((OC,), 3.0, dtype=torch.bfloat16, device=dev),
         "dout": torch.ones(B * T, OC, dtype=torch.bfloat16, device=dev),
         "inp": torch.ones(B * T, C, dtype=torch.bfloat16, device=dev),
         "weight": torch.ones(OC, C, dtype=torch.bfloat16, device=dev)}
    layer = synth.Layer("too_big", B, T, C, OC, "bf16", True)
    assert _call(mm.mmbwd_run_static_scratch, t, layer) == mm.ERR_SCRATCH
    torch.cuda.synchronize()
    assert bool((t["dinp"] == 0).all()) and bool((t["dweight"] == 0).all())
    assert bool((t["dbias"] == 3.0).all())
    assert "scratch" in mm.strerror(mm.ERR_SCRATCH)


def test_without_bias_matches_mmbwd_run_and_leaves_dbias_alone(monkeypatch):
    import torch

    monkeypatch.setenv("MMBWD_SPLITK", "2")
    monkeypatch.delenv("MMBWD_GRID", raising=False)
    layer = synth.Layer("no_alloc_nobias", 1, 640, 264, 392, "bf16", False, init_std=0.01, dout_std=1e-2, layer=4)
    x = synth.make_inputs(layer, seed=12)
    ref = {k: to_dev(v, "bf16") for k, v in x.items()}
    got = {k: to_dev(v, "bf16") for k, v in x.items()}
    dbias0 = got["dbias"].clone()
    for call in range(2):
        assert _call(mm.mmbwd_run, ref, layer, bias=False) == mm.OK
        assert _call(mm.mmbwd_run_static_scratch, got, layer, bias=False) == mm.OK
        torch.cuda.synchronize()
        for name in ("dinp", "dweight"):
            assert np.array_equal(to_host(ref[name], "bf16"), to_host(got[name], "bf16")), (call, name)
        assert torch.equal(got["dbias"], dbias0)


# fp32 takes mmbwd_run's path here (neither fp32 path uses scratch), so the
# bits agree with mmbwd_run: (1,8200,64,72) on the FMA kernel (a reduction
# longer than 8192), (1,1024,512,256) on the three-tf32 path; both against the
# oracle too.
@pytest.mark.parametrize("shape", [(1, 8200, 64, 72), (1, 1024, 512, 256)], ids=lambda s: "x".join(map(str, s)))
def test_fp32_matches_the_oracle_on_two_calls_in_a_row(shape):
    import torch

    B, T, C, OC = shape
    layer = synth.Layer("no_alloc_f32", B, T, C, OC, "f32", True, init_std=0.01, dout_std=1.0, layer=5)
    x = synth.make_inputs(layer, seed=13)
    ref = {k: to_dev(v, "f32") for k, v in x.items()}
    got = {k: to_dev(v, "f32") for k, v in x.items()}
    orc = oracle.get("omp")
    dinp_o, dw_o = x["dinp"], x["dweight"]
    for call in range(2):
        assert _call(mm.mmbwd_run, ref, layer) == mm.OK
        assert _call(mm.mmbwd_run_static_scratch, got, layer) == mm.OK
        torch.cuda.synchronize()
        assert mm.mmbwd_device_status()[0] == mm.OK
        want = orc.matmul_backward(x["dout"], x["inp"], x["weight"], "f32", dinp_o, dw_o)
        for name, w in zip(("dinp", "dweight", "dbias"), want):
            g = to_host(got[name], "f32")
            assert scaled_error(g, w) <= TOL["f32"], (call, name)
            assert scaled_error(to_host(ref[name], "f32"), w) <= TOL["f32"], (call, name)
            assert np.array_equal(g, to_host(ref[name], "f32")), (call, name)
        # the next call starts from this call's outputs (as the device buffers do)
        dinp_o = to_host(got["dinp"], "f32").astype(np.float32)
        dw_o = to_host(got["dweight"], "f32").astype(np.float32)
        ref = {**ref, "dinp": to_dev(dinp_o, "f32"), "dweight": to_dev(dw_o, "f32")}


def test_allocates_nothing(monkeypatch):
    """With the library's workspace released and the next allocation set to
    fail, a call that splits its reduction still succeeds and leaves free
    device memory unchanged; mmbwd_run, which must grow the workspace for the
    same shape, then meets the pending failure."""
    import torch

    monkeypatch.setenv("MMBWD_SPLITK", "3")
    monkeypatch.delenv("MMBWD_GRID", raising=False)
    layer = synth.Layer("no_alloc_grow", 1, 1000, 264, 392, "bf16", True, init_std=0.01, dout_std=1e-2, layer=6)
    assert mm.mmbwd_workspace_bytes(layer.B, layer.T, layer.C, layer.OC, mm.BF16) > 0
    x = synth.make_inputs(layer, seed=14)
    t = {k: to_dev(v, "bf16") for k, v in x.items()}
    assert _call(mm.mmbwd_run_static_scratch, t, layer) == mm.OK  # first call on the device: set-up
    torch.cuda.synchronize()
    assert mm.mmbwd_release() == mm.OK
    free0 = torch.cuda.mem_get_info()[0]
    mm.mmbwd_debug_fail_next_alloc(1)
    try:
        for _ in range(2):
            assert _call(mm.mmbwd_run_static_scratch, t, layer) == mm.OK
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0
        assert mm.mmbwd_device_status()[0] == mm.OK
        assert _call(mm.mmbwd_run, t, layer) == mm.ERR_ALLOC  # the injected failure was still pending
    finally:
        mm.mmbwd_debug_fail_next_alloc(0)
    assert _call(mm.mmbwd_run, t, layer) == mm.OK
    torch.cuda.synchronize()

"""The library's calls inside a CUDA graph: one slice of a training step (the
linear-layer backward with a split dweight reduction, its forward, the
LayerNorm backward, the encoder backward in its two calls) captured on a
stream once the workspace has grown, then replayed twice from the same initial
values; every output must equal, bit for bit, the same calls run eagerly."""
import numpy as np
import pytest

import linear_layer_gemms_gb300 as mm
import synth
from gpu_helpers import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    mm.load()
    yield


def _inputs():
    import torch

    lin = synth.Layer("graph_lin", 2, 512, 392, 520, "bf16", True, init_std=0.01)
    xl = synth.make_inputs(lin, seed=3)
    lnp = synth.LNProblem("graph_ln", 2, 256, 768, "bf16")
    xn = synth.make_ln_inputs(lnp, seed=4)
    x32 = synth.bf16_bits_to_f64(xn["inp"])
    mean = x32.mean(axis=1)
    rstd = 1.0 / np.sqrt(((x32 - mean[:, None]) ** 2).mean(axis=1) + 1e-5)
    enc = synth.ENC_WORKLOADS["enc_gpt2_small"]
    xe = synth.make_enc_inputs(enc, seed=5)
    t = {"lin_" + k: to_dev(v, "bf16") for k, v in xl.items()}
    t.update({"ln_" + k: to_dev(v, "bf16") for k, v in xn.items()})
    t["ln_mean"] = to_dev(mean.astype(np.float32), "f32")
    t["ln_rstd"] = to_dev(rstd.astype(np.float32), "f32")
    t.update({"enc_" + k: to_dev(xe[k], "bf16") for k in ("dout", "dwte", "dwpe")})
    t["enc_inp"] = torch.from_numpy(xe["inp"]).to("cuda:0")
    t["fwd_out"] = torch.zeros((lin.BT, lin.OC), dtype=torch.bfloat16, device="cuda:0")
    nplan = mm.encbwd_plan_bytes(enc.B, enc.T, enc.C, enc.V, mm.BF16)
    t["enc_plan"] = torch.zeros(nplan, dtype=torch.uint8, device="cuda:0")
    return lin, lnp, enc, nplan, t


def _step(lin, lnp, enc, nplan, t, stream):
    BF = mm.BF16
    s = stream.cuda_stream
    rcs = [
        mm.mmbwd_run(t["lin_dinp"], t["lin_dweight"], t["lin_dbias"], t["lin_dout"], t["lin_inp"], t["lin_weight"],
                     lin.B, lin.T, lin.C, lin.OC, BF, s),
        mm.mmbwd_forward(t["fwd_out"], t["lin_inp"], t["lin_weight"], t["lin_dbias"], lin.B, lin.T, lin.C, lin.OC,
                         BF, s),
        mm.lnbwd_run(t["ln_dinp"], t["ln_dweight"], t["ln_dbias"], t["ln_dout"], t["ln_inp"], t["ln_weight"],
                     t["ln_mean"], t["ln_rstd"], lnp.B, lnp.T, lnp.C, BF, s),
        mm.encbwd_prepare(t["enc_plan"], nplan, t["enc_inp"], enc.B, enc.T, enc.C, enc.V, BF, s),
        mm.encbwd_run_planned(t["enc_dwte"], t["enc_dwpe"], t["enc_dout"], t["enc_plan"], enc.B, enc.T, enc.C,
                              enc.V, BF, None, s),
    ]
    assert rcs == [mm.OK] * len(rcs), [mm.strerror(rc) for rc in rcs]


OUTPUTS = ("lin_dinp", "lin_dweight", "lin_dbias", "fwd_out", "ln_dinp", "ln_dweight", "ln_dbias", "enc_dwte",
           "enc_dwpe")


def test_graph_replay_equals_eager(monkeypatch):
    import torch

    monkeypatch.setenv("MMBWD_SPLITK", "3")  # the split reduction and its second launch
    lin, lnp, enc, nplan, t = _inputs()
    init = {k: t[k].clone() for k in OUTPUTS}
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        _step(lin, lnp, enc, nplan, t, s)  # eager; grows the workspace
    torch.cuda.synchronize()
    eager = {k: t[k].clone() for k in OUTPUTS}
    assert mm.mmbwd_device_status(reset=True)[0] == mm.OK

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        _step(lin, lnp, enc, nplan, t, s)
    for _ in range(2):
        for k in OUTPUTS:
            t[k].copy_(init[k])
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        for k in OUTPUTS:
            assert torch.equal(t[k].view(torch.uint8), eager[k].view(torch.uint8)), k
    assert mm.mmbwd_device_status(reset=True)[0] == mm.OK


def test_fp32_tensor_core_path_captures_without_a_workspace(monkeypatch):
    """The fp32 tensor-core path splits its operands in shared memory, so it
    needs no workspace: with the library's workspace released, the first call
    of a shape may already be captured (a call that had to allocate would
    return MMBWD_ERR_CAPTURE). The replays equal the same call run eagerly,
    bit for bit; the forward likewise."""
    import torch

    monkeypatch.setenv("MMBWD_F32_PATH", "x3")
    B, T, C, OC = 1, 777, 392, 520
    assert mm.mmbwd_plan_info(B, T, C, OC, mm.F32)["path"] == 2
    assert mm.mmbwd_forward_path(B, T, C, OC, mm.F32) == 2
    layer = synth.Layer("graph_f32", B, T, C, OC, "f32", True, init_std=0.01, dout_std=1.0, layer=3)
    x = synth.make_inputs(layer, seed=21)
    t = {k: to_dev(v, "f32") for k, v in x.items()}
    t["out"] = torch.zeros(B * T * OC, dtype=torch.float32, device="cuda")
    outs = ("dinp", "dweight", "dbias", "out")
    init = {k: t[k].clone() for k in outs}

    def calls(stream):
        s = stream.cuda_stream
        return [mm.mmbwd_run(t["dinp"], t["dweight"], t["dbias"], t["dout"], t["inp"], t["weight"], B, T, C, OC,
                             mm.F32, s),
                mm.mmbwd_forward(t["out"], t["inp"], t["weight"], t["dbias"], B, T, C, OC, mm.F32, s)]

    assert mm.mmbwd_release() == mm.OK
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        rcs = calls(s)
    assert rcs == [mm.OK, mm.OK], [mm.strerror(rc) for rc in rcs]
    torch.cuda.synchronize()
    for k in outs:
        t[k].copy_(init[k])
    with torch.cuda.stream(s):
        assert calls(s) == [mm.OK, mm.OK]
    torch.cuda.synchronize()
    eager = {k: t[k].clone() for k in outs}
    for _ in range(2):
        for k in outs:
            t[k].copy_(init[k])
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        for k in outs:
            assert torch.equal(t[k].view(torch.uint8), eager[k].view(torch.uint8)), k
    assert mm.mmbwd_device_status(reset=True)[0] == mm.OK

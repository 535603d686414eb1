"""Out-of-bounds writes and the launch error path, without a sanitizer.

Guard bands: every output lives inside a larger device buffer whose bytes
before and after it hold a canary pattern; after each run, ragged shapes
through every kind of plan (split reductions, both tile widths, no bias,
stochastic rounding, the forward, both fp32 paths, the no-allocation entry,
LayerNorm, encoder one-call and planned), the canaries must be intact and
the inputs unchanged. A TMA store, a partial store or a vector store that
strays past the end (or before the start) of an output shows up here even
where the output itself compares equal to the oracle.

Launch errors: a test hook makes the next launch step of an entry point fail
as the runtime does when it refuses a launch; the call must return
MMBWD_ERR_CUDA with nothing enqueued and the outputs untouched, and the next
call must work.
"""
import numpy as np
import pytest

import linear_layer_gemms_gb300 as mm
import oracle
import synth
from gpu_helpers import TOL, scaled_error, to_host

pytestmark = pytest.mark.gpu

GUARD = 4096  # canary bytes on each side of an output
CANARY = 0xA5


@pytest.fixture(scope="module", autouse=True)
def lib():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    mm.load()
    yield


class Guarded:
    """A device tensor with GUARD canary bytes on each side."""

    def __init__(self, host: np.ndarray, dtype: str):
        import torch

        raw = np.ascontiguousarray(host).view(np.uint8).reshape(-1)
        self.n = raw.size
        buf = np.full(self.n + 2 * GUARD, CANARY, dtype=np.uint8)
        buf[GUARD:GUARD + self.n] = raw
        self.buf = torch.from_numpy(buf).to("cuda:0")
        body = self.buf[GUARD:GUARD + self.n]
        if dtype == "u8":
            self.t = body
        else:
            self.t = body.view(torch.bfloat16 if dtype == "bf16" else torch.float32).view(host.shape)
        assert self.t.data_ptr() % 16 == 0

    def intact(self) -> bool:
        b = self.buf.cpu().numpy()
        return bool((b[:GUARD] == CANARY).all() and (b[GUARD + self.n:] == CANARY).all())


def _inputs_unchanged(dev_inputs, host_inputs, dtype):
    for k, t in dev_inputs.items():
        want = synth.to_f64(host_inputs[k], dtype) if dtype in ("bf16", "f32") else host_inputs[k]
        assert np.array_equal(to_host(t, dtype), want), f"input {k} changed"


def _backward_case(B, T, C, OC, dtype, bias=True, sr=False, static=False, seed=1):
    import torch

    layer = synth.Layer("guard", B, T, C, OC, dtype, bias, init_std=0.01, dout_std=0.1, layer=seed)
    x = synth.make_inputs(layer, seed=seed)
    outs = {k: Guarded(x[k], dtype) for k in ("dinp", "dweight", "dbias")}
    ins = {k: Guarded(x[k], dtype).t for k in ("dout", "inp", "weight")}
    args = (outs["dinp"].t, outs["dweight"].t, outs["dbias"].t if bias else None, ins["dout"], ins["inp"],
            ins["weight"], B, T, C, OC, mm.BF16 if dtype == "bf16" else mm.F32)
    if sr:
        rc = mm.mmbwd_run_sr(*args, 99)
    elif static:
        rc = mm.mmbwd_run_static_scratch(*args)
    else:
        rc = mm.mmbwd_run(*args)
    assert rc == mm.OK, mm.strerror(rc)
    torch.cuda.synchronize()
    assert mm.mmbwd_device_status()[0] == mm.OK
    for k, g in outs.items():
        assert g.intact(), f"canary around {k} overwritten"
    _inputs_unchanged(ins, x, dtype)
    ref = oracle.get("omp").matmul_backward(x["dout"], x["inp"], x["weight"], dtype, x["dinp"], x["dweight"],
                                            bias=bias)
    for k, r in zip(("dinp", "dweight", "dbias"), ref):
        if r is not None:
            assert scaled_error(to_host(outs[k].t, dtype), r) <= TOL[dtype], k
    if not bias:
        assert np.array_equal(to_host(outs["dbias"].t, dtype), synth.to_f64(x["dbias"], dtype))


SHAPES = [(1, 300, 392, 1032), (3, 100, 136, 264), (1, 8, 8, 8), (2, 257, 520, 776)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("plan", ["default", "split3", "tile128", "nobias", "sr", "static"])
def test_backward_bf16_guard_bands(monkeypatch, shape, plan):
    monkeypatch.delenv("MMBWD_GRID", raising=False)
    monkeypatch.setenv("MMBWD_SPLITK", "3" if plan == "split3" else "0")
    if plan == "tile128":
        monkeypatch.setenv("MMBWD_TILE_N", "128,128")
    else:
        monkeypatch.delenv("MMBWD_TILE_N", raising=False)
    _backward_case(*shape, "bf16", bias=plan != "nobias", sr=plan == "sr", static=plan == "static")


@pytest.mark.parametrize("shape", [(1, 300, 392, 1032), (2, 257, 520, 776), (1, 64, 64, 192)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("path", ["x3", "ffma"])
def test_backward_f32_guard_bands(monkeypatch, shape, path):
    monkeypatch.setenv("MMBWD_F32_PATH", path)
    _backward_case(*shape, "f32")


@pytest.mark.parametrize("dtype,path", [("bf16", None), ("f32", "x3"), ("f32", "ffma")])
@pytest.mark.parametrize("shape", [(300, 392, 1032), (129, 136, 264)], ids=lambda s: "x".join(map(str, s)))
def test_forward_guard_bands(monkeypatch, dtype, path, shape):
    import torch

    if path:
        monkeypatch.setenv("MMBWD_F32_PATH", path)
    BT, C, OC = shape
    inp = synth.normal((BT, C), dtype, 2, 61, 0.0, 1.0)
    w = synth.normal((OC, C), dtype, 2, 62, 0.0, 0.02)
    b = synth.normal((OC,), dtype, 2, 63, 0.0, 0.02)
    out = Guarded(synth.normal((BT, OC), dtype, 2, 64), dtype)
    ins = {"inp": Guarded(inp, dtype).t, "weight": Guarded(w, dtype).t, "bias": Guarded(b, dtype).t}
    rc = mm.mmbwd_forward(out.t, ins["inp"], ins["weight"], ins["bias"], 1, BT, C, OC,
                          mm.BF16 if dtype == "bf16" else mm.F32)
    assert rc == mm.OK, mm.strerror(rc)
    torch.cuda.synchronize()
    assert out.intact()
    _inputs_unchanged(ins, {"inp": inp, "weight": w, "bias": b}, dtype)
    ref = oracle.get("omp").forward_rows(inp, w, dtype, bias=b)
    assert scaled_error(to_host(out.t, dtype), ref) <= TOL[dtype]


@pytest.mark.parametrize("dtype,C", [("bf16", 264), ("bf16", 1600), ("f32", 392), ("bf16", 6408), ("f32", 2060)])
def test_layernorm_guard_bands(dtype, C):
    import torch

    p = synth.LNProblem("guard_ln", 2, 77, C, dtype, dout_std=1.0)
    x = synth.make_ln_inputs(p, seed=3)
    orc = oracle.get("omp")
    _, mean, rstd = orc.layernorm_forward(x["inp"], x["weight"], None, dtype, want_out=False)
    mean, rstd = mean.astype(np.float32), rstd.astype(np.float32)
    outs = {k: Guarded(x[k], dtype) for k in ("dinp", "dweight", "dbias")}
    ins = {k: Guarded(x[k], dtype).t for k in ("dout", "inp", "weight")}
    gm, gr = torch.from_numpy(mean).to("cuda:0"), torch.from_numpy(rstd).to("cuda:0")
    rc = mm.lnbwd_run(outs["dinp"].t, outs["dweight"].t, outs["dbias"].t, ins["dout"], ins["inp"], ins["weight"],
                      gm, gr, p.B, p.T, p.C, mm.BF16 if dtype == "bf16" else mm.F32)
    assert rc == mm.OK, mm.strerror(rc)
    torch.cuda.synchronize()
    for k, g in outs.items():
        assert g.intact(), k
    _inputs_unchanged(ins, x, dtype)
    ref = orc.layernorm_dinp_rows(x["dout"], x["inp"], x["weight"], mean, rstd, dtype, dinp_init=x["dinp"])
    assert scaled_error(to_host(outs["dinp"].t, dtype), ref) <= TOL[dtype]


@pytest.mark.parametrize("planned", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_encoder_guard_bands(dtype, planned):
    import torch

    p = synth.EncProblem("guard_enc", 3, 333, 264, 1000, dtype, V_used=200, dout_std=1.0)
    x = synth.make_enc_inputs(p, seed=4)
    outs = {k: Guarded(x[k], dtype) for k in ("dwte", "dwpe")}
    dout = Guarded(x["dout"], dtype).t
    ids = torch.from_numpy(x["inp"]).to("cuda:0")
    dt = mm.BF16 if dtype == "bf16" else mm.F32
    if planned:
        n = mm.encbwd_plan_bytes(p.B, p.T, p.C, p.V, dt)
        plan = Guarded(np.zeros(n, dtype=np.uint8), "u8")
        plan_ptr = plan.buf.data_ptr() + GUARD
        assert plan_ptr % 256 == 0
        assert mm.encbwd_prepare(plan_ptr, n, ids, p.B, p.T, p.C, p.V, dt) == mm.OK
        rc = mm.encbwd_run_planned(outs["dwte"].t, outs["dwpe"].t, dout, plan_ptr, p.B, p.T, p.C, p.V, dt)
    else:
        rc = mm.encbwd_run(outs["dwte"].t, outs["dwpe"].t, dout, ids, p.B, p.T, p.C, p.V, dt)
    assert rc == mm.OK, mm.strerror(rc)
    torch.cuda.synchronize()
    assert mm.mmbwd_device_status()[0] == mm.OK
    for k, g in outs.items():
        assert g.intact(), k
    if planned:
        assert plan.intact()
    assert np.array_equal(to_host(dout, dtype), synth.to_f64(x["dout"], dtype))
    assert np.array_equal(ids.cpu().numpy(), x["inp"])
    rte, rpe = oracle.get("omp").encoder_backward(x["dout"], x["inp"], p.B, p.T, p.V, dtype, x["dwte"], x["dwpe"])
    assert scaled_error(to_host(outs["dwte"].t, dtype), rte) <= TOL[dtype]
    assert scaled_error(to_host(outs["dwpe"].t, dtype), rpe) <= TOL[dtype]


# ----------------------------------------------------------------------------- launch errors

def _fresh_backward(dtype, B=1, T=300, C=392, OC=1032):
    import torch

    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = torch.Generator(device="cpu").manual_seed(9)
    mk = lambda *s: (torch.randn(*s, generator=g) * 0.1).to(tdt).to("cuda:0")  # noqa: E731
    return (B, T, C, OC), {"dinp": mk(B * T, C), "dweight": mk(OC, C), "dbias": mk(OC), "dout": mk(B * T, OC),
                           "inp": mk(B * T, C), "weight": mk(OC, C)}


ORDER = ("dinp", "dweight", "dbias", "dout", "inp", "weight")


@pytest.mark.parametrize("entry", ["run", "run_sr", "static", "run_f32_x3", "run_f32_ffma", "run_split"])
def test_injected_launch_failure_enqueues_nothing(monkeypatch, entry):
    import torch

    dtype = "f32" if entry.startswith("run_f32") else "bf16"
    if entry == "run_f32_x3":
        monkeypatch.setenv("MMBWD_F32_PATH", "x3")
    if entry == "run_f32_ffma":
        monkeypatch.setenv("MMBWD_F32_PATH", "ffma")
    monkeypatch.setenv("MMBWD_SPLITK", "3" if entry in ("run_split", "static") else "0")
    (B, T, C, OC), t = _fresh_backward(dtype)
    before = {k: v.clone() for k, v in t.items()}
    dt = mm.BF16 if dtype == "bf16" else mm.F32
    args = [t[k] for k in ORDER] + [B, T, C, OC, dt]
    call = {"run_sr": lambda: mm.mmbwd_run_sr(*args, 5),
            "static": lambda: mm.mmbwd_run_static_scratch(*args)}.get(entry, lambda: mm.mmbwd_run(*args))
    assert call() == mm.OK  # grows any workspace first
    torch.cuda.synchronize()
    before = {k: v.clone() for k, v in t.items()}
    mm.mmbwd_debug_fail_next_launch(1)
    try:
        assert call() == mm.ERR_CUDA
    finally:
        mm.mmbwd_debug_fail_next_launch(0)
    torch.cuda.synchronize()
    for k in ORDER:
        assert torch.equal(t[k], before[k]), k
    assert mm.mmbwd_device_status()[0] == mm.OK
    assert call() == mm.OK
    torch.cuda.synchronize()
    assert not torch.equal(t["dinp"], before["dinp"])


def test_injected_launch_failure_other_entry_points():
    import torch

    dev = torch.device("cuda:0")
    bf = torch.bfloat16
    BT, C, OC, V = 256, 264, 392, 500
    out = torch.zeros(BT, OC, dtype=bf, device=dev)
    inp, w = torch.ones(BT, C, dtype=bf, device=dev), torch.ones(OC, C, dtype=bf, device=dev)
    mm.mmbwd_debug_fail_next_launch(1)
    assert mm.mmbwd_forward(out, inp, w, None, 1, BT, C, OC, mm.BF16) == mm.ERR_CUDA
    x = {k: torch.zeros(BT, C, dtype=bf, device=dev) for k in ("dinp", "dout", "inp")}
    p = {k: torch.zeros(C, dtype=bf, device=dev) for k in ("dweight", "dbias", "weight")}
    mean, rstd = torch.zeros(BT, device=dev), torch.ones(BT, device=dev)
    mm.mmbwd_debug_fail_next_launch(1)
    assert mm.lnbwd_run(x["dinp"], p["dweight"], p["dbias"], x["dout"], x["inp"], p["weight"], mean, rstd, 1, BT, C,
                        mm.BF16) == mm.ERR_CUDA
    dwte, dwpe = torch.zeros(V, C, dtype=bf, device=dev), torch.zeros(BT, C, dtype=bf, device=dev)
    ids = torch.arange(BT, dtype=torch.int32, device=dev)
    mm.mmbwd_debug_fail_next_launch(1)
    assert mm.encbwd_run(dwte, dwpe, x["dout"] + 1, ids, 1, BT, C, V, mm.BF16) == mm.ERR_CUDA
    mm.mmbwd_debug_fail_next_launch(0)
    torch.cuda.synchronize()
    assert bool((out == 0).all()) and bool((dwte == 0).all()) and bool((dwpe == 0).all())
    assert mm.mmbwd_device_status()[0] == mm.OK

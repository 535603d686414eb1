"""Every entry point accepts only device memory of the current device.

The kernels and their tensor maps address the caller's tensors directly, so
a tensor in host memory (pageable or pinned) must be refused before anything
is enqueued: the call returns MMBWD_ERR_MEMORY and the outputs keep their
values.
"""
import numpy as np
import pytest

import linear_layer_gemms_gb300 as mm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    mm.load()
    yield


def _backward_tensors(B, T, C, OC, dtype):
    import torch

    dev = torch.device("cuda:0")
    g = torch.Generator(device="cpu").manual_seed(5)
    mk = lambda *s: (torch.randn(*s, generator=g) * 0.1).to(dtype).to(dev)  # noqa: E731
    return {"dinp": mk(B * T, C), "dweight": mk(OC, C), "dbias": mk(OC), "dout": mk(B * T, OC),
            "inp": mk(B * T, C), "weight": mk(OC, C)}


def _host_copies(t, pinned):
    out = {k: v.cpu() for k, v in t.items()}
    return {k: (v.pin_memory() if pinned else v) for k, v in out.items()}


ORDER = ("dinp", "dweight", "dbias", "dout", "inp", "weight")


@pytest.mark.parametrize("pinned", [False, True], ids=["pageable", "pinned"])
@pytest.mark.parametrize("which", ORDER)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_backward_refuses_host_memory(pinned, which, dtype):
    import torch

    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    B, T, C, OC = 2, 128, 256, 384
    t = _backward_tensors(B, T, C, OC, tdt)
    before = {k: v.clone() for k, v in t.items()}
    host = _host_copies(t, pinned)
    args = [host[k] if k == which else t[k] for k in ORDER]
    dt = mm.BF16 if dtype == "bf16" else mm.F32
    torch.cuda.synchronize()
    for fn in (mm.mmbwd_run, mm.mmbwd_run_static_scratch):
        assert fn(*args, B, T, C, OC, dt) == mm.ERR_MEMORY
    if dtype == "bf16":
        assert mm.mmbwd_run_sr(*args, B, T, C, OC, dt, 7) == mm.ERR_MEMORY
    torch.cuda.synchronize()
    for k in ORDER:
        assert torch.equal(t[k], before[k]), k  # nothing ran
    if which in ("dinp", "dweight", "dbias"):
        assert torch.equal(host[which], before[which].cpu())
    assert mm.mmbwd_device_status()[0] == mm.OK
    # the same call on device memory goes through
    assert mm.mmbwd_run(*[t[k] for k in ORDER], B, T, C, OC, dt) == mm.OK
    torch.cuda.synchronize()


def test_forward_layernorm_encoder_refuse_host_memory():
    import torch

    dev = torch.device("cuda:0")
    bf = torch.bfloat16
    BT, C, OC = 256, 256, 384
    out = torch.zeros(BT, OC, dtype=bf, device=dev)
    inp, w, b = (torch.ones(BT, C, dtype=bf, device=dev), torch.ones(OC, C, dtype=bf, device=dev),
                 torch.ones(OC, dtype=bf, device=dev))
    assert mm.mmbwd_forward(out, inp.cpu(), w, b, 1, BT, C, OC, mm.BF16) == mm.ERR_MEMORY
    assert mm.mmbwd_forward(out, inp, w, b.cpu().pin_memory(), 1, BT, C, OC, mm.BF16) == mm.ERR_MEMORY
    torch.cuda.synchronize()
    assert bool((out == 0).all())

    # LayerNorm backward: mean in host memory
    x = {k: torch.zeros(BT, C, dtype=bf, device=dev) for k in ("dinp", "dout", "inp")}
    p = {k: torch.zeros(C, dtype=bf, device=dev) for k in ("dweight", "dbias", "weight")}
    mean, rstd = torch.zeros(BT, device=dev), torch.ones(BT, device=dev)
    assert mm.lnbwd_run(x["dinp"], p["dweight"], p["dbias"], x["dout"], x["inp"], p["weight"], mean.cpu(), rstd,
                        1, BT, C, mm.BF16) == mm.ERR_MEMORY

    # encoder backward: token ids in host memory, and a plan in host memory
    V = 512
    dwte = torch.zeros(V, C, dtype=bf, device=dev)
    dwpe = torch.zeros(BT, C, dtype=bf, device=dev)
    dout = torch.ones(BT, C, dtype=bf, device=dev)
    ids = torch.arange(BT, dtype=torch.int32, device=dev)
    assert mm.encbwd_run(dwte, dwpe, dout, ids.cpu(), 1, BT, C, V, mm.BF16) == mm.ERR_MEMORY
    nplan = mm.encbwd_plan_bytes(1, BT, C, V, mm.BF16)
    host_plan = torch.zeros(nplan + 256, dtype=torch.uint8).pin_memory()
    addr = (host_plan.data_ptr() + 255) // 256 * 256
    assert mm.encbwd_prepare(addr, nplan, ids, 1, BT, C, V, mm.BF16) == mm.ERR_MEMORY
    torch.cuda.synchronize()
    assert bool((dwte == 0).all()) and bool((dwpe == 0).all())
    assert "device memory" in mm.strerror(mm.ERR_MEMORY)


def test_empty_tensors_are_not_checked():
    """A tensor with no elements is never touched, so its pointer is not
    checked (the degenerate sizes keep their meaning)."""
    import torch

    dev = torch.device("cuda:0")
    OC = 64
    dbias = torch.full((OC,), 5.0, dtype=torch.bfloat16, device=dev)
    host = np.zeros(64, dtype=np.uint16)
    hp = (host.ctypes.data + 15) // 16 * 16  # a 16-byte aligned host address
    # B*T == 0: dout, inp, dinp are empty; weight and dweight still hold OC x C
    w = torch.ones(OC, 32, dtype=torch.bfloat16, device=dev)
    dw = torch.zeros(OC, 32, dtype=torch.bfloat16, device=dev)
    assert mm.mmbwd_run(hp, dw, dbias, hp, hp, w, 0, 1, 32, OC, mm.BF16) == mm.OK
    torch.cuda.synchronize()
    assert bool((dbias == 0).all())

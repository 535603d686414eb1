"""Helpers for the GPU parity tests: move seeded host inputs to the device,
call the library through its C ABI, bring results back as float64."""
from __future__ import annotations

import numpy as np

import linear_layer_gemms_gb300 as mm
import synth

TOL = {"bf16": 2e-2, "f32": 1e-4}  # |gpu - ref| <= tau * (|ref| + rms(ref))


def torch_dev():
    import torch

    return torch.device("cuda:0")


def to_dev(a: np.ndarray, dtype: str):
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype == "bf16":
        t = t.view(torch.bfloat16)
    return t.to(torch_dev())


def to_host(t, dtype: str) -> np.ndarray:
    import torch

    if dtype == "bf16":
        return synth.bf16_bits_to_f64(t.view(torch.int16).cpu().numpy().view(np.uint16))
    return t.cpu().numpy().astype(np.float64)


def run_gpu(x: dict, B: int, T: int, C: int, OC: int, dtype: str, bias: bool = True, repeat: int = 1):
    """Run mmbwd_run `repeat` times from the given initial buffers; returns the
    device tensors after the last run (outputs accumulate with each run)."""
    import torch

    g = {k: to_dev(v, dtype) for k, v in x.items()}
    for _ in range(repeat):
        rc = mm.mmbwd_run(g["dinp"], g["dweight"], g["dbias"] if bias else None, g["dout"], g["inp"],
                          g["weight"], B, T, C, OC, mm.BF16 if dtype == "bf16" else mm.F32)
        assert rc == mm.OK, mm.strerror(rc)
    torch.cuda.synchronize()
    status, info = mm.mmbwd_device_status(reset=True)
    assert status == mm.OK, (status, info)
    return g


def scaled_error(got: np.ndarray, ref: np.ndarray) -> float:
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    denom = np.abs(ref) + rms
    denom = np.where(denom == 0, 1.0, denom)
    return float(np.max(np.abs(got - ref) / denom))


def assert_close(got, ref, dtype, what=""):
    err = scaled_error(got, ref)
    assert err <= TOL[dtype], f"{what}: scaled error {err:.3e} > {TOL[dtype]}"
    return err

"""Full-size workloads through the C ABI, in the plan the benchmark times,
checked against the oracle on sampled outputs: whole rows of dinp and dweight
(including rows at 128/256-row tile boundaries and the last rows), and every
element of dbias (the oracle's column sums, run with a zero-width inp)."""
import numpy as np
import pytest

import linear_layer_gemms_gb300 as mm
import oracle
import synth
from gpu_helpers import TOL, scaled_error, to_dev, to_host

pytestmark = pytest.mark.gpu

CONFIGS = ["tiny", "attn_proj", "mlp:0", "mlp:1", "lm_head", "xl_fc_bf16", "xl_qkv_bf16",
           "xl_fc_f32", "xl_qkv_f32", "xl_fc_f32@ffma"]  # @ffma: the fp32 FMA kernel forced


@pytest.fixture(scope="module", autouse=True)
def lib():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    mm.load()
    yield


def sample_rows(n, seed):
    """First and last rows, rows around tile edges, and seeded random rows."""
    edges = [0, 1, 127, 128, 129, 255, 256, 257, n // 2, n - 129, n - 128, n - 2, n - 1]
    rng = np.random.default_rng(seed)
    rows = set(r for r in edges if 0 <= r < n)
    rows.update(int(r) for r in rng.integers(0, n, size=min(24, n)))
    return np.array(sorted(rows), dtype=np.int64)


def _layer(name):
    if ":" in name:
        wl, i = name.split(":")
        return synth.WORKLOADS[wl].layers[int(i)]
    return synth.WORKLOADS[name].layers[0]


@pytest.mark.parametrize("name", CONFIGS)
def test_full_size_sampled_parity(name, monkeypatch):
    import torch

    monkeypatch.delenv("MMBWD_SPLITK", raising=False)
    monkeypatch.delenv("MMBWD_GRID", raising=False)
    monkeypatch.delenv("MMBWD_F32_PATH", raising=False)
    if name.endswith("@ffma"):
        name = name[: -len("@ffma")]
        monkeypatch.setenv("MMBWD_F32_PATH", "ffma")
    layer = _layer(name)
    dt = layer.dtype
    x = synth.make_inputs(layer, seed=0)
    g = {k: to_dev(v, dt) for k, v in x.items()}
    rc = mm.mmbwd_run(g["dinp"], g["dweight"], g["dbias"] if layer.bias else None, g["dout"],
                      g["inp"], g["weight"], layer.B, layer.T, layer.C, layer.OC,
                      mm.BF16 if dt == "bf16" else mm.F32)
    assert rc == mm.OK, mm.strerror(rc)
    torch.cuda.synchronize()
    assert mm.mmbwd_device_status()[0] == mm.OK

    orc = oracle.get("omp")
    rows_bt = sample_rows(layer.BT, 1)
    rows_o = sample_rows(layer.OC, 2)
    ref_dinp = orc.dinp_rows(x["dout"], x["weight"], dt, rows_bt, x["dinp"])
    ref_dw, _ = orc.dweight_rows(x["dout"], x["inp"], dt, rows_o, x["dweight"], bias=False)
    got_dinp = to_host(g["dinp"][torch.from_numpy(rows_bt).to(g["dinp"].device)], dt)
    got_dw = to_host(g["dweight"][torch.from_numpy(rows_o).to(g["dweight"].device)], dt)
    e1 = scaled_error(got_dinp, ref_dinp)
    e2 = scaled_error(got_dw, ref_dw)
    assert e1 <= TOL[dt], f"dinp {e1:.3e}"
    assert e2 <= TOL[dt], f"dweight {e2:.3e}"
    if layer.bias:
        empty = np.zeros((layer.BT, 0), dtype=x["inp"].dtype)
        _, ref_db = orc.dweight_rows(x["dout"], empty, dt, None, None, bias=True)
        e3 = scaled_error(to_host(g["dbias"], dt), ref_db)
        assert e3 <= TOL[dt], f"dbias {e3:.3e}"
    else:  # no bias requested: dbias untouched
        assert np.array_equal(to_host(g["dbias"], dt), synth.to_f64(x["dbias"], dt))


def _ordered(bits_i16):
    """bf16 patterns as integers in value order (adjacent bf16 values differ by 1)."""
    b = bits_i16.astype(np.int32) & 0xFFFF
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


@pytest.mark.parametrize("name", ["mlp:0", "mlp:1", "attn_proj"])
def test_full_size_stochastic_rounding(name, monkeypatch):
    """mmbwd_run_sr in the benchmark's plan (attn_proj: a split reduction):
    every output is one bf16 step or less from mmbwd_run's on the same inputs
    (the same fp32 value rounded to a neighbour), a plausible share differs,
    sampled rows match the oracle, and the same seed repeats the same bits."""
    import torch

    monkeypatch.delenv("MMBWD_SPLITK", raising=False)
    monkeypatch.delenv("MMBWD_GRID", raising=False)
    layer = _layer(name)
    x = synth.make_inputs(layer, seed=0)

    def run(seed):
        g = {k: to_dev(v, "bf16") for k, v in x.items()}
        args = (g["dinp"], g["dweight"], g["dbias"], g["dout"], g["inp"], g["weight"], layer.B, layer.T, layer.C,
                layer.OC, mm.BF16)
        rc = mm.mmbwd_run(*args) if seed is None else mm.mmbwd_run_sr(*args, seed)
        assert rc == mm.OK, mm.strerror(rc)
        torch.cuda.synchronize()
        assert mm.mmbwd_device_status()[0] == mm.OK
        return g

    rne, sr, sr2 = run(None), run(2024), run(2024)
    for k in ("dinp", "dweight", "dbias"):
        a = _ordered(rne[k].view(torch.int16).cpu().numpy())
        b = _ordered(sr[k].view(torch.int16).cpu().numpy())
        assert np.max(np.abs(a - b)) <= 1, k
        if k != "dbias":
            frac = np.mean(a != b)
            assert 0.10 < frac < 0.45, (k, frac)
        assert torch.equal(sr[k], sr2[k]), k
    orc = oracle.get("omp")
    rows_bt = sample_rows(layer.BT, 3)
    ref = orc.dinp_rows(x["dout"], x["weight"], "bf16", rows_bt, x["dinp"])
    got = to_host(sr["dinp"][torch.from_numpy(rows_bt).to(sr["dinp"].device)], "bf16")
    assert scaled_error(got, ref) <= TOL["bf16"]

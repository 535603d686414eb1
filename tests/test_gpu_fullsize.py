"""Full-size workloads through the C ABI, in the plan the benchmark times,
checked against the oracle element by element (every element of dinp,
dweight and dbias, computed by the OpenMP build of the oracle), and run ten
times from identical buffers to show that the results repeat bit for bit."""
import numpy as np
import pytest

import linear_layer_gemms_gb300 as mm
import oracle
import synth
from gpu_helpers import TOL, scaled_error, to_dev, to_host

pytestmark = pytest.mark.gpu

CONFIGS = ["tiny", "qkv", "attn_proj", "mlp:0", "mlp:1", "lm_head", "xl_fc_bf16", "xl_qkv_bf16",
           "xl_fc_f32", "xl_qkv_f32", "xl_fc_f32@ffma"]  # @ffma: the fp32 FMA kernel forced
REPEATS = 10


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


def _setup(name, monkeypatch):
    monkeypatch.delenv("MMBWD_SPLITK", raising=False)
    monkeypatch.delenv("MMBWD_GRID", raising=False)
    monkeypatch.delenv("MMBWD_TILE_N", raising=False)
    monkeypatch.delenv("MMBWD_F32_PATH", raising=False)
    if name.endswith("@ffma"):
        name = name[: -len("@ffma")]
        monkeypatch.setenv("MMBWD_F32_PATH", "ffma")
    layer = _layer(name)
    return layer, synth.make_inputs(layer, seed=0)


def _run(g, layer):
    import torch

    rc = mm.mmbwd_run(g["dinp"], g["dweight"], g["dbias"] if layer.bias else None, g["dout"],
                      g["inp"], g["weight"], layer.B, layer.T, layer.C, layer.OC,
                      mm.BF16 if layer.dtype == "bf16" else mm.F32)
    assert rc == mm.OK, mm.strerror(rc)
    torch.cuda.synchronize()
    assert mm.mmbwd_device_status()[0] == mm.OK


@pytest.mark.parametrize("name", CONFIGS)
def test_full_size_parity(name, monkeypatch):
    layer, x = _setup(name, monkeypatch)
    dt = layer.dtype
    g = {k: to_dev(v, dt) for k, v in x.items()}
    _run(g, layer)
    ref = oracle.get("omp").matmul_backward(x["dout"], x["inp"], x["weight"], dt, x["dinp"], x["dweight"],
                                            bias=layer.bias)
    for key, r in zip(("dinp", "dweight", "dbias"), ref):
        if r is None:  # no bias requested: dbias untouched
            assert np.array_equal(to_host(g["dbias"], dt), synth.to_f64(x["dbias"], dt))
            continue
        got = to_host(g[key], dt)
        assert got.shape == r.shape
        err = scaled_error(got, r)
        assert err <= TOL[dt], f"{key} {err:.3e}"


@pytest.mark.parametrize("name", [c for c in CONFIGS if c != "tiny"])
def test_full_size_bitwise_repeatable(name, monkeypatch):
    """The benchmarked plan (split reductions with their fixup launch, the LM
    head's long schedule, the fp32 paths) run ten times from identical
    buffers: every output bit is the same each time."""
    import torch

    layer, x = _setup(name, monkeypatch)
    dt = layer.dtype
    g0 = {k: to_dev(v, dt) for k, v in x.items()}
    first = None
    for _ in range(REPEATS):
        g = {k: v.clone() for k, v in g0.items()}
        _run(g, layer)
        bits = [g[k].view(torch.int16 if dt == "bf16" else torch.int32) for k in ("dinp", "dweight", "dbias")]
        if first is None:
            first = bits
            continue
        for k, a, b in zip(("dinp", "dweight", "dbias"), first, bits):
            assert torch.equal(a, b), k


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

"""mmbwd_run_sr (stochastic rounding of the bf16 outputs) through the C ABI
against the oracle (oracle/sr_oracle.c).

Integer problems whose fp32 sums are exact but whose results need more than
bf16's eight significant bits: the value rounded is then the same on both
sides, so every output element must match the oracle bit for bit — direct
epilogue, forced split reductions, no bias, C = 0 (column sums only). Normal
inputs: within the parity tolerance, repeatable for a seed, different for
another seed, and unbiased (the mean over seeds is closer to the exact value
than round-to-nearest)."""
import numpy as np
import pytest

import linear_layer_gemms_gb300 as mm
import oracle
import synth
from gpu_helpers import assert_close, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    mm.load()
    yield


def int_problem(BT, C, OC, seed, lim=3):
    """bf16 bit patterns of small integers (exact in bf16 and in every fp32 sum)."""
    rng = np.random.default_rng(seed)

    def ints(shape, lo, hi):
        v = rng.integers(lo, hi + 1, size=shape).astype(np.float32)
        return (v.view(np.uint32) >> 16).astype(np.uint16)  # exact: |v| <= 256

    return {"dout": ints((BT, OC), -lim, lim), "inp": ints((BT, C), -lim, lim), "weight": ints((OC, C), -lim, lim),
            "dinp": ints((BT, C), -200, 200), "dweight": ints((OC, C), -200, 200), "dbias": ints((OC,), -5, 5)}


def run_sr(x, BT, C, OC, seed, bias=True):
    import torch

    g = {k: to_dev(v, "bf16") for k, v in x.items()}
    rc = mm.mmbwd_run_sr(g["dinp"], g["dweight"], g["dbias"] if bias else None, g["dout"], g["inp"], g["weight"],
                         1, BT, C, OC, mm.BF16, seed)
    assert rc == mm.OK, mm.strerror(rc)
    torch.cuda.synchronize()
    assert mm.mmbwd_device_status(reset=True)[0] == mm.OK
    return g


def bits(t):
    import torch

    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def check_exact(x, g, seed, bias=True):
    want = oracle.get("st").matmul_backward_sr(x["dout"], x["inp"], x["weight"], seed, x["dinp"], x["dweight"], bias)
    assert np.array_equal(bits(g["dinp"]), want[0]), "dinp"
    assert np.array_equal(bits(g["dweight"]), want[1]), "dweight"
    if bias:
        assert np.array_equal(bits(g["dbias"]), want[2]), "dbias"


@pytest.mark.parametrize("shape", [(400, 200, 264), (256, 256, 512), (1000, 72, 136)], ids=str)
def test_sr_integer_exact(shape):
    BT, C, OC = shape
    x = int_problem(BT, C, OC, seed=BT + C)
    seed = 0x5EED0000 + OC
    g = run_sr(x, BT, C, OC, seed)
    check_exact(x, g, seed)
    # results of more than eight significant bits were rounded (both ways)
    exact = oracle.get("st").matmul_backward(x["dout"], x["inp"], x["weight"], "bf16", x["dinp"], x["dweight"])[0]
    got = to_host(g["dinp"], "bf16")
    assert np.any(got > exact) and np.any(got < exact)


@pytest.mark.parametrize("splits", [2, 3])
def test_sr_integer_exact_split_reduction(monkeypatch, splits):
    monkeypatch.setenv("MMBWD_SPLITK", str(splits))
    BT, C, OC = 2048, 64, 128
    assert mm.mmbwd_plan_info(1, BT, C, OC, mm.BF16, 0)["splits"] == splits
    x = int_problem(BT, C, OC, seed=splits)
    g = run_sr(x, BT, C, OC, seed=12345)
    check_exact(x, g, 12345)


def test_sr_integer_exact_no_bias_and_no_columns():
    BT, C, OC = 300, 128, 96
    x = int_problem(BT, C, OC, seed=9)
    before = x["dbias"].copy()
    g = run_sr(x, BT, C, OC, seed=7, bias=False)
    check_exact(x, g, 7, bias=False)
    assert np.array_equal(bits(g["dbias"]), before)
    # C == 0: only the column sums of dout, rounded stochastically
    x0 = int_problem(5000, 0, 64, seed=10, lim=7)
    g0 = run_sr(x0, 5000, 0, 64, seed=8)
    want = oracle.get("st").sr_round(synth.bf16_bits_to_f64(x0["dout"]).sum(axis=0), 8, oracle.SR_DBIAS)
    assert np.array_equal(bits(g0["dbias"]), want)


def normal_problem(seed):
    """bf16 (RNE) normal inputs of the GPT-2 scales at a small ragged shape."""
    rng = np.random.default_rng(seed)
    BT, C, OC = 256, 192, 320

    def bf(shape, std):
        u = (rng.normal(size=shape) * std).astype(np.float32).view(np.uint32).astype(np.uint64)
        return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)

    x = {"dout": bf((BT, OC), 1e-2), "inp": bf((BT, C), 1.0), "weight": bf((OC, C), 0.02),
         "dinp": bf((BT, C), 1e-2), "dweight": bf((OC, C), 1e-2), "dbias": bf((OC,), 1e-2)}
    return x, BT, C, OC


def test_sr_normal_inputs_tolerance_repeat_and_seed():
    x, BT, C, OC = normal_problem(3)
    ref = oracle.get("st").matmul_backward(x["dout"], x["inp"], x["weight"], "bf16", x["dinp"], x["dweight"])
    a = run_sr(x, BT, C, OC, seed=1)
    for k, r in zip(("dinp", "dweight", "dbias"), ref):
        assert_close(to_host(a[k], "bf16"), r, "bf16", k)
    b = run_sr(x, BT, C, OC, seed=1)
    c = run_sr(x, BT, C, OC, seed=2)
    for k in ("dinp", "dweight", "dbias"):
        assert np.array_equal(bits(a[k]), bits(b[k])), k
    assert np.mean(bits(a["dinp"]) != bits(c["dinp"])) > 0.2


def test_sr_unbiased_over_seeds():
    """The mean of 16 stochastically rounded results is closer to the exact
    values than one round-to-nearest result (which mmbwd_run gives)."""
    import torch

    x, BT, C, OC = normal_problem(4)
    exact = oracle.get("st").matmul_backward(x["dout"], x["inp"], x["weight"], "bf16", x["dinp"], x["dweight"])[0]
    runs = [to_host(run_sr(x, BT, C, OC, seed=100 + s)["dinp"], "bf16") for s in range(16)]
    g = {k: to_dev(v, "bf16") for k, v in x.items()}
    assert mm.mmbwd_run(g["dinp"], g["dweight"], g["dbias"], g["dout"], g["inp"], g["weight"], 1, BT, C, OC,
                        mm.BF16) == mm.OK
    torch.cuda.synchronize()
    rne = to_host(g["dinp"], "bf16")
    err_sr = np.mean(np.abs(np.mean(runs, axis=0) - exact))
    err_rne = np.mean(np.abs(rne - exact))
    assert err_sr < 0.6 * err_rne, (err_sr, err_rne)

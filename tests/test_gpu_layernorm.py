"""The LayerNorm backward (lnbwd_run) through the C ABI against the oracle,
element by element: every dinp row at small sizes (several blocks, ragged
row counts and column widths), sampled dinp rows plus all of dweight and dbias
at the full sizes of the page's benchmark, run-to-run bitwise determinism,
accumulation over calls, empty problems and argument errors."""
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


def stats(x, dtype):
    """fp32 row statistics, as the forward caches them (oracle forward, double)."""
    C = x["inp"].shape[1]
    ones = synth.round_to(np.ones(C), dtype)
    _, m, r = oracle.get("omp").layernorm_forward(x["inp"], ones, None, dtype, want_out=False)
    return m.astype(np.float32), r.astype(np.float32)


def run_ln(x, mean, rstd, B, T, C, dtype, repeat=1):
    import torch

    g = {k: to_dev(v, dtype) for k, v in x.items()}
    gm, gr = to_dev(mean, "f32"), to_dev(rstd, "f32")
    for _ in range(repeat):
        rc = mm.lnbwd_run(g["dinp"], g["dweight"], g["dbias"], g["dout"], g["inp"], g["weight"], gm, gr,
                          B, T, C, mm.BF16 if dtype == "bf16" else mm.F32)
        assert rc == mm.OK, mm.strerror(rc)
    torch.cuda.synchronize()
    return g


def problem(B, T, C, dtype, seed=0):
    return synth.make_ln_inputs(synth.LNProblem("t", B, T, C, dtype, dout_std=1.0), seed)


def check(x, g, mean, rstd, dtype, rows=None):
    orc = oracle.get("omp")
    ref = orc.layernorm_dinp_rows(x["dout"], x["inp"], x["weight"], mean, rstd, dtype, rows=rows,
                                  dinp_init=x["dinp"])
    got = to_host(g["dinp"], dtype)
    assert_close(got if rows is None else got[rows], ref, dtype, "dinp")
    dw, db = orc.layernorm_params(x["dout"], x["inp"], mean, rstd, dtype, x["dweight"], x["dbias"])
    assert_close(to_host(g["dweight"], dtype), dw, dtype, "dweight")
    assert_close(to_host(g["dbias"], dtype), db, dtype, "dbias")


# (B, T, C): one row; fewer rows than warps; ragged rows over many blocks;
# column widths that leave lanes idle (C = 8, 264) or use the widest lanes;
# rows wider than the fused kernel takes (bf16 above 4096, fp32 above 2048:
# row sums, then column tiles), ragged in both directions.
SHAPES = {"bf16": [(1, 1, 8), (1, 5, 264), (3, 37, 264), (2, 333, 768), (2, 64, 1600), (1, 300, 4096),
                   (1, 3, 4104), (2, 150, 6400), (1, 77, 12800), (3, 501, 8200)],
          "f32": [(1, 1, 4), (2, 48, 72), (3, 37, 260), (2, 333, 768), (1, 300, 1600), (1, 200, 2048),
                  (1, 7, 2052), (2, 150, 5000), (1, 64, 16384)]}


@pytest.mark.parametrize("dtype,shape", [(d, s) for d in SHAPES for s in SHAPES[d]],
                         ids=lambda v: v if isinstance(v, str) else "x".join(map(str, v)))
def test_layernorm_parity(dtype, shape):
    B, T, C = shape
    x = problem(B, T, C, dtype)
    mean, rstd = stats(x, dtype)
    g = run_ln(x, mean, rstd, B, T, C, dtype)
    check(x, g, mean, rstd, dtype)


@pytest.mark.parametrize("name", ["ln_tiny", "ln_gpt2_small", "ln_xl", "ln_xl_f32"])
def test_layernorm_workloads(name):
    """The workload shapes bench.py times (B=8, T=1024, C=768 / 1600): 512
    sampled dinp rows (first, last, random) and every dweight / dbias element."""
    p = synth.LN_WORKLOADS[name]
    x = synth.make_ln_inputs(p)
    mean, rstd = stats(x, p.dtype)
    g = run_ln(x, mean, rstd, p.B, p.T, p.C, p.dtype)
    rng = np.random.default_rng(5)
    rows = None if p.BT <= 512 else np.unique(np.concatenate(
        [[0, p.BT - 1], rng.choice(p.BT, 510, replace=False)]))
    check(x, g, mean, rstd, p.dtype, rows)


@pytest.mark.parametrize("dtype,C", [("bf16", 1600), ("f32", 768), ("bf16", 6400), ("f32", 4096)])
def test_layernorm_deterministic(dtype, C):
    """Ten runs from the same initial buffers give identical bits (the fused
    kernel and the two-pass path for wide rows)."""
    import torch

    B, T = 4, 700
    x = problem(B, T, C, dtype, seed=3)
    mean, rstd = stats(x, dtype)
    first = None
    for _ in range(10):
        g = run_ln(x, mean, rstd, B, T, C, dtype)
        cur = [bytes(g[k].cpu().view(-1).view(torch.uint8).numpy()) for k in ("dinp", "dweight", "dbias")]
        if first is None:
            first = cur
        else:
            assert cur == first


def test_layernorm_accumulates_over_calls():
    """Two calls add two gradients: dweight and dbias after two calls equal the
    oracle's with the first call's result as the initial value."""
    B, T, C, dtype = 2, 100, 264, "f32"
    x = problem(B, T, C, dtype, seed=4)
    mean, rstd = stats(x, dtype)
    g = run_ln(x, mean, rstd, B, T, C, dtype, repeat=2)
    orc = oracle.get("omp")
    dw1, db1 = orc.layernorm_params(x["dout"], x["inp"], mean, rstd, dtype, x["dweight"], x["dbias"])
    dw2, db2 = orc.layernorm_params(x["dout"], x["inp"], mean, rstd, dtype, dw1.astype(np.float32),
                                    db1.astype(np.float32))
    assert_close(to_host(g["dweight"], dtype), dw2, dtype, "dweight")
    assert_close(to_host(g["dbias"], dtype), db2, dtype, "dbias")


def test_layernorm_empty_and_errors():
    import torch

    x = problem(1, 4, 16, "bf16")
    mean, rstd = stats(x, "bf16")
    g = {k: to_dev(v, "bf16") for k, v in x.items()}
    gm, gr = to_dev(mean, "f32"), to_dev(rstd, "f32")
    before = {k: v.clone() for k, v in g.items()}
    # B*T == 0 or C == 0: the empty sums leave every output unchanged
    assert mm.lnbwd_run(g["dinp"], g["dweight"], g["dbias"], g["dout"], g["inp"], g["weight"], gm, gr,
                        0, 4, 16, mm.BF16) == mm.OK
    assert mm.lnbwd_run(g["dinp"], g["dweight"], g["dbias"], g["dout"], g["inp"], g["weight"], gm, gr,
                        1, 4, 0, mm.BF16) == mm.OK
    torch.cuda.synchronize()
    for k in g:
        assert g[k].equal(before[k]), k
    # an output overlapping an input, a misaligned pointer, C above the limit:
    # rejected on the host, nothing enqueued
    assert mm.lnbwd_run(g["dout"], g["dweight"], g["dbias"], g["dout"], g["inp"], g["weight"], gm, gr,
                        1, 4, 16, mm.BF16) == mm.ERR_ALIAS
    assert mm.lnbwd_run(g["dinp"].data_ptr() + 2, g["dweight"], g["dbias"], g["dout"], g["inp"],
                        g["weight"], gm, gr, 1, 4, 16, mm.BF16) == mm.ERR_ALIGN
    assert mm.lnbwd_run(g["dinp"], g["dweight"], g["dbias"], g["dout"], g["inp"], g["weight"], gm, gr,
                        1, 1, (1 << 20) + 8, mm.BF16) == mm.ERR_SHAPE
    torch.cuda.synchronize()
    for k in g:
        assert g[k].equal(before[k]), k

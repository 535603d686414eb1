"""The encoder backward (encbwd_run) through the C ABI against the oracle,
element by element on every dwte and dwpe element: ragged position counts
(not powers of two), a token repeated far beyond one chunk, the largest sort
(B*T = 16384), the GPT-2 small workload with Zipf-distributed tokens,
run-to-run bitwise determinism, a token id out of range, empty problems; with
stochastic rounding (encbwd_run_sr), bit-exact against the oracle on integer
problems (fp32 sums exact, results wider than bf16) and repeatable per seed."""
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


def run_enc(x, B, T, C, V, dtype):
    import torch

    g = {k: to_dev(x[k], dtype) for k in ("dout", "dwte", "dwpe")}
    gi = torch.from_numpy(x["inp"]).to("cuda:0")
    rc = mm.encbwd_run(g["dwte"], g["dwpe"], g["dout"], gi, B, T, C, V, mm.BF16 if dtype == "bf16" else mm.F32)
    assert rc == mm.OK, mm.strerror(rc)
    torch.cuda.synchronize()
    return g


def check(x, g, B, T, V, dtype):
    ref_wte, ref_wpe = oracle.get("st").encoder_backward(x["dout"], x["inp"], B, T, V, dtype, x["dwte"], x["dwpe"])
    assert_close(to_host(g["dwte"], dtype), ref_wte, dtype, "dwte")
    assert_close(to_host(g["dwpe"], dtype), ref_wpe, dtype, "dwpe")


def problem(B, T, C, V, dtype, v_used=None, seed=0):
    p = synth.EncProblem("t", B, T, C, V, dtype, V_used=v_used or V, dout_std=1.0)
    return synth.make_enc_inputs(p, seed)


# (B, T, C, V, dtype): one position; a one-token vocabulary; a ragged count;
# fp32; Zipf with long repeats; every position the same token (one segment of
# many chunks); the largest sort with a narrow C; a vocabulary of 2^16 ids.
CASES = [(1, 1, 8, 3, "bf16"), (1, 40, 16, 1, "f32"), (2, 37, 264, 50, "bf16"), (2, 64, 72, 97, "f32"),
         (4, 300, 768, 1000, "bf16"), (3, 500, 128, 7, "f32"), (16, 1024, 16, 50304, "bf16"),
         (2, 700, 32, 65536, "bf16")]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_encoder_parity(case):
    B, T, C, V, dtype = case
    x = problem(B, T, C, V, dtype)
    g = run_enc(x, B, T, C, V, dtype)
    check(x, g, B, T, V, dtype)
    assert mm.mmbwd_device_status()[0] == mm.OK


def test_encoder_single_token():
    B, T, C, V, dtype = 4, 1000, 256, 10, "bf16"
    x = problem(B, T, C, V, dtype)
    x["inp"][:] = 3
    g = run_enc(x, B, T, C, V, dtype)
    check(x, g, B, T, V, dtype)


@pytest.mark.parametrize("name", ["enc_tiny", "enc_gpt2_small", "enc_gpt2_small_f32"])
def test_encoder_workloads(name):
    p = synth.ENC_WORKLOADS[name]
    x = synth.make_enc_inputs(p)
    g = run_enc(x, p.B, p.T, p.C, p.V, p.dtype)
    check(x, g, p.B, p.T, p.V, p.dtype)


def test_encoder_deterministic():
    import torch

    p = synth.ENC_WORKLOADS["enc_gpt2_small"]
    x = synth.make_enc_inputs(p, seed=2)
    outs = []
    for _ in range(3):
        g = run_enc(x, p.B, p.T, p.C, p.V, p.dtype)
        outs.append([bytes(g[k].cpu().view(-1).view(torch.uint8).numpy()) for k in ("dwte", "dwpe")])
    assert outs[0] == outs[1] == outs[2]


def test_encoder_bad_token_reported():
    """A token id outside [0, V) is skipped and reported; with its dout row
    zero, every output equals the oracle's with that id replaced."""
    B, T, C, V, dtype = 1, 50, 64, 20, "f32"
    x = problem(B, T, C, V, dtype)
    x["inp"][17] = V + 5
    x["dout"][17] = 0.0
    mm.mmbwd_device_status(reset=True)
    g = run_enc(x, B, T, C, V, dtype)
    status, info = mm.mmbwd_device_status(reset=True)
    assert status == mm.ERR_SHAPE and info[0] == 17 and info[1] == V + 5
    fixed = dict(x)
    fixed["inp"] = x["inp"].copy()
    fixed["inp"][17] = 0
    check(fixed, g, B, T, V, dtype)


def test_encoder_empty_and_errors():
    import torch

    x = problem(1, 8, 16, 5, "bf16")
    g = {k: to_dev(x[k], "bf16") for k in ("dout", "dwte", "dwpe")}
    gi = torch.from_numpy(x["inp"]).to("cuda:0")
    before = {k: v.clone() for k, v in g.items()}
    assert mm.encbwd_run(g["dwte"], g["dwpe"], g["dout"], gi, 0, 8, 16, 5, mm.BF16) == mm.OK
    assert mm.encbwd_run(g["dwte"], g["dwpe"], g["dout"], gi, 1, 8, 0, 5, mm.BF16) == mm.OK
    assert mm.encbwd_run(g["dwte"], g["dwte"], g["dout"], gi, 1, 8, 16, 5, mm.BF16) == mm.ERR_ALIAS
    assert mm.encbwd_run(g["dwte"], g["dwpe"], g["dout"], gi.data_ptr() + 2, 1, 8, 16, 5, mm.BF16) == mm.ERR_ALIGN
    torch.cuda.synchronize()
    for k in g:
        assert g[k].equal(before[k]), k


def test_encoder_bad_tokens_among_last_id():
    """Invalid ids interleaved with copies of the largest valid id of a
    power-of-two vocabulary: the invalid positions are skipped (their dout
    rows are zero here) and every valid one is summed."""
    B, T, C, V, dtype = 2, 150, 64, 8, "bf16"
    x = problem(B, T, C, V, dtype)
    bad = np.arange(3, B * T, 7)
    x["inp"][bad - 1] = V - 1
    x["inp"][bad] = np.array([V, -1, 100, V + 1])[np.arange(bad.size) % 4]
    x["dout"][bad] = 0
    mm.mmbwd_device_status(reset=True)
    g = run_enc(x, B, T, C, V, dtype)
    status, info = mm.mmbwd_device_status(reset=True)
    assert status == mm.ERR_SHAPE and info[0] in set(bad.tolist())
    fixed = dict(x)
    fixed["inp"] = x["inp"].copy()
    fixed["inp"][bad] = 0
    check(fixed, g, B, T, V, dtype)


def test_encoder_sr_integer_exact_and_repeatable():
    import torch

    B, T, C, V = 4, 500, 64, 40
    rng = np.random.default_rng(17)

    def ints(shape, lim, scale=1):
        v = (rng.integers(-lim, lim + 1, size=shape) * scale).astype(np.float32)  # exact in bf16: |v / scale| < 256
        return (v.view(np.uint32) >> 16).astype(np.uint16)

    # initial values multiples of 8 up to 1600, so that old + sum needs more
    # than bf16's eight significant bits; the last 5 ids are unused (rows kept)
    x = {"dout": ints((B * T, C), 3), "dwte": ints((V, C), 200, 8), "dwpe": ints((T, C), 200, 8),
         "inp": synth.zipf_tokens(B * T, V - 5, 1.1, 3, 0)}
    want = oracle.get("st").encoder_backward_sr(x["dout"], x["inp"], B, T, V, 99, x["dwte"], x["dwpe"])
    outs = []
    for seed in (99, 99, 100):
        g = {k: to_dev(x[k], "bf16") for k in ("dout", "dwte", "dwpe")}
        gi = torch.from_numpy(x["inp"]).to("cuda:0")
        assert mm.encbwd_run_sr(g["dwte"], g["dwpe"], g["dout"], gi, B, T, C, V, mm.BF16, seed) == mm.OK
        torch.cuda.synchronize()
        outs.append([g[k].view(torch.int16).cpu().numpy().view(np.uint16) for k in ("dwte", "dwpe")])
    assert np.array_equal(outs[0][0], want[0]) and np.array_equal(outs[0][1], want[1])
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
    exact = synth.bf16_bits_to_f64(x["dwpe"]) + synth.bf16_bits_to_f64(x["dout"]).reshape(B, T, C).sum(axis=0)
    trunc = ((exact.astype(np.float32).view(np.uint32) >> 16) << 16).view(np.float32).astype(np.float64)
    rounded = trunc != exact  # sums that are not bf16 values
    assert rounded.mean() > 0.5  # most sums are not bf16 values
    assert np.mean(outs[0][1][rounded] != outs[2][1][rounded]) > 0.2  # another seed, other roundings
    got = synth.bf16_bits_to_f64(outs[0][1])
    assert np.any(got > exact) and np.any(got < exact)  # rounded both ways
    assert mm.encbwd_run_sr(None, None, None, None, B, T, C, V, mm.F32, 1) == mm.ERR_DTYPE


def test_encoder_planned_matches_one_call_and_plan_reuse():
    """encbwd_prepare + encbwd_run_planned gives the bits of encbwd_run (and of
    encbwd_run_sr with a seed); one plan serves repeated runs; a plan of
    another problem is reported and changes nothing."""
    import torch

    for name in ("enc_gpt2_small", "enc_tiny"):
        p = synth.ENC_WORKLOADS[name]
        x = synth.make_enc_inputs(p, seed=5)
        dt = mm.BF16 if p.dtype == "bf16" else mm.F32
        gi = torch.from_numpy(x["inp"]).to("cuda:0")
        one = run_enc(x, p.B, p.T, p.C, p.V, p.dtype)
        nbytes = mm.encbwd_plan_bytes(p.B, p.T, p.C, p.V, dt)
        plan = torch.empty(nbytes, dtype=torch.uint8, device="cuda:0")
        assert mm.encbwd_prepare(plan, nbytes, gi, p.B, p.T, p.C, p.V, dt) == mm.OK
        for _ in range(2):  # the same plan twice, from fresh initial values
            g = {k: to_dev(x[k], p.dtype) for k in ("dout", "dwte", "dwpe")}
            assert mm.encbwd_run_planned(g["dwte"], g["dwpe"], g["dout"], plan, p.B, p.T, p.C, p.V, dt) == mm.OK
            torch.cuda.synchronize()
            for k in ("dwte", "dwpe"):
                assert torch.equal(g[k].view(torch.uint8), one[k].view(torch.uint8)), (name, k)
        assert mm.mmbwd_device_status(reset=True)[0] == mm.OK
        if p.dtype == "bf16":
            a = {k: to_dev(x[k], "bf16") for k in ("dout", "dwte", "dwpe")}
            b = {k: to_dev(x[k], "bf16") for k in ("dout", "dwte", "dwpe")}
            assert mm.encbwd_run_sr(a["dwte"], a["dwpe"], a["dout"], gi, p.B, p.T, p.C, p.V, dt, 77) == mm.OK
            assert mm.encbwd_run_planned(b["dwte"], b["dwpe"], b["dout"], plan, p.B, p.T, p.C, p.V, dt, 77) == mm.OK
            torch.cuda.synchronize()
            for k in ("dwte", "dwpe"):
                assert torch.equal(a[k].view(torch.uint8), b[k].view(torch.uint8)), ("sr", k)
            # the plan of another problem (T halved): reported, nothing written
            c = {k: to_dev(x[k], "bf16") for k in ("dout", "dwte", "dwpe")}
            before = {k: v.clone() for k, v in c.items()}
            mm.mmbwd_device_status(reset=True)
            assert mm.encbwd_run_planned(c["dwte"], c["dwpe"], c["dout"], plan, p.B, p.T // 2, p.C, p.V, dt) == mm.OK
            torch.cuda.synchronize()
            status, info = mm.mmbwd_device_status(reset=True)
            assert status == mm.ERR_SHAPE and info[0] == -1
            for k in c:
                assert torch.equal(c[k], before[k]), k


# Above 16384 positions the sort runs over many blocks (a radix sort of
# 64-bit keys, three launches a pass): ragged counts just past the one-block
# limit, GPT-2 sized batches of 65536 positions, a one-token run spanning
# every tile, invalid ids, fp32 and stochastic rounding, the planned form.
LARGE = [(1, 16385, 64, 50304, "bf16"), (2, 10007, 96, 1000, "f32"), (64, 1024, 768, 50304, "bf16"),
         (16, 4096, 128, 131071, "bf16")]


@pytest.mark.parametrize("case", LARGE, ids=lambda c: "x".join(map(str, c)))
def test_encoder_multiblock_sort_parity(case):
    B, T, C, V, dtype = case
    x = problem(B, T, C, V, dtype, v_used=min(V, 50257))
    g = run_enc(x, B, T, C, V, dtype)
    check(x, g, B, T, V, dtype)
    assert mm.mmbwd_device_status()[0] == mm.OK
    again = run_enc(x, B, T, C, V, dtype)
    for k in ("dwte", "dwpe"):
        assert np.array_equal(to_host(g[k], dtype), to_host(again[k], dtype)), k


def test_encoder_multiblock_one_token_and_invalid_ids():
    B, T, C, V, dtype = 4, 9000, 64, 300, "bf16"
    x = problem(B, T, C, V, dtype)
    x["inp"][:] = 7
    g = run_enc(x, B, T, C, V, dtype)
    check(x, g, B, T, V, dtype)
    # invalid ids are skipped (and reported), the rest is summed
    x = problem(B, T, C, V, dtype, seed=2)
    bad = np.array([5, 17000, 35999])
    x["inp"][bad] = V + 3
    g = run_enc(x, B, T, C, V, dtype)
    status, info = mm.mmbwd_device_status(reset=True)
    assert status == mm.ERR_SHAPE and info[1] == V + 3
    keep = x["inp"] < V
    ref_x = dict(x, inp=np.where(keep, x["inp"], 0).astype(np.int32),
                 dout=np.where(keep[:, None], x["dout"], 0).astype(x["dout"].dtype))
    ref_wte, _ = oracle.get("omp").encoder_backward(ref_x["dout"], ref_x["inp"], B, T, V, dtype, x["dwte"], x["dwpe"])
    assert_close(to_host(g["dwte"], dtype), ref_wte, dtype, "dwte")


def test_encoder_multiblock_planned_and_sr():
    import torch

    B, T, C, V = 8, 4096, 256, 50304
    x = problem(B, T, C, V, "bf16", v_used=50257, seed=3)
    one = run_enc(x, B, T, C, V, "bf16")
    g = {k: to_dev(x[k], "bf16") for k in ("dout", "dwte", "dwpe")}
    gi = torch.from_numpy(x["inp"]).to("cuda:0")
    n = mm.encbwd_plan_bytes(B, T, C, V, mm.BF16)
    plan = torch.empty(n, dtype=torch.uint8, device="cuda:0")
    assert mm.encbwd_prepare(plan, n, gi, B, T, C, V, mm.BF16) == mm.OK
    assert mm.encbwd_run_planned(g["dwte"], g["dwpe"], g["dout"], plan, B, T, C, V, mm.BF16) == mm.OK
    torch.cuda.synchronize()
    for k in ("dwte", "dwpe"):
        assert torch.equal(g[k], one[k]), k
    # stochastic rounding, repeatable per seed
    outs = []
    for _ in range(2):
        h = {k: to_dev(x[k], "bf16") for k in ("dout", "dwte", "dwpe")}
        assert mm.encbwd_run_sr(h["dwte"], h["dwpe"], h["dout"], gi, B, T, C, V, mm.BF16, 99) == mm.OK
        torch.cuda.synchronize()
        outs.append(h)
    for k in ("dwte", "dwpe"):
        assert torch.equal(outs[0][k], outs[1][k]), k
    check(x, outs[0], B, T, V, "bf16")

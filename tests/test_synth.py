"""The seeded input generator (shared by the oracle checks and the CUDA path)."""
import os
import subprocess
import sys

import numpy as np

import synth


def test_reproducible_and_streams_independent():
    a = synth.normal((1000,), "f32", 0, 1)
    b = synth.normal((1000,), "f32", 0, 1)
    c = synth.normal((1000,), "f32", 0, 2)
    d = synth.normal((1000,), "f32", 1, 1)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, c) and not np.array_equal(a, d)


def test_normal_moments():
    x = synth.normal((1 << 20,), "f64", 0, 3, 0.5, 2.0)
    n = x.size
    assert abs(x.mean() - 0.5) < 5 * 2.0 / np.sqrt(n)
    assert abs(x.std() - 2.0) < 0.01
    # Box-Muller pairs are independent: correlation of even/odd draws ~ 0
    r = np.corrcoef(x[0::2], x[1::2])[0, 1]
    assert abs(r) < 5 / np.sqrt(n / 2)
    u = synth.uniform(1 << 16, 0, 9)
    assert u.min() > 0 and u.max() <= 1 and abs(u.mean() - 0.5) < 0.01


def _rne_bf16_bits(f32):
    b = f32.view(np.uint32).astype(np.uint64)
    b = b + 0x7FFF + ((b >> 16) & 1)
    return (b >> 16).astype(np.uint16)


def test_bf16_is_rne_of_f32():
    f = synth.normal((50000,), "f32", 0, 5, 0.0, 3.0)
    h = synth.normal((50000,), "bf16", 0, 5, 0.0, 3.0)
    assert np.array_equal(h, _rne_bf16_bits(f))
    # exact decode of a few known patterns
    known = np.array([0x3F80, 0xBF80, 0x4049, 0x0000, 0x3C00], dtype=np.uint16)
    assert np.array_equal(synth.bf16_bits_to_f64(known), [1.0, -1.0, 3.140625, 0.0, 2.0 ** -7])


def test_lmhead_rows_have_one_spike():
    rows, cols, spike = 64, 1000, -1.0 / 64
    x = synth.lmhead_dout(rows, cols, "f64", 0, 3, 7, 1e-4, spike)
    for r in range(rows):
        hot = synth.lmhead_hot_index(r, cols, 0, 7)
        assert np.argmin(x[r]) == hot
        assert abs(x[r, hot] - spike) < 1e-3
    assert abs(np.delete(x, [synth.lmhead_hot_index(r, cols, 0, 7) + r * cols
                             for r in range(rows)]).std() - 1e-4) < 2e-6


def test_independent_of_thread_count():
    code = ("import sys; sys.path.insert(0, %r); import synth, hashlib;"
            "print(hashlib.sha1(synth.normal((300001,), 'bf16', 0, 3).tobytes()).hexdigest())"
            % os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    outs = set()
    for t in ("1", "3"):
        env = dict(os.environ, OMP_NUM_THREADS=t)
        outs.add(subprocess.check_output([sys.executable, "-c", code], env=env).strip())
    assert len(outs) == 1


def test_workload_recipes_match_the_configs():
    mlp = synth.WORKLOADS["mlp"]
    assert [(l.B, l.T, l.C, l.OC, l.dtype, l.bias) for l in mlp.layers] == [
        (8, 1024, 768, 3072, "bf16", True), (8, 1024, 3072, 768, "bf16", True)]
    assert mlp.flops() == 2 * (4 * 8192 * 768 * 3072) + 8192 * 3072 + 8192 * 768
    tiny = synth.WORKLOADS["tiny"].layers[0]
    x = synth.make_inputs(tiny)
    assert x["dinp"].dtype == np.float32 and np.std(x["dinp"]) > 0.005


def test_round_to_matches_the_generators_rounding():
    """synth.round_to (used for the LayerNorm inputs) rounds like the C
    generator: float64 -> f32 (RNE) -> bf16 (RNE)."""
    for dt in ("f32", "bf16"):
        a = synth.normal((4000,), dt, 7, 5, 0.3, 2.0)
        b = synth.round_to(synth.normal((4000,), "f64", 7, 5, 0.3, 2.0), dt)
        assert a.dtype == b.dtype and np.array_equal(a, b)


def test_layernorm_inputs_are_seeded_and_shaped():
    p = synth.LN_WORKLOADS["ln_tiny"]
    a, b = synth.make_ln_inputs(p), synth.make_ln_inputs(p)
    for k in a:
        assert np.array_equal(a[k], b[k])
    assert a["inp"].shape == (p.BT, p.C) and a["weight"].shape == (p.C,)
    rows = a["inp"].astype(np.float64)
    assert np.std(rows.mean(axis=1)) > 0.2 and np.std(np.log(rows.std(axis=1))) > 0.2

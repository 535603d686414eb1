"""Pins of the stochastic-rounding oracle to facts that do not come from it.

The oracle states the option from the definition (the two bf16 neighbours of
a value, the distance to the lower one as a fraction of the spacing) in double
arithmetic. The pins use instead: published splitmix64 outputs, the rule
restated on bit patterns (the draw added to the fp32 pattern, the low 16 bits
dropped: a carry means rounding up), and statistics every unbiased, per-element
independent rounding must show.
"""
from __future__ import annotations

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _bf16_value(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def pin_sr_published_generator(orc):
    """splitmix64 from seed 1234567 gives the published outputs."""
    with open(os.path.join(GOLDEN, "splitmix64_seed1234567.txt")) as f:
        vals = [int(x) for x in f.read().split() if x.strip() and not x.startswith("#") and x.isdigit()]
    seed, want = vals[0], vals[1:]
    assert [orc.splitmix64(seed, n) for n in range(len(want))] == want


def pin_sr_bit_rule(orc):
    """Every result equals the high half of (fp32 pattern + draw), the draw
    being 16 bits of the generator's output chosen by the element index."""
    rng = np.random.default_rng(31)
    x = np.concatenate([rng.normal(size=3000) * 10.0 ** rng.integers(-30, 30, size=3000),
                        rng.normal(size=200) * 1e-40])  # the last ones are fp32 subnormals
    x32 = x.astype(np.float32)
    seed, k, e0 = 77, 1, 5
    got = orc.sr_round(x, seed, k, e0)
    e = e0 + np.arange(x.size)
    words = np.array([orc.splitmix64(seed, (k << 58) | int(i >> 2)) for i in e], dtype=np.uint64)
    r = ((words >> (16 * (e & 3)).astype(np.uint64)) & np.uint64(0xFFFF)).astype(np.uint64)
    want = ((x32.view(np.uint32).astype(np.uint64) + r) >> np.uint64(16)).astype(np.uint16)
    assert np.array_equal(got, want)


def pin_sr_representable_kept(orc):
    """bf16 values (and zeros of both signs, infinities) are returned as they are."""
    rng = np.random.default_rng(32)
    bits = rng.integers(0, 1 << 16, size=4000).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]  # finite
    v = np.concatenate([_bf16_value(bits), [0.0, -0.0, np.inf, -np.inf]])
    for seed in (0, 1, 2**63 + 5):
        got = orc.sr_round(v, seed, 0)
        assert np.array_equal(got[:-4], bits)
        assert list(got[-4:]) == [0x0000, 0x8000, 0x7F80, 0xFF80]


def pin_sr_unbiased_and_neighbours(orc):
    """Over many elements one value rounds to its two neighbours only, up with
    probability equal to its position between them (binomial bound)."""
    n = 1 << 15
    for x, lo, hi in ((1.0 + 3 * 2.0 ** -9, 1.0, 1.0 + 2.0 ** -7),
                      (-(2.0 ** 20) * (1 + 2.0 ** -8), -(2.0 ** 20), -(2.0 ** 20) * (1 + 2.0 ** -7)),
                      (2.0 ** -130 + 2.0 ** -134, 2.0 ** -130, 2.0 ** -130 + 2.0 ** -133)):  # subnormal
        got = _bf16_value(orc.sr_round(np.full(n, x), 9, 0))
        assert set(np.unique(got)) <= {lo, hi}
        p = (abs(x) - abs(lo)) / (abs(hi) - abs(lo))
        frac = np.mean(got == hi)
        assert abs(frac - p) < 5 * np.sqrt(p * (1 - p) / n) + 1e-12, (x, frac, p)


def pin_sr_independent_draws(orc):
    """Neighbouring elements (four share one generator output) round
    independently: a value half way between neighbours rounds two consecutive
    elements the same way half of the time."""
    n = 1 << 15
    got = orc.sr_round(np.full(n, 1.0 + 2.0 ** -8), 3, 1)  # half way between 1 and 1 + 2^-7
    up = got == 0x3F81
    agree = np.mean(up[0::2] == up[1::2])
    assert abs(agree - 0.5) < 5 * np.sqrt(0.25 / (n // 2))
    assert abs(np.mean(up) - 0.5) < 5 * np.sqrt(0.25 / n)


def pin_sr_tensors_and_seeds_differ(orc):
    """The three output tensors and two seeds give different draws; one seed and
    tensor repeat themselves."""
    x = np.full(4096, 1.0 + 2.0 ** -8)
    a = orc.sr_round(x, 5, 0)
    assert np.array_equal(a, orc.sr_round(x, 5, 0))
    for other in (orc.sr_round(x, 5, 1), orc.sr_round(x, 5, 2), orc.sr_round(x, 6, 0)):
        assert np.mean(a != other) > 0.4


SR_PINS = [pin_sr_published_generator, pin_sr_bit_rule, pin_sr_representable_kept,
           pin_sr_unbiased_and_neighbours, pin_sr_independent_draws, pin_sr_tensors_and_seeds_differ]

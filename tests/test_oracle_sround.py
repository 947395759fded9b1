"""Pins for the FP16-checkpoint oracle: the generator, stochastic rounding and the replay model.

- Philox4x32-10 against its published known-answer vectors (tests/golden).
- Rounding toward zero against brute force over every binary16 value.
- Stochastic rounding: exact values stay, results are the two neighbours,
  the rounding is unbiased exactly (closed-form average over an even grid of
  words), saturation and signs.
- The FP16 replay oracle: between flushes its outputs equal the conventional
  recurrence started from the stored FP16 checkpoint; a fold stores a value
  within one binary16 ulp of the float32 rounding of the exact fold.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import sround

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _kat():
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            left, right = line.split("->")
            a = [int(x, 16) for x in left.split()]
            rows.append((a[:4], a[4:], [int(x, 16) for x in right.split()]))
    return rows


def test_philox_known_answers():
    rows = _kat()
    assert len(rows) == 3
    for ctr, key, out in rows:
        got = sround.philox4x32_10(np.array(ctr, np.uint32), np.array(key, np.uint32))
        assert [int(x) for x in got] == out


def test_philox_words_are_uniform_and_counter_distinct():
    w = sround.sr_words(1 << 16, 0, 3, 12345)
    assert w.dtype == np.uint32 and len(np.unique(w)) > (1 << 16) - 8
    hist = np.bincount((w >> 24).astype(np.int64), minlength=256)
    chi2 = float((((hist - 256.0) ** 2) / 256.0).sum())
    assert chi2 < 400  # 255 degrees of freedom
    assert not np.array_equal(w[:64], sround.sr_words(64, 0, 4, 12345))  # another epoch
    assert np.array_equal(w[64:128], sround.sr_words(64, 64, 3, 12345))  # counters are positions


def test_toward_zero_matches_brute_force():
    allf16 = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)  # finite, >= 0
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 5, 4000),
                        allf16[rng.integers(0, len(allf16), 500)]]).astype(np.float32)
    x = x[np.abs(x) < 65504]
    got = sround.f16_toward_zero(x)
    idx = np.searchsorted(allf16, np.abs(x.astype(np.float64)), side="right") - 1
    want = np.sign(x) * allf16[idx]
    assert np.array_equal(np.abs(got.astype(np.float64)), np.abs(want))


def test_stochastic_rounding_neighbours_and_exact_values():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(20000) * 10.0 ** rng.integers(-8, 4, 20000)).astype(np.float32)
    w = rng.integers(0, 2 ** 32, x.shape, dtype=np.uint64).astype(np.uint32)
    y = sround.stochastic_round_f16(x, w).astype(np.float64)
    lo = sround.f16_toward_zero(x).astype(np.float64)
    hi = np.abs(lo) + (np.nextafter(np.abs(lo).astype(np.float16), np.float16(np.inf)).astype(np.float64) - np.abs(lo))
    assert np.all((np.abs(y) == np.abs(lo)) | (np.abs(y) == hi))
    assert np.all(np.signbit(y) == np.signbit(x))
    exact = x.astype(np.float16).astype(np.float32)
    assert np.array_equal(sround.stochastic_round_f16(exact, w).astype(np.float32), exact)


def test_stochastic_rounding_is_unbiased_exactly():
    """Over the words r = k 2^19 (k = 0 .. 8191) the average is the input, exactly,
    for values in the binary16 normal range (13 dropped bits)."""
    rng = np.random.default_rng(2)
    x = (rng.uniform(1.0, 2.0, 64) * 2.0 ** rng.integers(-14, 15, 64)).astype(np.float32)
    x *= np.where(rng.random(64) < 0.5, -1, 1).astype(np.float32)
    words = (np.arange(8192, dtype=np.uint64) << np.uint64(19)).astype(np.uint32)
    for xi in x:
        y = sround.stochastic_round_f16(np.full(8192, xi, np.float32), words).astype(np.float64)
        assert y.mean() == float(xi)


def test_stochastic_rounding_special_values():
    w = np.array([0, 2 ** 31, 2 ** 32 - 1], dtype=np.uint32)
    for big in (65504.0, 70000.0, 1e30):
        assert np.all(sround.stochastic_round_f16(np.full(3, big, np.float32), w) == np.float16(65504))
        assert np.all(sround.stochastic_round_f16(np.full(3, -big, np.float32), w) == np.float16(-65504))
    assert np.all(np.isnan(sround.stochastic_round_f16(np.full(3, np.nan, np.float32), w)))
    z = sround.stochastic_round_f16(np.array([-0.0, 0.0, -0.0], np.float32), w)
    assert np.array_equal(np.signbit(z), [True, False, True]) and np.all(z == 0)
    tiny = np.float32(2.0 ** -26)  # a quarter of the smallest binary16 subnormal
    y = sround.stochastic_round_f16(np.full(3, tiny, np.float32), w).astype(np.float64)
    assert list(y) == [2.0 ** -24, 0.0, 0.0]  # rounds up only for r < 2^30


@pytest.mark.parametrize("mode", ["sr", "rn"])
def test_f16_replay_oracle_against_recurrence(mode):
    shape = synth.Shape(B=2, H=4, P=8, N=16, G=2, L=4, in_dtype="f32", seed=5)
    gen = synth.make_generator(shape.seed)
    S0 = synth.initial_state(shape, gen).to(torch.float16).to(torch.float64).numpy()
    orc = sround.ReplayOracleF16(S0, L=shape.L, R=shape.R, G=shape.G, seed=99, mode=mode)
    ck = orc.ckpt.copy()
    S_conv = ck.copy()  # conventional recurrence restarted from each stored checkpoint
    for t in range(3 * shape.L):
        a, v, k, q = (oracle.to_f64(x) for x in synth.decode_step_inputs(shape, gen))
        S_conv, o_conv = oracle.conventional_step(S_conv, a, v, k, q)
        o, flushed = orc.decode(a, v, k, q)
        assert np.allclose(o, o_conv, rtol=1e-12, atol=1e-14), f"step {t}"
        if flushed.any():
            assert flushed.all()
            x32 = S_conv.astype(np.float32).astype(np.float64)
            lo = sround.f16_toward_zero(x32).astype(np.float64)
            ulp = np.abs(np.nextafter(np.abs(lo).astype(np.float16), np.float16(np.inf)).astype(np.float64) - np.abs(lo))
            assert np.all(np.abs(orc.ckpt - x32) <= ulp)
            assert np.array_equal(orc.ckpt.astype(np.float16).astype(np.float64), orc.ckpt)
            S_conv = orc.ckpt.copy()
    assert list(orc.epoch) == [3, 3]

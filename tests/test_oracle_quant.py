"""Pins for the oracle's read-copy quantizers. These checks depend on no GPU.

The quantizers are checked against the format definitions (golden code
tables), an independent library conversion (torch's float8_e4m3fn cast, below
its saturation point), exhaustive round trips and tie cases, native binary32
arithmetic, and the stated per-element error bound. The read-copy branch of
ReplayOracle and the fully quantized comparator are pinned by hand-worked
examples in tests/golden/ (dyadic values, exact in E4M3), and planted slips in
copies of both (on the CPU) must fail those examples.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import quant
from tests.golden_io import read_codes, read_keyed


def test_golden_code_tables():
    for fmt, code, val in read_codes("ocp_fp8_fp4_codes.txt"):
        got = float((oracle.e4m3_value if fmt == "e4m3" else oracle.e2m1_value)(code))
        if np.isnan(val):
            assert np.isnan(got), (fmt, hex(code))
        else:
            assert got == val and np.signbit(got) == np.signbit(val), (fmt, hex(code), got, val)


def test_round_trip_every_code():
    c4 = np.array([c for c in range(256) if (c & 0x7F) != 0x7F])
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_value(c4)), c4.astype(np.uint8))
    c2 = np.arange(16)
    assert np.array_equal(oracle.e2m1_encode(oracle.e2m1_value(c2)), c2.astype(np.uint8))


def test_e4m3_matches_torch_cast_below_saturation():
    """torch's fp32 -> float8_e4m3fn cast (round to nearest even) is an independent routine.
    It does not saturate (it returns NaN from 464 up), so compare below that."""
    rng = np.random.default_rng(0)
    mags = oracle.e4m3_value(np.arange(127))
    mids = ((mags[1:] + mags[:-1]) / 2).astype(np.float32)
    xs = np.concatenate([
        rng.uniform(-463, 463, 400_000), rng.normal(0, 1e-2, 200_000), rng.normal(0, 1, 200_000),
        mids, -mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9)),
    ]).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(xs.astype(np.float64)), ref)


def test_saturation_and_signed_zero():
    assert list(oracle.e4m3_encode([448.0, 1e30, -1e30, 470.0, -0.0, -1e-30])) == [0x7E, 0x7E, 0xFE, 0x7E, 0x80, 0x80]
    assert list(oracle.e2m1_encode([6.0, 7.0, 1e9, -6.5, -0.0, -0.1])) == [0x7, 0x7, 0x7, 0xF, 0x8, 0x8]


def test_e2m1_ties_to_even():
    # midpoints between grid values: 0.25 (0|0.5), 0.75 (0.5|1), 1.25, 1.75, 2.5, 3.5, 5
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    # even codes win: 0.25->0 (0), 0.75->1.0 (2), 1.25->1.0 (2), 1.75->2 (4), 2.5->2 (4), 3.5->4 (6), 5->4 (6)
    assert list(oracle.e2m1_encode(mids)) == [0, 2, 2, 4, 4, 6, 6]
    eps = 1e-6
    assert list(oracle.e2m1_encode([0.25 + eps, 0.75 - eps, 5.0 + eps])) == [1, 1, 7]


def _f32_native_e4m3(X):
    """Same row recipe computed with native numpy float32 arithmetic."""
    X = X.astype(np.float32)
    a = np.abs(X).max(-1)
    with np.errstate(divide="ignore"):
        inv = np.where(a > quant.ZERO_ROW_AMAX, np.float32(448) / a, np.float32(0)).astype(np.float32)
        s = np.where(a > quant.ZERO_ROW_AMAX, a / np.float32(448), np.float32(0)).astype(np.float32)
    y = (X * inv[:, None]).astype(np.float32)
    return oracle.e4m3_encode(y), s


def test_row_recipe_matches_native_binary32_arithmetic():
    rng = np.random.default_rng(1)
    X = (rng.standard_t(3, size=(512, 128)) * np.exp(rng.uniform(-20, 5, size=(512, 1)))).astype(np.float32)
    X[0] = 0
    c, s = quant.quantize_rows_e4m3(X)
    c2, s2 = _f32_native_e4m3(X)
    assert np.array_equal(c, c2) and np.array_equal(s, s2)


def _adversarial_rows(rng, n=2048, N=128):
    X = rng.normal(size=(n, N)) * np.exp(rng.uniform(-30, 8, size=(n, 1)))
    X[:64, 5] *= 1e4  # one dominant element per row
    X[64:128, :16] *= 1e-6  # a nearly empty block
    X[128:160] = 0.0
    X[160:192, 16:] = 0.0  # one live block
    X[192:256] = rng.standard_t(1.5, size=(64, N))  # heavy tails
    return X.astype(np.float32)


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
def test_element_error_bound_holds_and_is_tight(fmt):
    rng = np.random.default_rng(2)
    X = _adversarial_rows(rng)
    if fmt == "e4m3":
        Xh = quant.dequantize_rows_e4m3(*quant.quantize_rows_e4m3(X))
    else:
        Xh = quant.dequantize_rows_e2m1(*quant.quantize_rows_e2m1(X))
    err = np.abs(Xh - X.astype(np.float64))
    bound = quant.element_error_bound(fmt, X)
    assert np.all(err <= bound)
    ratio = err[bound > 0] / bound[bound > 0]
    assert ratio.max() > 0.5  # the bound is not vacuous


def test_e2m1_block_layout():
    """Block scales follow 16-element blocks along the row; a zero block stays zero."""
    X = np.zeros((1, 64), np.float32)
    X[0, 16:32] = np.linspace(-1, 1, 16)
    X[0, 48:64] = 3.0
    codes, bcodes, s_r = quant.quantize_rows_e2m1(X)
    assert bcodes[0, 0] == 0 and bcodes[0, 2] == 0
    assert np.all(codes[0, :16] == 0) and np.all(codes[0, 32:48] == 0)
    assert np.all(codes[0, 48:] == 0x7)  # the block maximum maps to 6
    Xh = quant.dequantize_rows_e2m1(codes, bcodes, s_r)
    assert np.allclose(Xh[0, 48:], 3.0, rtol=2 ** -4)


def test_split_precision_error_does_not_grow_but_quantized_state_does():
    """The read copy's error stays bounded, while a quantized state accumulates error
    ([RU] §06, last paragraph; [AR] quantization section). Long-memory decays keep
    the effect visible in 600 steps."""
    rng = np.random.default_rng(3)
    B, H, P, N, G, L = 1, 2, 16, 32, 1, 16
    S0 = rng.normal(0, 0.1, size=(B, H, P, N))
    exact = oracle.ReplayOracle(S0, L=L, R=L, G=G)
    split = oracle.ReplayOracle(S0, L=L, R=L, G=G, read_fmt="e2m1")
    full = oracle.FullyQuantizedState(S0, "e2m1")
    e_split, e_full = [], []
    for t in range(600):
        a = np.exp(-np.logaddexp(0, rng.normal(-4, 1, size=(B, H))))
        v = rng.normal(size=(B, H, P)) / np.sqrt(N)
        k = rng.normal(size=(B, G, N)) / np.sqrt(N)
        q = rng.normal(size=(B, G, N)) / np.sqrt(N)
        o, _ = exact.decode(a, v, k, q)
        o_s, _ = split.decode(a, v, k, q)
        o_f = full.step(a, v, k, q)
        sc = np.abs(o).max()
        e_split.append(np.abs(o_s - o).max() / sc)
        e_full.append(np.abs(o_f - o).max() / sc)
    e_split, e_full = np.array(e_split), np.array(e_full)
    assert e_split[-100:].max() <= 2.0 * e_split[:100].max()
    assert np.median(e_full[-100:]) > 2.0 * np.median(e_split[-100:])


# ----------------------------------------------------------- hand-worked read-copy goldens
def _read_copy_golden_holds(cls) -> bool:
    """Three decode steps of tests/golden/hand_read_copy_e4m3.txt through a ReplayOracle
    class (L = 2): the copy at creation, the non-flush outputs read from the copy, the flush
    output from the exact state, and the copy refreshed from the folded state."""
    g = read_keyed("hand_read_copy_e4m3.txt")
    orc = cls(g["S0"].reshape(1, 1, 1, 2), L=2, R=2, G=1, read_fmt="e4m3")
    ok = np.array_equal(orc.copy.ravel(), g["copy0"])
    for i in (1, 2, 3):
        a = np.array([[g["alpha"][i - 1]]])
        o, _ = orc.decode(a, g[f"v{i}"].reshape(1, 1, 1), g[f"k{i}"].reshape(1, 1, 2), g[f"q{i}"].reshape(1, 1, 2))
        ok &= np.array_equal(o.ravel(), g[f"o{i}"]) and np.array_equal(orc.S.ravel(), g[f"S{i}"])
        if i == 2:
            ok &= np.array_equal(orc.copy.ravel(), g["copy2"])
    return bool(ok)


def _fully_quantized_golden_holds(cls) -> bool:
    """Two steps of tests/golden/hand_fully_quantized_e4m3.txt through a FullyQuantizedState class."""
    g = read_keyed("hand_fully_quantized_e4m3.txt")
    f = cls(g["S0"].reshape(1, 1, 2, 2), "e4m3")
    ok = np.array_equal(f.S.ravel(), g["S0"])
    for i in (1, 2):
        o = f.step(np.array([[g[f"alpha{i}"][0]]]), g[f"v{i}"].reshape(1, 1, 2), g[f"k{i}"].reshape(1, 1, 2),
                   g[f"q{i}"].reshape(1, 1, 2))
        ok &= np.array_equal(o.ravel(), g[f"o{i}"]) and np.array_equal(f.S.ravel(), g[f"Sq{i}"])
    return bool(ok)


def test_hand_worked_read_copy_codes():
    g = read_keyed("hand_read_copy_e4m3.txt")
    codes, scale = quant.quantize_rows_e4m3(np.array([g["S0"]], np.float32))
    assert list(codes.ravel()) == [int(x) for x in g["copy_codes0"]]
    assert float(scale[0]) == g["copy_scale0"][0]


def test_hand_worked_read_copy_replay():
    assert _read_copy_golden_holds(oracle.ReplayOracle)


def test_hand_worked_fully_quantized_steps():
    assert _fully_quantized_golden_holds(oracle.FullyQuantizedState)


# Planted mistakes in copies of the read-copy branch and of the quantized-state step (CPU only).
class _FlushReadsCopy(oracle.ReplayOracle):
    """Slip: the flush step's output also comes from the read copy."""

    def decode(self, alpha, v, k, q):
        copy_before = self.copy.copy()
        recs = [list(r) for r in self.records]
        o, flush = super().decode(alpha, v, k, q)
        for b in np.nonzero(flush)[0]:
            a_, v_, k_ = (np.stack(x) for x in zip(*(recs[b] + [(alpha[b], v[b], k[b])])))
            o[b] = oracle.replay_output(copy_before[b], a_, v_, k_, q[b])
        return o, flush


class _CopyNotRefreshed(oracle.ReplayOracle):
    """Slip: the flush folds the checkpoint but keeps the old read copy."""

    def _fold(self, mask, n_records):
        old = None if self.copy is None else self.copy.copy()
        idx = super()._fold(mask, n_records)
        if old is not None:
            self.copy = old
        return idx


class _CopyNotQuantized(oracle.ReplayOracle):
    """Slip: the copy is the exact state (no quantization)."""

    def _quantize(self, X):
        return np.array(X, np.float64)


class _NonFlushReadsExact(oracle.ReplayOracle):
    """Slip: non-flush outputs come from the exact state instead of the copy."""

    def decode(self, alpha, v, k, q):
        S_before = self.S.copy()
        o, flush = super().decode(alpha, v, k, q)
        _, o_exact = oracle.conventional_step(S_before, alpha, v, k, q)
        return o_exact, flush


class _OutputFromQuantized(oracle.FullyQuantizedState):
    """Slip: the output reads the re-quantized state instead of the fresh update."""

    def step(self, alpha, v, k, q):
        super().step(alpha, v, k, q)
        g = oracle.head_groups(self.S.shape[1], q.shape[1])
        return (self.S * q[:, g][:, :, None, :]).sum(-1)


class _StateKeptExact(oracle.FullyQuantizedState):
    """Slip: the updated state is stored without re-quantization."""

    def step(self, alpha, v, k, q):
        S_pre, o = oracle.conventional_step(self.S, alpha, v, k, q)
        self.S = S_pre
        return o


@pytest.mark.parametrize("mutant", [_FlushReadsCopy, _CopyNotRefreshed, _CopyNotQuantized, _NonFlushReadsExact],
                         ids=lambda m: m.__name__)
def test_read_copy_golden_catches_planted_mistakes(mutant):
    assert not _read_copy_golden_holds(mutant)


@pytest.mark.parametrize("mutant", [_OutputFromQuantized, _StateKeptExact], ids=lambda m: m.__name__)
def test_fully_quantized_golden_catches_planted_mistakes(mutant):
    assert not _fully_quantized_golden_holds(mutant)

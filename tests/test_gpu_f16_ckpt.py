"""GPU parity for the FP16 recurrent checkpoint (stochastic rounding and round to nearest).

Bit-exact: the device's binary32 -> binary16 store rounding (rssm_round_f16,
the same device function as the fold's store) against the oracle's, word for
word from the same Philox4x32-10 counters, for both modes.

Within a derived bound: decode, verify, commit and flush against the FP16
replay oracle. The device folds in FP32 and the oracle in float64, so a
stochastic (or nearest) decision can differ where the two values fall on
different sides of the word's threshold (or a midpoint); each stored element
may then differ, and the difference is carried into later folds scaled by the
window's decay. The test tracks, per element, the bound
    d_new = g d_old + 2 ulp16(stored magnitude)      (at every flush, d = 0 at the start)
where g is the window's decay product from the inputs (each side rounds within
one ulp of its own value). Outputs must stay within
    g_h sum_n d_n |q_n| + 1e-4 max|o*|      (normwise slack per head)
and at most 1% of stored elements may differ. Pointers and epochs are bit-exact.
"""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from oracle import sround
from hybrid_model_ssm_gb300 import ReplaySSM, round_f16
from tests.gpu_helpers import dev, f64, layer_shape, require_gpu

pytestmark = pytest.mark.gpu



def oracle_groups(shape):
    import oracle
    return oracle.head_groups(shape.H, shape.G)


def _values(n, rng):
    x = rng.standard_normal(n) * 10.0 ** rng.integers(-9, 5, n)
    x[:12] = [0.0, -0.0, 65504.0, -65504.0, 70000.0, -1e30, 2.0 ** -24, 2.0 ** -26, -3.0 * 2.0 ** -26,
              6.1e-5, 1.0, np.nan]
    return x.astype(np.float32)


@pytest.mark.parametrize("stochastic", [True, False])
def test_store_rounding_is_bit_exact(stochastic):
    require_gpu()
    rng = np.random.default_rng(60)
    x = _values(20000, rng)
    base, epoch, seed = 4 * 12345, 7, 0x1234_5678_9ABC_DEF0
    y = round_f16(torch.from_numpy(x).cuda(), base=base, epoch=epoch, seed=seed, stochastic=stochastic).cpu().numpy()
    if stochastic:
        ref = sround.stochastic_round_f16(x, sround.sr_words(len(x), base, epoch, seed))
    else:
        ref = sround.nearest_f16(x)
    nan = np.isnan(x)
    assert np.all(np.isnan(y[nan]))
    bad = np.nonzero(y[~nan].view(np.uint16) != ref[~nan].view(np.uint16))[0]
    assert len(bad) == 0, f"{len(bad)} values differ, first x={x[~nan][bad[:3]]}"


def _bit_patterns(rng):
    """Random binary32 bit patterns over every exponent, and every finite binary16
    value with its two binary32 neighbours, both signs."""
    pat = rng.integers(0, 2 ** 32, 1 << 18, dtype=np.uint64).astype(np.uint32).view(np.float32)
    h = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float32)
    grid = np.concatenate([h, np.nextafter(h, np.float32(np.inf)), np.nextafter(h, np.float32(0))])
    return np.concatenate([pat, grid, -grid]).astype(np.float32)


@pytest.mark.parametrize("stochastic", [True, False])
def test_store_rounding_is_bit_exact_over_bit_patterns(stochastic):
    require_gpu()
    x = _bit_patterns(np.random.default_rng(62))
    base, epoch, seed = 4 * 777, 3, 0x0F1E_2D3C_4B5A_6978
    y = round_f16(torch.from_numpy(x).cuda(), base=base, epoch=epoch, seed=seed, stochastic=stochastic).cpu().numpy()
    with np.errstate(invalid="ignore", over="ignore"):
        if stochastic:
            ref = sround.stochastic_round_f16(x, sround.sr_words(len(x), base, epoch, seed))
        else:
            ref = sround.nearest_f16(x)
    nan = np.isnan(x)
    assert np.all(np.isnan(y[nan]))
    if stochastic:  # the stochastic store writes one NaN code
        assert np.all(y[nan].view(np.uint16) == 0x7E00)
    bad = np.nonzero(y[~nan].view(np.uint16) != ref[~nan].view(np.uint16))[0]
    assert len(bad) == 0, f"{len(bad)} values differ, first x={x[~nan][bad[:3]]}"


def _f16_model(shape, mode, seed):
    gen = synth.make_generator(shape.seed)
    S0 = synth.initial_state(shape, gen).to(torch.float16)
    ls = dataclasses.replace(layer_shape(shape), ckpt="f16_" + mode, seed=seed)
    model = ReplaySSM(ls, S0.cuda())
    orc = sround.ReplayOracleF16(S0.double().numpy(), L=shape.L, R=shape.R, G=shape.G, seed=seed, mode=mode)
    return model, orc, gen


def _ulp16(mag):
    lo = sround.f16_toward_zero(np.asarray(mag, np.float32)).astype(np.float64)
    return np.nextafter(lo.astype(np.float16), np.float16(np.inf)).astype(np.float64) - lo


def _check_ckpt(model, orc, bound, where):
    ck = model.ckpt.float().cpu().numpy().astype(np.float64)
    diff = np.abs(ck - orc.ckpt)
    assert np.all(diff <= bound * (1 + 1e-9)), f"{where}: checkpoint differs beyond the propagated bound"
    frac = float(np.mean(diff > 0))
    assert frac < 1e-2, f"{where}: {frac:.2%} of checkpoint elements differ"


def _out_bound(d, gam, q, g, o_ref):
    """g_h sum_n d[b,h,p,n] |q[b,g(h),n]| + 1e-4 max|o*| per (b,h)."""
    qa = np.abs(q)[:, g, :]  # [B,H,N]
    return gam[:, :, None] * np.einsum("bhpn,bhn->bhp", d, qa) + 1e-4 * np.abs(o_ref).max(-1, keepdims=True)


@pytest.mark.parametrize("mode", ["sr", "rn"])
@pytest.mark.parametrize("N", [64, 128])
def test_f16_decode_matches_oracle(mode, N):
    require_gpu()
    shape = synth.Shape(B=3, H=8, P=32, N=N, G=2, L=6, seed=61)
    model, orc, gen = _f16_model(shape, mode, seed=2024)
    d = np.zeros((shape.B, shape.H, shape.P, shape.N))  # bound on |checkpoint - oracle checkpoint|
    gam = np.ones((shape.B, shape.H))  # decays since the last flush, this step's included
    g = oracle_groups(shape)
    for t in range(3 * shape.L + 2):
        a, v, k, q = synth.decode_step_inputs(shape, gen, -2.0)
        o = model.decode_step(dev(a), dev(v), dev(k), dev(q)).cpu().numpy().astype(np.float64)
        o_ref, flushed = orc.decode(f64(a), f64(v), f64(k), f64(q))
        gam = gam * f64(a)
        bnd = _out_bound(d, gam, f64(q), g, o_ref)
        assert np.all(np.abs(o - o_ref) <= bnd), f"step {t}: output beyond the bound"
        if flushed.any():
            d = gam[:, :, None, None] * d + 2 * _ulp16(np.abs(orc.ckpt))
            _check_ckpt(model, orc, d, f"step {t}")
            gam = np.ones_like(gam)
    start, count, err = model.read_pointers()
    assert err == 0
    assert np.array_equal(start.numpy(), orc.start) and np.array_equal(count.numpy(), orc.count)
    pb = (shape.B * 4 + 255) // 256 * 256  # pointer block: start, count, ticket, error word (256 B), epoch
    epoch = model.ptrs[3 * pb + 256: 3 * pb + 256 + 4 * shape.B].view(torch.int32)
    assert epoch.cpu().tolist() == orc.epoch.tolist() == [3] * shape.B


def test_f16_verify_commit_flush_match_oracle():
    require_gpu()
    shape = synth.Shape(B=4, H=8, P=32, N=128, G=2, L=8, T_max=4, seed=62)
    model, orc, gen = _f16_model(shape, "sr", seed=77)
    d = np.zeros((shape.B, shape.H, shape.P, shape.N))
    g = oracle_groups(shape)
    ones = np.ones((shape.B, shape.H))
    for r in range(12):
        T = 1 + r % shape.T_max
        a, v, k, q = synth.verify_round_inputs(shape, T, gen)
        O = model.verify(dev(a), dev(v), dev(k), dev(q)).cpu().numpy().astype(np.float64)
        O_ref = orc.verify(f64(a), f64(v), f64(k), f64(q))
        for t in range(T):  # decays are below 1, so g = 1 bounds every query
            bnd = _out_bound(d, ones, f64(q)[:, t], g, O_ref[:, t])
            assert np.all(np.abs(O[:, t] - O_ref[:, t]) <= bnd), f"round {r} query {t}: beyond the bound"
        acc = synth.accepted_lengths(shape.B, T, gen)
        model.commit(dev(acc))
        orc.commit(acc.numpy())
        model.flush(shape.L)
        fl = orc.flush(shape.L)
        start, count, err = model.read_pointers()
        assert err == 0
        assert np.array_equal(start.numpy(), orc.start) and np.array_equal(count.numpy(), orc.count), f"round {r}"
        if fl.any():
            d = np.where(fl[:, None, None, None], d + 2 * _ulp16(np.abs(orc.ckpt)), d)
            _check_ckpt(model, orc, d, f"round {r}")

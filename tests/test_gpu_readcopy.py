"""GPU parity for the low-precision read copy (E4M3 rows, E2M1 with 16-element blocks).

Bit-exact: on identical fp32 inputs the device quantizer must produce the
oracle quantizer's codes and scales byte for byte. This holds for the copy
built at creation from the initial checkpoint, and for every copy refreshed
at a flush (quantizing the device's own new checkpoint).
Parity: non-flush outputs read the dequantized copy. Since the device copy is
bit-exact, the oracle's output-only form evaluated on that copy (its
dequantized codes and scales) and the buffered records gives the exact
expected value, and the device output must match it within the FP32 path's
relative tolerance (1e-4 per (sequence, head)).
Bounded: the same outputs against the exact float64 output (the unquantized
recurrence) must stay within the stated per-format bound,
    |o - o*|_p <= 1.05 * g_{1:h} * sum_n bound(S_ckpt[p, n]) |q_n| + 1e-5 * max|o*|,
where bound() is the per-element bound of the format (oracle.quant) applied
to the fp32 checkpoint.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import quant
from hybrid_model_ssm_gb300 import ReplaySSM, read_copy_layout
from tests.gpu_helpers import REL_TOL, dev, f64, layer_shape, require_gpu, slice_rel_err

pytestmark = pytest.mark.gpu

S = synth.Shape
FMTS = ["e4m3", "e2m1"]


def _special_state(shape, gen):
    S0 = synth.initial_state(shape, gen)
    S0[0, 0, 0] = 0.0  # zero row
    S0[0, 0, 1] = 1e-35  # below the zero-row threshold
    S0[0, 0, 2, 5] = 1e30  # one huge element
    S0[0, 0, 3] = -0.0  # negative zeros
    S0[0, 0, 4] = torch.linspace(-1e-40, 1e-40, shape.N)  # subnormals
    S0[0, 1, 0, :16] *= 1e-7  # a nearly empty block
    S0[0, 1, 1, :] = torch.tensor([448.0 * (1 + i / 64) for i in range(shape.N)])  # saturation region
    return S0


def _split_copy(copy: torch.Tensor, shape, fmt):
    """Per-(b,h) views of the copy bytes: codes, block codes, row scales (numpy)."""
    ls = layer_shape(shape, fmt)
    stride, bsc, rsc = read_copy_layout(ls)
    buf = copy.cpu().numpy().reshape(shape.B, shape.H, stride)
    P, N = shape.P, shape.N
    if fmt == "e4m3":
        codes = buf[:, :, : P * N].reshape(shape.B, shape.H, P, N)
        bcodes = None
    else:
        packed = buf[:, :, : P * N // 2].reshape(shape.B, shape.H, P, N // 2)
        codes = np.empty((shape.B, shape.H, P, N), np.uint8)
        codes[..., 0::2] = packed & 0xF
        codes[..., 1::2] = packed >> 4
        bcodes = buf[:, :, bsc: bsc + P * N // 16].reshape(shape.B, shape.H, P, N // 16)
    rscale = buf[:, :, rsc: rsc + 4 * P].copy().view(np.float32).reshape(shape.B, shape.H, P)
    return codes, bcodes, rscale


def _dequantized_copy(copy, shape, fmt) -> np.ndarray:
    """The device read copy as the values a non-flush step reads, [B,H,P,N] float64 (oracle decoder)."""
    codes, bcodes, rscale = _split_copy(copy, shape, fmt)
    if fmt == "e4m3":
        return quant.dequantize_rows_e4m3(codes, rscale)
    return quant.dequantize_rows_e2m1(codes, bcodes, rscale)


def _oracle_codes(X32: np.ndarray, fmt):
    if fmt == "e4m3":
        c, s = quant.quantize_rows_e4m3(X32)
        return c, None, s
    return quant.quantize_rows_e2m1(X32)


def _assert_copy_matches(copy, X32, shape, fmt, where):
    codes, bcodes, rscale = _split_copy(copy, shape, fmt)
    c_ref, b_ref, s_ref = _oracle_codes(X32, fmt)
    bad = np.argwhere(codes != c_ref)
    assert len(bad) == 0, f"{where}: {len(bad)} codes differ, first at {bad[:3].tolist()}"
    if fmt == "e2m1":
        assert np.array_equal(bcodes, b_ref), f"{where}: block scales differ"
    assert np.array_equal(rscale.view(np.uint32), s_ref.view(np.uint32)), f"{where}: row scales differ"


@pytest.mark.parametrize("fmt", FMTS)
def test_copy_at_creation_is_bit_exact(fmt):
    require_gpu()
    shape = S(B=3, H=8, P=64, N=128, G=2, L=16, seed=50)
    gen = synth.make_generator(shape.seed)
    S0 = _special_state(shape, gen)
    model = ReplaySSM(layer_shape(shape, fmt), dev(S0))
    torch.cuda.synchronize()
    _assert_copy_matches(model.copy, S0.numpy(), shape, fmt, "creation")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("N", [64, 128])
def test_decode_with_read_copy(fmt, N):
    """Non-flush outputs equal the oracle's read-copy form on the device copy (1e-4) and stay
    within the per-format bound of the exact output; flush outputs exact; each refreshed
    copy bit-exact against the oracle quantizer of the device's new checkpoint."""
    require_gpu()
    shape = S(B=3, H=8, P=32, N=N, G=2, L=8, seed=51)
    gen = synth.make_generator(shape.seed)
    S0 = synth.initial_state(shape, gen)
    orc = oracle.ReplayOracle(f64(S0), L=shape.L, R=shape.R, G=shape.G)
    model = ReplaySSM(layer_shape(shape, fmt), dev(S0))
    ck32 = S0.numpy().astype(np.float64)  # fp32 checkpoint the copy was made from
    worst = 0.0
    for t in range(3 * shape.L + 3):
        recs_before = [list(r) for r in orc.records]
        torch.cuda.synchronize()
        copy_vals = _dequantized_copy(model.copy, shape, fmt)  # what this step's non-flush heads read
        a, v, k, q = synth.decode_step_inputs(shape, gen)
        o = model.decode_step(dev(a), dev(v), dev(k), dev(q)).cpu().numpy().astype(np.float64)
        o_ref, flushed = orc.decode(f64(a), f64(v), f64(k), f64(q))
        g = oracle.head_groups(shape.H, shape.G)
        for b in range(shape.B):
            if flushed[b]:
                assert slice_rel_err(o[b], o_ref[b], 1) <= REL_TOL
                continue
            alphas = np.stack([r[0] for r in recs_before[b]] + [f64(a)[b]])  # [h, H]
            vs = np.stack([r[1] for r in recs_before[b]] + [f64(v)[b]])
            ks = np.stack([r[2] for r in recs_before[b]] + [f64(k)[b]])
            o_copy = oracle.replay_output(copy_vals[b], alphas, vs, ks, f64(q)[b])
            rel = slice_rel_err(o[b], o_copy, 1)
            assert rel <= REL_TOL, f"step {t} seq {b}: {rel:.3g} against the oracle's read-copy output"
            gam = np.prod(alphas, axis=0)  # [H]
            qb = f64(q)[b][g]  # [H, N]
            eb = quant.element_error_bound(fmt, ck32[b].astype(np.float32))  # [H, P, N]
            bound = gam[:, None] * (eb * np.abs(qb)[:, None, :]).sum(-1)
            err = np.abs(o[b] - o_ref[b])
            slack = 1e-5 * np.abs(o_ref[b]).max(axis=-1, keepdims=True)
            assert np.all(err <= 1.05 * bound + slack), f"step {t} seq {b}: error above the {fmt} bound"
            worst = max(worst, float((err / (bound + slack)).max()))
        if flushed.any():
            ck_dev = model.ckpt.cpu().numpy()
            for b in np.nonzero(flushed)[0]:
                assert slice_rel_err(ck_dev[b], orc.ckpt[b], 2) <= REL_TOL
                ck32[b] = ck_dev[b]
            torch.cuda.synchronize()
            # every flushed head's copy equals the oracle quantizer of the device checkpoint
            codes, bcodes, rscale = _split_copy(model.copy, shape, fmt)
            c_ref, b_ref, s_ref = _oracle_codes(ck_dev, fmt)
            for b in np.nonzero(flushed)[0]:
                assert np.array_equal(codes[b], c_ref[b]), f"step {t}: refreshed codes differ"
                assert np.array_equal(rscale[b].view(np.uint32), s_ref[b].view(np.uint32))
                if fmt == "e2m1":
                    assert np.array_equal(bcodes[b], b_ref[b])
    assert worst > 0.0


def _unit_scale_rows(fmt, N):
    """Rows whose scales come out exactly 1, so that each element's code is the
    format's own conversion of the element itself. They hold every finite code
    value, every midpoint between neighbouring codes (a tie, resolved to the even
    code) and the binary32 neighbours of each midpoint, with both signs.

    E4M3: a row whose max |x| is 448 gets inv = 448/448 = 1.
    E2M1: a row whose max |x| is 2688 gets s_r = 1 and d6 = 6; a block of 16 whose
    max |x| is 6 then gets the block code of 1.0, so d = r = 1.
    """
    f32 = np.float32
    if fmt == "e4m3":
        vals = quant.e4m3_value(np.arange(0x7F)).astype(f32)  # 0 .. 448, every finite non-negative code
        top = f32(448.0)
    else:
        vals = np.array(sorted(set(quant.e2m1_value(np.arange(8)).tolist())), f32)  # 0, 0.5, .., 6
        top = f32(6.0)
    mids = ((vals[:-1].astype(np.float64) + vals[1:]) / 2).astype(f32)
    tests = np.concatenate([vals, mids, np.nextafter(mids, f32(np.inf)), np.nextafter(mids, f32(0))])
    tests = np.concatenate([tests, -tests])
    if fmt == "e4m3":
        per_row = N - 1
        rows = []
        for i in range(0, len(tests), per_row):
            r = np.zeros(N, f32)
            r[0] = top
            chunk = tests[i:i + per_row]
            r[1:1 + len(chunk)] = chunk
            rows.append(r)
        return np.stack(rows)
    per_block, nblk = 15, N // 16
    blocks = [tests[i:i + per_block] for i in range(0, len(tests), per_block)]
    nrows = -(-len(blocks) // (nblk - 1))
    rows = np.zeros((nrows, N), f32)
    for i in range(nrows * (nblk - 1)):  # every block after block 0 filled (the values repeat to fill the last row)
        r, bi = divmod(i, nblk - 1)
        blk = blocks[i % len(blocks)]
        base = 16 * (bi + 1)
        rows[r, base] = top
        rows[r, base + 1: base + 1 + len(blk)] = blk
    rows[:, 0] = f32(2688.0)  # block 0 pins the row scale
    return rows


def _saturation_row(N):
    """E4M3 row with a scale other than 1 whose largest elements scale to the top code or just below it."""
    r = np.zeros(N, np.float32)
    r[:6] = [1000.0, 999.0, -1000.0, 1000.0 * 448.5 / 448, 1000.0 * 463.9 / 448, 1000.0 * 464.0 / 448]
    return r


@pytest.mark.parametrize("fmt", FMTS)
def test_copy_codes_of_every_code_value_and_midpoint(fmt):
    """The device quantizer (the CUDA conversions) against the oracle encoder, bit for
    bit, on every code value, every tie between neighbouring codes and their binary32
    neighbours (unit scales), plus (E4M3) a row whose largest elements scale to the top code."""
    require_gpu()
    shape = S(B=1, H=2, P=64, N=128, G=1, L=4, seed=52)
    gen = synth.make_generator(shape.seed)
    S0 = synth.initial_state(shape, gen)
    rows = _unit_scale_rows(fmt, shape.N)
    assert len(rows) < shape.P
    S0[0, 0, : len(rows)] = torch.from_numpy(rows)
    if fmt == "e4m3":
        S0[0, 0, len(rows)] = torch.from_numpy(_saturation_row(shape.N))
    c_ref, b_ref, s_ref = _oracle_codes(S0.numpy(), fmt)
    # the crafted rows really have unit scales: their codes are the conversion of x itself
    assert np.all(s_ref[0, 0, : len(rows)] == 1.0)
    if fmt == "e2m1":
        assert np.all(quant.e4m3_value(b_ref[0, 0, : len(rows), 1:]) == 1.0)
    model = ReplaySSM(layer_shape(shape, fmt), dev(S0))
    torch.cuda.synchronize()
    _assert_copy_matches(model.copy, S0.numpy(), shape, fmt, "every code and midpoint")

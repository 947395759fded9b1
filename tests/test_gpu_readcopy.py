"""GPU parity for the low-precision read copy (E4M3 rows, E2M1 with 16-element blocks).

Bit-exact: on identical fp32 inputs the device quantizer must produce the
oracle quantizer's codes and scales byte for byte. This holds for the copy
built at creation from the initial checkpoint, and for every copy refreshed
at a flush (quantizing the device's own new checkpoint).
Bounded: non-flush outputs read the dequantized copy. Their error against
the exact float64 output must stay within the stated per-format bound,
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
    """Non-flush outputs within the per-format bound; flush outputs exact;
    each refreshed copy bit-exact against the oracle quantizer of the device's new checkpoint."""
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
        a, v, k, q = synth.decode_step_inputs(shape, gen)
        o = model.decode_step(dev(a), dev(v), dev(k), dev(q)).cpu().numpy().astype(np.float64)
        o_ref, flushed = orc.decode(f64(a), f64(v), f64(k), f64(q))
        g = oracle.head_groups(shape.H, shape.G)
        for b in range(shape.B):
            if flushed[b]:
                assert slice_rel_err(o[b], o_ref[b], 1) <= REL_TOL
                continue
            alphas = np.stack([r[0] for r in recs_before[b]] + [f64(a)[b]])  # [h, H]
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

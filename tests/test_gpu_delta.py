"""GPU parity: replay decoding of gated delta-rule (Gated DeltaNet) layers.

Every step's output is compared with the float64 delta-rule oracle on the same
seeded inputs (normwise relative error per (sequence, head) within 1e-4). The
pointers, the flush events and the appended ring records (alpha, k) must
match bit for bit, and each appended pseudo-value w = beta (v - alpha y) must
match the oracle's (same tolerance); the checkpoint is compared at every flush and must stay
bit-identical between flushes. The conventional delta-rule kernel is checked
against the definition step by step, and the entry points that do not apply
to delta-rule layers must refuse them.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from hybrid_model_ssm_gb300 import LayerShape, ReplaySSM, RssmError, conventional_step
from hybrid_model_ssm_gb300.rssm import RSSM_EINVAL, lib
from tests.gpu_helpers import REL_TOL, dev, f64, require_gpu, slice_rel_err

pytestmark = pytest.mark.gpu

S = synth.Shape
CASES = [
    ("b5_h6_g3_p24_n64_l5_bf16", S(B=5, H=6, P=24, N=64, G=3, L=5, seed=31), 24),
    ("b3_h16_g2_p64_n128_l16_bf16", S(B=3, H=16, P=64, N=128, G=2, L=16, seed=32), 40),
    ("two_row_passes_b2_h4_p128_n128_l16_f32", S(B=2, H=4, P=128, N=128, G=1, L=16, in_dtype="f32", seed=33), 34),
    ("every_step_flushes_l1_n64_f32", S(B=2, H=2, P=16, N=64, G=1, L=1, in_dtype="f32", seed=34), 6),
    ("window_32_b2_h2_p16_n64", S(B=2, H=2, P=16, N=64, G=1, L=32, seed=35), 70),
    ("ragged_rows_p8_n64_b3_h4_g2", S(B=3, H=4, P=8, N=64, G=2, L=3, seed=36), 20),
    ("largest_f32_p128_n128_l28", S(B=2, H=2, P=128, N=128, G=1, L=28, in_dtype="f32", seed=39), 58),
    ("largest_ring_p128_n128_l32_bf16", S(B=2, H=2, P=128, N=128, G=1, L=32, seed=40), 66),
]


def delta_shape(s: synth.Shape) -> LayerShape:
    return LayerShape(B=s.B, H=s.H, P=s.P, N=s.N, G=s.G, L=s.L, T_max=1, in_dtype=s.in_dtype, recurrence="delta")


def _check_step(model, orc, shape, t, o_gpu, o_ref, flushed, ckpt_prev, inputs):
    e = slice_rel_err(o_gpu, o_ref, 1)
    assert e <= REL_TOL, f"step {t}: output rel err {e:.3g}"
    start, count, err = model.read_pointers()
    assert err == 0
    assert np.array_equal(start.numpy(), orc.start) and np.array_equal(count.numpy(), orc.count), f"step {t}"
    ck = model.ckpt.cpu()
    for b in range(shape.B):
        if flushed[b]:
            es = slice_rel_err(ck[b], orc.ckpt[b], 2)
            assert es <= REL_TOL, f"step {t} seq {b}: checkpoint rel err {es:.3g}"
        else:
            assert torch.equal(ck[b], ckpt_prev[b]), f"step {t}: non-flush step wrote the checkpoint"
    if inputs is None:
        return ck
    a, k, w_ref = inputs
    ra, _, rk = model.ring_views()
    rw = model.ring_pseudo_values().cpu().numpy()
    for b in range(shape.B):
        if flushed[b]:
            continue
        slot = (int(start[b]) + int(count[b]) - 1) % shape.R
        assert torch.equal(ra[b, :, slot].cpu(), a[b])
        assert torch.equal(rk[b, :, slot].cpu(), k[b])
        # the appended pseudo-value against the oracle's, relative to the value scale
        err = np.abs(rw[b, :, slot] - w_ref[b]).max() / max(np.abs(w_ref[b]).max(), 1e-30)
        assert err <= REL_TOL, f"step {t} seq {b}: pseudo-value rel err {err:.3g}"
    return ck


def run_delta_parity(shape: synth.Shape, steps: int, mu: float = 0.0, flush_at=None):
    require_gpu()
    gen = synth.make_generator(shape.seed)
    S0 = synth.initial_state(shape, gen)
    orc = oracle.DeltaReplayOracle(f64(S0), L=shape.L, R=shape.R, G=shape.G)
    model = ReplaySSM(delta_shape(shape), dev(S0))
    ckpt_prev = model.ckpt.cpu()
    for t in range(steps):
        if flush_at is not None and t in flush_at:
            mc = flush_at[t]
            model.flush(mc)
            mask = orc.flush(mc)
            ckpt_prev = _check_step(model, orc, shape, f"flush@{t}", np.zeros(1), np.zeros(1), mask, ckpt_prev, None)
        a, beta, v, k, q = synth.delta_step_inputs(shape, gen, mu)
        o_gpu = model.decode_step(dev(a), dev(v), dev(k), dev(q), beta=dev(beta)).cpu()
        w_ref = oracle.delta_pseudo_value(orc.S, f64(a), f64(beta), f64(v), f64(k))
        o_ref, flushed = orc.decode(f64(a), f64(beta), f64(v), f64(k), f64(q))
        ckpt_prev = _check_step(model, orc, shape, t, o_gpu, o_ref, flushed, ckpt_prev, (a, k, w_ref))


@pytest.mark.parametrize("name,shape,steps", CASES, ids=[c[0] for c in CASES])
def test_delta_decode_matches_oracle(name, shape, steps):
    run_delta_parity(shape, steps)


def test_delta_decode_long_memory_decays():
    """Decays near 1 (u ~ N(-4, 1)): every buffered record keeps its weight."""
    run_delta_parity(S(B=2, H=8, P=64, N=128, G=2, L=16, seed=37), 48, mu=-4.0)


def test_delta_standalone_flush_staggers_the_sequences():
    """A flush between steps folds the sequences with count >= min_count; they
    then flush on their own schedule, out of step with the others."""
    run_delta_parity(S(B=6, H=4, P=32, N=128, G=2, L=8, seed=38), 30, flush_at={3: 2, 11: 5, 20: 1})


def test_delta_pure_decay_and_full_write():
    """beta = 0 leaves S_t = (prod alpha) S_0; beta = 1 with orthonormal keys
    (the first N/2 unit vectors) stores each value exactly: S_t k_t = v_t."""
    require_gpu()
    shape = S(B=2, H=2, P=16, N=64, G=1, L=8, in_dtype="f32", seed=39)
    gen = synth.make_generator(shape.seed)
    S0 = synth.initial_state(shape, gen)
    orc = oracle.DeltaReplayOracle(f64(S0), L=shape.L, R=shape.R, G=shape.G)
    model = ReplaySSM(delta_shape(shape), dev(S0))
    eye = torch.eye(64)
    for t in range(12):
        a, beta, v, k, q = synth.delta_step_inputs(shape, gen)
        if t < 6:
            beta = torch.zeros_like(beta)
        else:
            beta = torch.ones_like(beta)
            a = torch.ones_like(a)
            k = eye[t].expand(2, 1, 64).contiguous()
            q = eye[t].expand(2, 1, 64).contiguous()
        o = model.decode_step(dev(a), dev(v), dev(k), dev(q), beta=dev(beta)).cpu()
        o_ref, _ = orc.decode(f64(a), f64(beta), f64(v), f64(k), f64(q))
        assert slice_rel_err(o, o_ref, 1) <= REL_TOL, f"step {t}"
        if t >= 6:  # the query equals the key just written: the output is that value
            assert torch.allclose(o, v, rtol=1e-5, atol=1e-6), f"step {t}"


@pytest.mark.parametrize("shape", [
    S(B=3, H=8, P=64, N=128, G=2, L=16, seed=40),
    S(B=2, H=4, P=40, N=64, G=4, L=16, in_dtype="f32", seed=41),
], ids=["b3_h8_p64_n128_bf16", "p40_n64_f32"])
def test_conventional_delta_kernel_matches_definition(shape):
    require_gpu()
    gen = synth.make_generator(shape.seed)
    S0 = synth.initial_state(shape, gen)
    state = dev(S0)
    S_ref = f64(S0)
    ls = delta_shape(shape)
    for t in range(12):
        a, beta, v, k, q = synth.delta_step_inputs(shape, gen)
        o = conventional_step(ls, state, dev(a), dev(v), dev(k), dev(q), beta=dev(beta)).cpu()
        S_ref, o_ref = oracle.delta_step(S_ref, f64(a), f64(beta), f64(v), f64(k), f64(q))
        assert slice_rel_err(o, o_ref, 1) <= REL_TOL, f"step {t}"
        assert slice_rel_err(state.cpu(), S_ref, 2) <= REL_TOL, f"step {t}"


def test_entry_points_that_do_not_apply_refuse_delta_layers():
    require_gpu()
    shape = S(B=2, H=2, P=16, N=64, G=1, L=4, seed=42)
    gen = synth.make_generator(shape.seed)
    S0 = synth.initial_state(shape, gen)
    a, beta, v, k, q = (dev(x) for x in synth.delta_step_inputs(shape, gen))
    o = torch.empty((2, 2, 16), device="cuda")
    model = ReplaySSM(delta_shape(shape), dev(S0))
    L = lib()
    assert L.rssm_decode_step(model._h, a.data_ptr(), v.data_ptr(), k.data_ptr(), q.data_ptr(), o.data_ptr(),
                              None) == RSSM_EINVAL
    assert L.rssm_decode_step_delta(model._h, a.data_ptr(), None, v.data_ptr(), k.data_ptr(), q.data_ptr(),
                                    o.data_ptr(), None) == RSSM_EINVAL
    with pytest.raises(ValueError):
        model.decode_step(a, v, k, q)
    outer = LayerShape(B=2, H=2, P=16, N=64, G=1, L=4)
    plain = ReplaySSM(outer, dev(S0))
    assert L.rssm_decode_step_delta(plain._h, a.data_ptr(), beta.data_ptr(), v.data_ptr(), k.data_ptr(),
                                    q.data_ptr(), o.data_ptr(), None) == RSSM_EINVAL
    with pytest.raises(RssmError) as ei:  # the outer-product comparator refuses a delta-rule shape
        conventional_step(delta_shape(shape), dev(S0), a, v, k, q)
    assert ei.value.status == RSSM_EINVAL
    cfg = delta_shape(shape).config()
    # a delta-rule layer verifies with rssm_verify_delta (tests/test_gpu_delta_verify.py)
    assert L.rssm_verify(model._h, 1, a.data_ptr(), v.data_ptr(), k.data_ptr(), q.data_ptr(), o.data_ptr(),
                         None) == RSSM_EINVAL
    assert isinstance(cfg, ctypes.Structure)
    torch.cuda.synchronize()
    assert model.read_pointers()[2] == 0 and plain.read_pointers()[2] == 0

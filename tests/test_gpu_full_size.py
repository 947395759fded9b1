"""Parity at the full workload sizes, in the launch configuration bench.py times.

Mamba-2 layer decode: B=256, H=128, P=64, N=128, G=8, L=16, bf16 inputs, 256
steps from an N(0, 0.1^2) state. Speculative verify: the same layer at B=512,
T=4, 64 rounds with seeded accepted lengths in 0..4, flushing every sequence
that reaches 16 records. The same layer as a gated delta-rule layer: 64
decode steps, and 32 speculative rounds at B=512, T=4. The outer-product layer
at T=16 on the tensor-core verify: 24 rounds. The GPU runs the whole batch; the float64 oracle
follows a sample of sequences (all heads) through every step. The pointers
of every sequence are compared bit for bit against the oracle's bookkeeping.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from hybrid_model_ssm_gb300 import ReplaySSM
from tests.gpu_helpers import REL_TOL, PointerShadow, dev, f64, layer_shape, require_gpu, slice_rel_err

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _sample(B, n=8):
    return np.unique(np.linspace(0, B - 1, n).round().astype(int))


def test_mamba2_layer_decode_b256_256_steps():
    require_gpu()
    shape = synth.PRESETS["mamba2_layer_b256_l16"]
    gen = synth.make_generator(shape.seed)
    S0 = synth.initial_state(shape, gen)
    model = ReplaySSM(layer_shape(shape), dev(S0))
    sample = _sample(shape.B)
    orc = oracle.ReplayOracle(f64(S0[sample]), L=shape.L, R=shape.R, G=shape.G)
    shadow = PointerShadow(shape.B, shape.L, shape.R)
    del S0
    worst_o = worst_s = 0.0
    for t in range(256):
        a, v, k, q = synth.decode_step_inputs(shape, gen)
        o = model.decode_step(dev(a), dev(v), dev(k), dev(q))
        o_s = o[torch.as_tensor(sample, device="cuda")].cpu()
        o_ref, flushed = orc.decode(f64(a[sample]), f64(v[sample]), f64(k[sample]), f64(q[sample]))
        shadow.decode()
        e = slice_rel_err(o_s, o_ref, 1)
        worst_o = max(worst_o, e)
        assert e <= REL_TOL, f"step {t}: rel err {e:.3g}"
        if flushed.any():
            ck = model.ckpt[torch.as_tensor(sample, device="cuda")].cpu()
            es = slice_rel_err(ck, orc.ckpt, 2)
            worst_s = max(worst_s, es)
            assert es <= REL_TOL, f"step {t}: checkpoint rel err {es:.3g}"
        if t % 16 == 15 or t < 3:
            start, count, err = model.read_pointers()
            assert err == 0
            assert np.array_equal(start.numpy(), shadow.start) and np.array_equal(count.numpy(), shadow.count)
    print(f"decode b256: worst output rel err {worst_o:.2e}, checkpoint {worst_s:.2e}")


def test_mamba2_verify_b512_t4_64_rounds():
    require_gpu()
    shape = synth.PRESETS["mamba2_verify_b512_t4"]
    T = shape.T_max
    gen = synth.make_generator(shape.seed)
    S0 = synth.initial_state(shape, gen)
    model = ReplaySSM(layer_shape(shape), dev(S0))
    sample = _sample(shape.B)
    sidx = torch.as_tensor(sample, device="cuda")
    orc = oracle.ReplayOracle(f64(S0[sample]), L=shape.L, R=shape.R, G=shape.G)
    shadow = PointerShadow(shape.B, shape.L, shape.R)
    del S0
    worst = 0.0
    flushes = 0
    for r in range(64):
        a, v, k, q = synth.verify_round_inputs(shape, T, gen)
        O = model.verify(dev(a), dev(v), dev(k), dev(q))
        O_ref = orc.verify(f64(a[sample]), f64(v[sample]), f64(k[sample]), f64(q[sample]))
        shadow.verify(T)
        e = slice_rel_err(O[sidx].cpu(), O_ref, 1)
        worst = max(worst, e)
        assert e <= REL_TOL, f"round {r}: verify rel err {e:.3g}"
        acc = synth.accepted_lengths(shape.B, T, gen)
        model.commit(dev(acc))
        orc.commit(acc.numpy()[sample])
        shadow.commit(acc.numpy())
        model.flush(shape.L)
        fl = orc.flush(shape.L)
        shadow.flush(shape.L)
        start, count, err = model.read_pointers()
        assert err == 0
        assert np.array_equal(start.numpy(), shadow.start) and np.array_equal(count.numpy(), shadow.count), f"round {r}"
        if fl.any():
            flushes += int(fl.sum())
            ck = model.ckpt[sidx].cpu()
            for i in np.nonzero(fl)[0]:
                assert slice_rel_err(ck[i], orc.ckpt[i], 2) <= REL_TOL, f"round {r}"
    assert flushes > 0
    print(f"verify b512: worst output rel err {worst:.2e}, sampled flushes {flushes}")


def test_delta_rule_layer_decode_b256_64_steps():
    """The same layer shape as a gated delta-rule layer (bench.py --recurrence
    delta): 64 steps (four flushes), a sample of sequences followed by the
    delta-rule oracle, pointers of every sequence bit for bit."""
    from hybrid_model_ssm_gb300 import LayerShape
    require_gpu()
    shape = synth.PRESETS["mamba2_layer_b256_l16"]
    gen = synth.make_generator(shape.seed + 100)
    S0 = synth.initial_state(shape, gen)
    ls = LayerShape(B=shape.B, H=shape.H, P=shape.P, N=shape.N, G=shape.G, L=shape.L, in_dtype=shape.in_dtype,
                    recurrence="delta")
    model = ReplaySSM(ls, dev(S0))
    sample = _sample(shape.B)
    orc = oracle.DeltaReplayOracle(f64(S0[sample]), L=shape.L, R=shape.R, G=shape.G)
    shadow = PointerShadow(shape.B, shape.L, shape.R)
    del S0
    idx = torch.as_tensor(sample, device="cuda")
    worst_o = worst_s = 0.0
    for t in range(64):
        a, b, v, k, q = synth.delta_step_inputs(shape, gen)
        o = model.decode_step(dev(a), dev(v), dev(k), dev(q), beta=dev(b))
        o_ref, flushed = orc.decode(*(f64(x[sample]) for x in (a, b, v, k, q)))
        shadow.decode()
        e = slice_rel_err(o[idx].cpu(), o_ref, 1)
        worst_o = max(worst_o, e)
        assert e <= REL_TOL, f"step {t}: rel err {e:.3g}"
        if flushed.any():
            es = slice_rel_err(model.ckpt[idx].cpu(), orc.ckpt, 2)
            worst_s = max(worst_s, es)
            assert es <= REL_TOL, f"step {t}: checkpoint rel err {es:.3g}"
        if t % 16 == 15 or t < 3:
            start, count, err = model.read_pointers()
            assert err == 0
            assert np.array_equal(start.numpy(), shadow.start) and np.array_equal(count.numpy(), shadow.count)
    print(f"delta b256: worst output rel err {worst_o:.2e}, checkpoint {worst_s:.2e}")


def test_delta_rule_verify_b512_t4_32_rounds():
    """Speculative rounds on the full-size layer as a gated delta-rule layer (B=512, T=4,
    verify + commit + flush at 16), a sample of sequences followed by the delta-rule
    oracle, pointers of every sequence bit for bit."""
    from hybrid_model_ssm_gb300 import LayerShape
    require_gpu()
    shape = synth.PRESETS["mamba2_verify_b512_t4"]
    T = shape.T_max
    gen = synth.make_generator(shape.seed + 100)
    S0 = synth.initial_state(shape, gen)
    ls = LayerShape(B=shape.B, H=shape.H, P=shape.P, N=shape.N, G=shape.G, L=shape.L, T_max=T,
                    in_dtype=shape.in_dtype, recurrence="delta")
    model = ReplaySSM(ls, dev(S0))
    sample = _sample(shape.B)
    sidx = torch.as_tensor(sample, device="cuda")
    orc = oracle.DeltaReplayOracle(f64(S0[sample]), L=shape.L, R=shape.R, G=shape.G)
    shadow = PointerShadow(shape.B, shape.L, shape.R)
    del S0
    worst = 0.0
    flushes = 0
    for r in range(32):
        a, b, v, k, q = synth.delta_verify_round_inputs(shape, T, gen)
        O = model.verify(dev(a), dev(v), dev(k), dev(q), beta=dev(b))
        O_ref = orc.verify(*(f64(x[sample]) for x in (a, b, v, k, q)))
        shadow.verify(T)
        e = slice_rel_err(O[sidx].cpu(), O_ref, 1)
        worst = max(worst, e)
        assert e <= REL_TOL, f"round {r}: verify rel err {e:.3g}"
        acc = synth.accepted_lengths(shape.B, T, gen)
        model.commit(dev(acc))
        orc.commit(acc.numpy()[sample])
        shadow.commit(acc.numpy())
        model.flush(shape.L)
        fl = orc.flush(shape.L)
        shadow.flush(shape.L)
        start, count, err = model.read_pointers()
        assert err == 0
        assert np.array_equal(start.numpy(), shadow.start) and np.array_equal(count.numpy(), shadow.count), f"round {r}"
        if fl.any():
            flushes += int(fl.sum())
            ck = model.ckpt[sidx].cpu()
            for i in np.nonzero(fl)[0]:
                assert slice_rel_err(ck[i], orc.ckpt[i], 2) <= REL_TOL, f"round {r}"
    assert flushes > 0
    print(f"delta verify b512: worst output rel err {worst:.2e}, sampled flushes {flushes}")


def test_tensor_core_verify_b512_t16_24_rounds():
    """The speculative workload at T=16 (L=16, R=31) on the tensor-core verify, a sample of
    sequences followed by the oracle, pointers of every sequence bit for bit."""
    require_gpu()
    shape = synth.PRESETS["mamba2_verify_b512_t4"].with_(T_max=16)
    T = shape.T_max
    gen = synth.make_generator(shape.seed + 200)
    S0 = synth.initial_state(shape, gen)
    model = ReplaySSM(layer_shape(shape), dev(S0))
    assert model.verify_kernel(T) == "tensor_cores"
    sample = _sample(shape.B)
    sidx = torch.as_tensor(sample, device="cuda")
    orc = oracle.ReplayOracle(f64(S0[sample]), L=shape.L, R=shape.R, G=shape.G)
    shadow = PointerShadow(shape.B, shape.L, shape.R)
    del S0
    worst = 0.0
    for r in range(24):
        a, v, k, q = synth.verify_round_inputs(shape, T, gen)
        O = model.verify(dev(a), dev(v), dev(k), dev(q))
        O_ref = orc.verify(f64(a[sample]), f64(v[sample]), f64(k[sample]), f64(q[sample]))
        shadow.verify(T)
        e = slice_rel_err(O[sidx].cpu(), O_ref, 1)
        worst = max(worst, e)
        assert e <= REL_TOL, f"round {r}: verify rel err {e:.3g}"
        acc = synth.accepted_lengths(shape.B, T, gen)
        model.commit(dev(acc))
        orc.commit(acc.numpy()[sample])
        shadow.commit(acc.numpy())
        model.flush(shape.L)
        orc.flush(shape.L)
        shadow.flush(shape.L)
        start, count, err = model.read_pointers()
        assert err == 0
        assert np.array_equal(start.numpy(), shadow.start) and np.array_equal(count.numpy(), shadow.count), f"round {r}"
    print(f"tensor-core verify b512 t16: worst output rel err {worst:.2e}")


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
def test_read_copy_decode_b256_64_steps(fmt):
    """The same Mamba-2 layer with a read copy, in bench.py's launch configuration (the
    warp-per-head non-flush kernel, then the head kernel): every non-flush output of the
    sampled sequences equals the oracle's output-only form on the device copy (1e-4), every
    flush output the exact recurrence, and every sequence's pointers the oracle's."""
    from tests.test_gpu_readcopy import _dequantized_copy

    require_gpu()
    shape = synth.PRESETS["mamba2_layer_b256_l16"]
    gen = synth.make_generator(shape.seed)
    S0 = synth.initial_state(shape, gen)
    model = ReplaySSM(layer_shape(shape, fmt), dev(S0))
    assert model.decode_kernel() == "warp_per_head"
    sample = _sample(shape.B)
    sub = synth.Shape(B=len(sample), H=shape.H, P=shape.P, N=shape.N, G=shape.G, L=shape.L, seed=shape.seed)
    orc = oracle.ReplayOracle(f64(S0[sample]), L=shape.L, R=shape.R, G=shape.G)
    shadow = PointerShadow(shape.B, shape.L, shape.R)
    del S0
    idx = torch.as_tensor(sample, device="cuda")
    worst = 0.0
    for t in range(64):
        a, v, k, q = synth.decode_step_inputs(shape, gen)
        torch.cuda.synchronize()
        copy_s = model.copy.view(shape.B, -1)[idx].reshape(-1)
        copy_vals = _dequantized_copy(copy_s, sub, fmt)  # what this step's non-flush heads read
        recs_before = [list(r) for r in orc.records]
        o = model.decode_step(dev(a), dev(v), dev(k), dev(q))
        o_s = o[idx].cpu().numpy().astype(np.float64)
        a_s, v_s, k_s, q_s = (f64(x[sample]) for x in (a, v, k, q))
        o_ref, flushed = orc.decode(a_s, v_s, k_s, q_s)
        shadow.decode()
        for i in range(len(sample)):
            if flushed[i]:
                e = slice_rel_err(o_s[i], o_ref[i], 1)
            else:
                alphas = np.stack([r[0] for r in recs_before[i]] + [a_s[i]])
                vs = np.stack([r[1] for r in recs_before[i]] + [v_s[i]])
                ks = np.stack([r[2] for r in recs_before[i]] + [k_s[i]])
                e = slice_rel_err(o_s[i], oracle.replay_output(copy_vals[i], alphas, vs, ks, q_s[i]), 1)
            worst = max(worst, e)
            assert e <= REL_TOL, f"step {t} sequence {sample[i]}: rel err {e:.3g}"
        if t % 16 == 15 or t < 3:
            start, count, err = model.read_pointers()
            assert err == 0
            assert np.array_equal(start.numpy(), shadow.start) and np.array_equal(count.numpy(), shadow.count)
    print(f"{fmt} read copy b256: worst output rel err {worst:.2e}")

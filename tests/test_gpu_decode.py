"""GPU parity: replay decode steps (non-flush and flush) and the conventional kernel.

Every step's output is compared with the float64 oracle on the same seeded
inputs. Pointers, flush events and the appended ring records must match bit
for bit. The checkpoint is compared at every flush. Between flushes it must
stay bit-identical, because a non-flush step writes no state.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from hybrid_model_ssm_gb300 import ReplaySSM, conventional_step
from tests.gpu_helpers import REL_TOL, PointerShadow, check_pointers, dev, f64, layer_shape, require_gpu, slice_rel_err

pytestmark = pytest.mark.gpu

S = synth.Shape
DECODE_CASES = [
    ("tiny_b2_h2_p16_n16_l4", synth.PRESETS["tiny_b2_h2_p16_n16_l4"], 64),
    ("ragged_b3_h4_g2_p8_n32_l3_f32", S(B=3, H=4, P=8, N=32, G=2, L=3, in_dtype="f32", seed=5), 20),
    ("b5_h6_g3_p24_n64_l5_bf16", S(B=5, H=6, P=24, N=64, G=3, L=5, seed=6), 24),
    ("b3_h16_g2_p64_n128_l16_bf16", S(B=3, H=16, P=64, N=128, G=2, L=16, seed=7), 40),
    ("two_row_passes_b2_h4_p128_n128_l16", S(B=2, H=4, P=128, N=128, G=1, L=16, seed=8), 34),
    ("every_step_flushes_l1", S(B=2, H=2, P=16, N=16, G=1, L=1, in_dtype="f32", seed=9), 6),
    ("window_32_b2_h2_p16_n64", S(B=2, H=2, P=16, N=64, G=1, L=32, seed=10), 70),
    ("one_sequence_b1_h1", S(B=1, H=1, P=8, N=16, G=1, L=4, in_dtype="f32", seed=11), 9),
    # the largest sizes: P = N = 128 with the longest ring that fits f32 inputs, and R = 32 with bf16
    ("largest_f32_p128_n128_l29", S(B=2, H=2, P=128, N=128, G=1, L=29, in_dtype="f32", seed=14), 60),
    ("largest_ring_p128_n128_l32_bf16", S(B=2, H=2, P=128, N=128, G=1, L=32, seed=15), 66),
]


def run_decode_parity(shape: synth.Shape, steps: int, mu: float = 0.0):
    require_gpu()
    gen = synth.make_generator(shape.seed)
    S0 = synth.initial_state(shape, gen)
    orc = oracle.ReplayOracle(f64(S0), L=shape.L, R=shape.R, G=shape.G)
    model = ReplaySSM(layer_shape(shape), dev(S0))
    ckpt_prev = model.ckpt.clone()
    worst_o = worst_s = 0.0
    for t in range(steps):
        a, v, k, q = synth.decode_step_inputs(shape, gen, mu)
        o_gpu = model.decode_step(dev(a), dev(v), dev(k), dev(q)).cpu()
        o_ref, flushed = orc.decode(f64(a), f64(v), f64(k), f64(q))
        e = slice_rel_err(o_gpu, o_ref, 1)
        worst_o = max(worst_o, e)
        assert e <= REL_TOL, f"step {t}: output rel err {e:.3g}"
        start, count, err = model.read_pointers()
        assert err == 0
        assert np.array_equal(start.numpy(), orc.start) and np.array_equal(count.numpy(), orc.count), f"step {t}"
        ck = model.ckpt.cpu()
        for b in range(shape.B):
            if flushed[b]:
                es = slice_rel_err(ck[b], orc.ckpt[b], 2)
                worst_s = max(worst_s, es)
                assert es <= REL_TOL, f"step {t} seq {b}: checkpoint rel err {es:.3g}"
            else:
                assert torch.equal(ck[b], ckpt_prev[b].cpu()), f"step {t}: non-flush step wrote the checkpoint"
        ckpt_prev = model.ckpt.clone()
        # the appended record sits at slot (start + count - 1) mod R, bit for bit
        ra, rv, rk = model.ring_views()
        for b in range(shape.B):
            if flushed[b]:
                continue
            slot = (int(start[b]) + int(count[b]) - 1) % shape.R
            assert torch.equal(ra[b, :, slot].cpu(), a[b])
            assert torch.equal(rv[b, :, slot].cpu(), v[b])
            assert torch.equal(rk[b, :, slot].cpu(), k[b])
    return worst_o, worst_s


@pytest.mark.parametrize("name,shape,steps", DECODE_CASES, ids=[c[0] for c in DECODE_CASES])
def test_decode_matches_oracle(name, shape, steps):
    run_decode_parity(shape, steps)


def test_decode_long_memory_decays():
    """Decays near 1 (u ~ N(-4, 1)) keep every buffered record relevant."""
    run_decode_parity(S(B=2, H=8, P=64, N=128, G=2, L=16, seed=12), 48, mu=-4.0)


def test_zero_initial_state_and_zero_inputs():
    """Degenerate case: an all-zero state and all-zero inputs give exact zeros."""
    require_gpu()
    shape = S(B=2, H=4, P=16, N=64, G=2, L=4, seed=13)
    model = ReplaySSM(layer_shape(shape), torch.zeros((2, 4, 16, 64), device="cuda"))
    for _ in range(6):
        o = model.decode_step(torch.ones((2, 4), device="cuda"), torch.zeros((2, 4, 16), dtype=torch.bfloat16, device="cuda"),
                              torch.zeros((2, 2, 64), dtype=torch.bfloat16, device="cuda"),
                              torch.zeros((2, 2, 64), dtype=torch.bfloat16, device="cuda"))
        assert torch.count_nonzero(o) == 0
    assert torch.count_nonzero(model.ckpt) == 0


def test_unit_keys_with_no_decay_are_exact():
    """Brute force: alpha = 1, every key a unit vector e_c and small-integer values
    and state. Then S_t = S_0 + sum_j v_j e_{c_j}^T, and a unit query e_i reads column
    i: o_t = S_0[:, i] + sum of the v_j written to column i. Every term is a small
    integer, so the replay (decode and flush) must reproduce it exactly."""
    require_gpu()
    B, H, P, N, G, L = 2, 4, 16, 64, 2, 4
    shape = S(B=B, H=H, P=P, N=N, G=G, L=L, seed=16)
    rng = np.random.default_rng(16)
    S0 = rng.integers(-4, 5, (B, H, P, N)).astype(np.float32)
    model = ReplaySSM(layer_shape(shape), dev(torch.from_numpy(S0)))
    S_int = S0.astype(np.int64)
    g = oracle.head_groups(H, G)
    ones = torch.ones((B, H), device="cuda")
    for t in range(3 * L + 2):
        col = rng.integers(0, N, (B, G))  # key e_col per (sequence, group)
        qi = rng.integers(0, N, (B, G))   # query e_qi
        v = rng.integers(-3, 4, (B, H, P))
        k = np.zeros((B, G, N), np.float32)
        q = np.zeros((B, G, N), np.float32)
        for b in range(B):
            for gg in range(G):
                k[b, gg, col[b, gg]] = 1.0
                q[b, gg, qi[b, gg]] = 1.0
        o = model.decode_step(ones, dev(torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16)),
                              dev(torch.from_numpy(k).to(torch.bfloat16)),
                              dev(torch.from_numpy(q).to(torch.bfloat16))).cpu().numpy()
        for b in range(B):
            for h in range(H):
                S_int[b, h, :, col[b, g[h]]] += v[b, h]
        want = np.stack([[S_int[b, h, :, qi[b, g[h]]] for h in range(H)] for b in range(B)])
        assert np.array_equal(o, want.astype(np.float32)), f"step {t}"
        if (t + 1) % L == 0:  # a flush step: the checkpoint now holds S_t exactly
            assert np.array_equal(model.ckpt.cpu().numpy(), S_int.astype(np.float32)), f"step {t}"
    _, count, err = model.read_pointers()
    assert err == 0 and np.array_equal(count.numpy(), np.full(B, (3 * L + 2) % L))


def test_zero_decay_keeps_only_the_last_record():
    """alpha = 0 forgets everything before the step: o_t = v_t (k_t . q_t), whatever
    the checkpoint and the buffered records hold, in decode and at a flush."""
    require_gpu()
    shape = S(B=3, H=4, P=32, N=64, G=2, L=4, seed=17)
    gen = synth.make_generator(shape.seed)
    S0 = synth.initial_state(shape, gen)
    orc = oracle.ReplayOracle(f64(S0), L=shape.L, R=shape.R, G=shape.G)
    model = ReplaySSM(layer_shape(shape), dev(S0))
    g = oracle.head_groups(shape.H, shape.G)
    for t in range(10):
        a, v, k, q = synth.decode_step_inputs(shape, gen)
        if t in (2, 3, 6):  # steps 3 and 7 flush (L = 4); step 6 is mid-window
            a = torch.zeros_like(a)
        elif t == 5:
            a[:, ::2] = 0.0  # half of the heads forget
        o = model.decode_step(dev(a), dev(v), dev(k), dev(q)).cpu()
        o_ref, _ = orc.decode(f64(a), f64(v), f64(k), f64(q))
        assert slice_rel_err(o, o_ref, 1) <= REL_TOL, f"step {t}"
        zero = (a == 0).numpy()
        if zero.any():
            kq = np.einsum("bgn,bgn->bg", f64(k), f64(q))[:, g]  # [B,H]
            last = f64(v) * kq[..., None]
            assert slice_rel_err(o.numpy()[zero], last[zero], 1) <= REL_TOL, f"step {t}: not the last record alone"
    _, _, err = model.read_pointers()
    assert err == 0


@pytest.mark.parametrize("shape", [
    S(B=2, H=2, P=16, N=16, G=1, L=4, in_dtype="f32", seed=20),
    S(B=3, H=8, P=64, N=128, G=2, L=16, seed=21),
    S(B=2, H=4, P=40, N=32, G=4, L=16, seed=22),
], ids=["tiny", "b3_h8_p64_n128", "p40_n32"])
def test_conventional_kernel_matches_oracle(shape):
    require_gpu()
    gen = synth.make_generator(shape.seed)
    S0 = synth.initial_state(shape, gen)
    state = dev(S0)
    S_ref = f64(S0)
    ls = layer_shape(shape)
    for t in range(12):
        a, v, k, q = synth.decode_step_inputs(shape, gen)
        o = conventional_step(ls, state, dev(a), dev(v), dev(k), dev(q)).cpu()
        S_ref, o_ref = oracle.conventional_step(S_ref, f64(a), f64(v), f64(k), f64(q))
        assert slice_rel_err(o, o_ref, 1) <= REL_TOL, f"step {t}"
        assert slice_rel_err(state.cpu(), S_ref, 2) <= REL_TOL, f"step {t}"

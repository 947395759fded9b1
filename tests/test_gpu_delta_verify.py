"""GPU parity: speculative verify and commit of gated delta-rule layers.

Each round verifies T drafts with rssm_verify_delta, commits a seeded accepted
length per sequence and flushes every sequence that holds L or more records,
with decode steps in between. The outputs are compared with the float64
delta-rule oracle, which runs the drafts on a scratch copy of the exact state
and then applies only the accepted ones (normwise relative error per
(sequence, head) within 1e-4). The drafts' decays and keys must land in the
ring bit for bit, and each draft's pseudo-value w' = beta (v - alpha y) must
match the oracle's write term of that draft at the same tolerance. Pointers
must match bit for bit, checkpoints at every flush at 1e-4, and rejected drafts
must not change anything that follows.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from hybrid_model_ssm_gb300 import LayerShape, ReplaySSM, RssmError
from tests.gpu_helpers import REL_TOL, dev, f64, require_gpu, slice_rel_err

pytestmark = pytest.mark.gpu

S = synth.Shape
CASES = [
    ("b3_h6_g3_p24_n64_l5_t3_bf16", S(B=3, H=6, P=24, N=64, G=3, L=5, T_max=3, seed=70), 24),
    ("b3_h16_g2_p64_n128_l16_t4_bf16", S(B=3, H=16, P=64, N=128, G=2, L=16, T_max=4, seed=71), 30),
    ("two_row_passes_p128_n128_t4_f32", S(B=2, H=4, P=128, N=128, G=1, L=16, T_max=4, in_dtype="f32", seed=72), 24),
    ("ragged_rows_p8_n64_l2_t4_f32", S(B=3, H=4, P=8, N=64, G=2, L=2, T_max=4, in_dtype="f32", seed=73), 20),
    ("largest_ring_p128_n128_l29_t4_bf16", S(B=2, H=2, P=128, N=128, G=1, L=29, T_max=4, seed=74), 40),
]


def delta_shape(s: synth.Shape) -> LayerShape:
    return LayerShape(B=s.B, H=s.H, P=s.P, N=s.N, G=s.G, L=s.L, T_max=s.T_max, in_dtype=s.in_dtype,
                      recurrence="delta")


def _draft_pseudo_values(S, a, b, v, k):
    """The oracle's write term of each draft, the drafts applied in turn to a scratch copy of S."""
    Sc = S.copy()
    out = []
    for t in range(a.shape[1]):
        out.append(oracle.delta_pseudo_value(Sc, a[:, t], b[:, t], v[:, t], k[:, t]))
        Sc, _ = oracle.delta_step(Sc, a[:, t], b[:, t], v[:, t], k[:, t], k[:, t])
    return np.stack(out, axis=1)  # [B,T,H,P]


def run_delta_verify_parity(shape: synth.Shape, rounds: int, decode_every: int = 3):
    require_gpu()
    gen = synth.make_generator(shape.seed)
    S0 = synth.initial_state(shape, gen)
    orc = oracle.DeltaReplayOracle(f64(S0), L=shape.L, R=shape.R, G=shape.G)
    model = ReplaySSM(delta_shape(shape), dev(S0))
    for r in range(rounds):
        if decode_every and r % decode_every == 0:
            a, b, v, k, q = synth.delta_step_inputs(shape, gen)
            o = model.decode_step(dev(a), dev(v), dev(k), dev(q), beta=dev(b)).cpu()
            o_ref, _ = orc.decode(*(f64(x) for x in (a, b, v, k, q)))
            assert slice_rel_err(o, o_ref, 1) <= REL_TOL, f"round {r}: decode"
        T = 1 + (r % shape.T_max)
        a, b, v, k, q = synth.delta_verify_round_inputs(shape, T, gen)
        w_ref = _draft_pseudo_values(orc.S, *(f64(x) for x in (a, b, v, k)))
        O = model.verify(dev(a), dev(v), dev(k), dev(q), beta=dev(b)).cpu()
        O_ref = orc.verify(*(f64(x) for x in (a, b, v, k, q)))
        e = slice_rel_err(O, O_ref, 1)
        assert e <= REL_TOL, f"round {r}: verify rel err {e:.3g}"
        ra, rw, rk = (x.cpu() for x in model.ring_views())
        for bb in range(shape.B):
            slots = [(int(orc.start[bb]) + int(orc.count[bb]) + t) % shape.R for t in range(T)]
            assert torch.equal(ra[bb][:, slots], a[bb].T), f"round {r} seq {bb}: draft decays in the ring"
            assert torch.equal(rk[bb][:, slots], k[bb].transpose(0, 1)), f"round {r} seq {bb}: draft keys"
            ew = slice_rel_err(rw[bb][:, slots].transpose(0, 1).numpy(), w_ref[bb], 1)
            assert ew <= REL_TOL, f"round {r} seq {bb}: draft pseudo-values {ew:.3g}"
        acc = synth.accepted_lengths(shape.B, T, gen)
        ck_before = model.ckpt.clone()
        model.commit(dev(acc))
        orc.commit(acc.numpy())
        flushed = orc.flush(shape.L)
        model.flush(shape.L)
        start, count, err = model.read_pointers()
        assert err == 0
        assert np.array_equal(start.numpy(), orc.start) and np.array_equal(count.numpy(), orc.count), f"round {r}"
        ck = model.ckpt.cpu()
        for bb in range(shape.B):
            if flushed[bb]:
                assert slice_rel_err(ck[bb], orc.ckpt[bb], 2) <= REL_TOL, f"round {r} seq {bb}: checkpoint"
            else:
                assert torch.equal(ck[bb], ck_before[bb].cpu())


@pytest.mark.parametrize("name,shape,rounds", CASES, ids=[c[0] for c in CASES])
def test_delta_verify_commit_flush_match_oracle(name, shape, rounds):
    run_delta_verify_parity(shape, rounds)


def test_delta_rejected_drafts_do_not_matter():
    """The same run with every rejected draft replaced by garbage gives bit-identical
    outputs of the accepted drafts, pointers, checkpoints and later decode outputs."""
    require_gpu()
    shape = S(B=4, H=8, P=32, N=64, G=2, L=6, T_max=4, seed=75)
    results = []
    for garbage in (False, True):
        gen = synth.make_generator(shape.seed)
        model = ReplaySSM(delta_shape(shape), dev(synth.initial_state(shape, gen)))
        outs = []
        for r in range(12):
            a, b, v, k, q = synth.delta_verify_round_inputs(shape, shape.T_max, gen)
            acc = synth.accepted_lengths(shape.B, shape.T_max, gen)
            if garbage:
                for bb in range(shape.B):
                    n = int(acc[bb])
                    a[bb, n:] = 0.37
                    b[bb, n:] = 0.9
                    v[bb, n:] = 1e4
                    k[bb, n:] = -2e3
            O = model.verify(dev(a), dev(v), dev(k), dev(q), beta=dev(b)).cpu()
            outs.append(torch.cat([O[bb, : int(acc[bb])].flatten() for bb in range(shape.B)]))
            model.commit(dev(acc))
            model.flush(shape.L)
            a2, b2, v2, k2, q2 = synth.delta_step_inputs(shape, gen)
            outs.append(model.decode_step(dev(a2), dev(v2), dev(k2), dev(q2), beta=dev(b2)).cpu().flatten())
        start, count, _ = model.read_pointers()
        results.append((outs, model.ckpt.cpu(), start, count))
    (o0, c0, s0, n0), (o1, c1, s1, n1) = results
    assert torch.equal(c0, c1) and torch.equal(s0, s1) and torch.equal(n0, n1)
    for x, y in zip(o0, o1):
        assert torch.equal(x, y)


def test_delta_verify_entry_points_refuse_the_other_recurrence():
    require_gpu()
    shape = S(B=2, H=2, P=16, N=64, G=1, L=4, T_max=2, in_dtype="f32", seed=76)
    gen = synth.make_generator(shape.seed)
    outer = ReplaySSM(LayerShape(B=2, H=2, P=16, N=64, G=1, L=4, T_max=2, in_dtype="f32"),
                      dev(synth.initial_state(shape, gen)))
    delta = ReplaySSM(delta_shape(shape), dev(synth.initial_state(shape, gen)))
    a, b, v, k, q = (dev(x) for x in synth.delta_verify_round_inputs(shape, 2, gen))
    with pytest.raises(ValueError):
        outer.verify(a, v, k, q, beta=b)  # the binding refuses beta for the outer-product recurrence
    with pytest.raises(ValueError):
        delta.verify(a, v, k, q)
    assert delta.verify_kernel(2) == "cuda_cores"
    with pytest.raises(RssmError):
        delta.set_verify_kernel("tensor_cores")

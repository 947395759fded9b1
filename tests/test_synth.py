"""The seeded input recipe (synth/inputs.py), checked on the CPU.

The recipe is stated in the design notes and shared by the tests and the
bench: S0 ~ N(0, 0.1^2); per step u ~ N(mu, 1), alpha = exp(-softplus(u));
v, k, q ~ N(0, 1)/sqrt(N) in the storage dtype; per verify round the same
with a draft axis, and accepted lengths uniform on 0..T; delta-rule steps add
beta = sigmoid(N(0, 1)) and unit-norm keys and queries. These checks pin the
shapes, dtypes, value ranges and moments, and that a seed fixes the draws.
"""
import math

import torch

import synth


def test_shapes_dtypes_and_determinism():
    s = synth.Shape(B=3, H=4, P=16, N=32, G=2, L=4, T_max=3, seed=7)
    g1, g2 = synth.make_generator(s.seed), synth.make_generator(s.seed)
    a1, a2 = synth.decode_step_inputs(s, g1), synth.decode_step_inputs(s, g2)
    assert all(torch.equal(x, y) for x, y in zip(a1, a2))
    alpha, v, k, q = a1
    assert alpha.shape == (3, 4) and alpha.dtype == torch.float32
    assert v.shape == (3, 4, 16) and k.shape == q.shape == (3, 2, 32) and v.dtype == torch.bfloat16
    A, V, K, Q = synth.verify_round_inputs(s, 3, g1)
    assert A.shape == (3, 3, 4) and V.shape == (3, 3, 4, 16) and K.shape == Q.shape == (3, 3, 2, 32)
    acc = synth.accepted_lengths(1000, 3, g1)
    assert acc.dtype == torch.int32 and acc.min() == 0 and acc.max() == 3
    assert synth.Shape(B=1, H=1, P=8, N=16, G=1, L=4, in_dtype="f32").torch_dtype == torch.float32


def test_value_distributions():
    s = synth.Shape(B=64, H=128, P=64, N=128, G=8, L=16, seed=3)
    g = synth.make_generator(s.seed)
    S0 = synth.initial_state(s.with_(B=4), g)
    assert S0.dtype == torch.float32 and abs(S0.std().item() - 0.1) < 2e-3 and abs(S0.mean().item()) < 2e-3
    alpha, v, k, q = synth.decode_step_inputs(s, g)
    assert (alpha > 0).all() and (alpha < 1).all()
    # alpha = exp(-softplus(u)) = sigmoid(-u), so E[alpha] = 1/2 for u ~ N(0, 1) by symmetry
    assert abs(alpha.mean().item() - 0.5) < 0.02
    for x in (v, k, q):
        assert abs(x.float().std().item() * math.sqrt(s.N) - 1.0) < 0.02
    long_alpha = synth.decode_step_inputs(s, g, mu=-4.0)[0]
    assert long_alpha.mean().item() > 0.95  # the long-memory variant


def test_delta_rule_inputs():
    s = synth.Shape(B=16, H=8, P=16, N=64, G=2, L=4, seed=5)
    alpha, beta, v, k, q = synth.delta_step_inputs(s, synth.make_generator(s.seed))
    assert (beta > 0).all() and (beta < 1).all() and abs(beta.mean().item() - 0.5) < 0.05
    for x in (k, q):
        assert torch.allclose(x.float().norm(dim=-1), torch.ones(16, 2), atol=1e-2)  # unit norm, then bf16

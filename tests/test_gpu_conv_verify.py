"""GPU parity: the conventional speculative verify used as the comparison path.

Each round advances the full state through T drafts and writes a snapshot
after each (rssm_conventional_verify), then points every sequence at the
snapshot after its accepted drafts (rssm_conventional_commit). The outputs
must match the float64 oracle's verify outputs, and the committed state the
oracle's exact state after only the accepted drafts.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from hybrid_model_ssm_gb300 import ConventionalVerifier
from tests.gpu_helpers import REL_TOL, dev, f64, layer_shape, require_gpu, slice_rel_err

pytestmark = pytest.mark.gpu

S = synth.Shape
CASES = [
    ("b3_h16_g2_p64_n128_t4", S(B=3, H=16, P=64, N=128, G=2, L=16, T_max=4, seed=70), 12),
    ("f32_b2_h4_p16_n32_t3", S(B=2, H=4, P=16, N=32, G=2, L=4, T_max=3, in_dtype="f32", seed=71), 10),
    ("b5_h6_g3_p24_n64_t8", S(B=5, H=6, P=24, N=64, G=3, L=8, T_max=8, seed=72), 8),
]


@pytest.mark.parametrize("name,shape,rounds", CASES, ids=[c[0] for c in CASES])
def test_conventional_verify_matches_oracle(name, shape, rounds):
    require_gpu()
    gen = synth.make_generator(shape.seed)
    S0 = synth.initial_state(shape, gen)
    conv = ConventionalVerifier(layer_shape(shape), dev(S0))
    orc = oracle.ReplayOracle(f64(S0), L=shape.L, R=shape.R, G=shape.G)
    for r in range(rounds):
        T = 1 + r % shape.T_max
        a, v, k, q = synth.verify_round_inputs(shape, T, gen)
        O = conv.verify(dev(a), dev(v), dev(k), dev(q)).cpu()
        O_ref = orc.verify(f64(a), f64(v), f64(k), f64(q))
        assert slice_rel_err(O, O_ref, 1) <= REL_TOL, f"round {r}: outputs"
        acc = synth.accepted_lengths(shape.B, T, gen)
        conv.commit(dev(acc))
        orc.commit(acc.numpy())
        orc.flush(shape.L)  # keeps the oracle's ring within capacity; its exact state is unchanged
        assert slice_rel_err(conv.state().cpu(), orc.S, 2) <= REL_TOL, f"round {r}: committed state"
    assert int(conv.err.item()) == 0


def test_conventional_verify_error_paths():
    """A slot index outside 0..T_max skips the sequence; a bad accepted length
    leaves its slot alone. Both set a bit in the error word and nothing faults."""
    require_gpu()
    shape = S(B=3, H=4, P=16, N=32, G=2, L=4, T_max=2, seed=73)
    gen = synth.make_generator(shape.seed)
    conv = ConventionalVerifier(layer_shape(shape), dev(synth.initial_state(shape, gen)))
    a, v, k, q = (dev(x) for x in synth.verify_round_inputs(shape, 2, gen))
    conv.cur[1] = conv.nslot  # out of range
    out = torch.full((3, 2, 4, 16), 7.0, device="cuda")
    conv.verify(a, v, k, q, out=out)
    torch.cuda.synchronize()
    assert int(conv.err.item()) & 1
    assert torch.all(out[1] == 7.0) and not torch.all(out[0] == 7.0) and not torch.all(out[2] == 7.0)
    conv.err.zero_()
    conv.cur[1] = 0
    conv.commit(torch.tensor([1, 3, -1], dtype=torch.int32, device="cuda"))  # 3 > T = 2, -1 < 0
    torch.cuda.synchronize()
    assert int(conv.err.item()) & 2
    assert conv.cur.tolist() == [1, 0, 0]

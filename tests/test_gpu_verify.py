"""GPU parity: speculative verify, commit and standalone flush, mixed with decode steps.

Each round verifies T drafts, commits a seeded accepted length per sequence,
and flushes every sequence holding L or more records. The outputs are
compared with the oracle, which runs the drafts on a scratch state and then
replays only the accepted ones. The pointers must match bit for bit, and so
must the checkpoint of every sequence that did not flush.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from hybrid_model_ssm_gb300 import ReplaySSM
from tests.gpu_helpers import REL_TOL, dev, f64, layer_shape, require_gpu, slice_rel_err

pytestmark = pytest.mark.gpu

S = synth.Shape
VERIFY_CASES = [
    ("tiny_t3_f32", S(B=3, H=2, P=16, N=16, G=1, L=4, T_max=3, in_dtype="f32", seed=30), 24),
    ("b4_h16_g2_p64_n128_l16_t4", S(B=4, H=16, P=64, N=128, G=2, L=16, T_max=4, seed=31), 30),
    ("t8_two_query_blocks_n64", S(B=3, H=4, P=24, N=64, G=2, L=8, T_max=8, seed=32), 16),
    ("t5_partial_block_n32", S(B=5, H=6, P=16, N=32, G=3, L=6, T_max=5, seed=33), 16),
    ("largest_ring_p128_n128_l25_t8", S(B=3, H=2, P=128, N=128, G=1, L=25, T_max=8, seed=35), 24),
]


def run_verify_parity(shape: synth.Shape, rounds: int, decode_every: int = 3, vary_T: bool = True,
                      verify_kernel: str = "auto", check_ring: bool = False):
    """Rounds of (decode every few rounds,) verify, commit and flush against the oracle.

    verify_kernel picks the verify launches' kernel ("auto", "cuda_cores",
    "tensor_cores"). check_ring also checks, after every verify, that the drafts'
    decays, values and keys sit in the ring slots after the committed records, bit for bit.
    """
    require_gpu()
    gen = synth.make_generator(shape.seed)
    S0 = synth.initial_state(shape, gen)
    orc = oracle.ReplayOracle(f64(S0), L=shape.L, R=shape.R, G=shape.G)
    model = ReplaySSM(layer_shape(shape), dev(S0))
    model.set_verify_kernel(verify_kernel)
    for r in range(rounds):
        if decode_every and r % decode_every == 0:
            a, v, k, q = synth.decode_step_inputs(shape, gen)
            o = model.decode_step(dev(a), dev(v), dev(k), dev(q)).cpu()
            o_ref, _ = orc.decode(f64(a), f64(v), f64(k), f64(q))
            assert slice_rel_err(o, o_ref, 1) <= REL_TOL, f"round {r} decode"
        T = 1 + (r % shape.T_max) if vary_T else shape.T_max
        a, v, k, q = synth.verify_round_inputs(shape, T, gen)
        O = model.verify(dev(a), dev(v), dev(k), dev(q)).cpu()
        O_ref = orc.verify(f64(a), f64(v), f64(k), f64(q))
        e = slice_rel_err(O, O_ref, 1)
        assert e <= REL_TOL, f"round {r}: verify rel err {e:.3g}"
        if check_ring:
            ra, rv, rk = (x.cpu() for x in model.ring_views())
            for b in range(shape.B):
                slots = [(int(orc.start[b]) + int(orc.count[b]) + t) % shape.R for t in range(T)]
                assert torch.equal(ra[b][:, slots], a[b].T), f"round {r} seq {b}: draft decays in the ring"
                assert torch.equal(rv[b][:, slots], v[b].transpose(0, 1)), f"round {r} seq {b}: draft values"
                assert torch.equal(rk[b][:, slots], k[b].transpose(0, 1)), f"round {r} seq {b}: draft keys"
        acc = synth.accepted_lengths(shape.B, T, gen)
        ck_before = model.ckpt.clone()
        model.commit(dev(acc))
        orc.commit(acc.numpy())
        flushed = orc.flush(shape.L)
        model.flush(shape.L)
        start, count, err = model.read_pointers()
        assert err == 0
        assert np.array_equal(start.numpy(), orc.start), f"round {r}"
        assert np.array_equal(count.numpy(), orc.count), f"round {r}"
        ck = model.ckpt.cpu()
        for b in range(shape.B):
            if flushed[b]:
                assert slice_rel_err(ck[b], orc.ckpt[b], 2) <= REL_TOL, f"round {r} seq {b}"
            else:
                assert torch.equal(ck[b], ck_before[b].cpu())


@pytest.mark.parametrize("name,shape,rounds", VERIFY_CASES, ids=[c[0] for c in VERIFY_CASES])
def test_verify_commit_flush_match_oracle(name, shape, rounds):
    run_verify_parity(shape, rounds)


def test_rejected_drafts_do_not_matter():
    """Rollback invariant on the device: the same run with every rejected draft
    replaced by garbage gives bit-identical outputs, pointers and checkpoints."""
    require_gpu()
    shape = S(B=4, H=8, P=32, N=64, G=2, L=6, T_max=4, seed=34)
    results = []
    for garbage in (False, True):
        gen = synth.make_generator(shape.seed)
        model = ReplaySSM(layer_shape(shape), dev(synth.initial_state(shape, gen)))
        outs = []
        for r in range(12):
            a, v, k, q = synth.verify_round_inputs(shape, shape.T_max, gen)
            acc = synth.accepted_lengths(shape.B, shape.T_max, gen)
            if garbage:
                for b in range(shape.B):
                    n = int(acc[b])
                    a[b, n:] = 0.37
                    v[b, n:] = 1e4
                    k[b, n:] = -2e3
            O = model.verify(dev(a), dev(v), dev(k), dev(q)).cpu()
            outs.append(torch.cat([O[b, : int(acc[b])].flatten() for b in range(shape.B)]))
            model.commit(dev(acc))
            model.flush(shape.L)
            a2, v2, k2, q2 = synth.decode_step_inputs(shape, gen)
            outs.append(model.decode_step(dev(a2), dev(v2), dev(k2), dev(q2)).cpu().flatten())
        start, count, _ = model.read_pointers()
        results.append((outs, model.ckpt.cpu(), start, count))
    (o0, c0, s0, n0), (o1, c1, s1, n1) = results
    assert torch.equal(c0, c1) and torch.equal(s0, s1) and torch.equal(n0, n1)
    for x, y in zip(o0, o1):
        assert torch.equal(x, y)


def test_save_and_resume_gives_identical_outputs():
    """The state is (checkpoint, ring, pointers): copying those buffers and
    copying them back resumes decoding bit-exactly."""
    require_gpu()
    shape = S(B=3, H=8, P=64, N=128, G=2, L=5, T_max=2, seed=35)
    gen = synth.make_generator(shape.seed)
    model = ReplaySSM(layer_shape(shape), dev(synth.initial_state(shape, gen)))
    steps = [synth.decode_step_inputs(shape, gen) for _ in range(14)]
    for a, v, k, q in steps[:7]:
        model.decode_step(dev(a), dev(v), dev(k), dev(q))
    saved = (model.ckpt.clone(), model.ring.clone(), model.ptrs.clone())
    first = [model.decode_step(dev(a), dev(v), dev(k), dev(q)).cpu() for a, v, k, q in steps[7:]]
    model.ckpt.copy_(saved[0])
    model.ring.copy_(saved[1])
    model.ptrs.copy_(saved[2])
    second = [model.decode_step(dev(a), dev(v), dev(k), dev(q)).cpu() for a, v, k, q in steps[7:]]
    for x, y in zip(first, second):
        assert torch.equal(x, y)


def test_mixed_calls_without_pointer_reads():
    """Decode steps, verify rounds, commits and flushes in a seeded random order,
    with no pointer read in between, so the launch plans rest on the host's
    count bounds alone. Outputs follow the oracle at every call; the pointers
    and the error word are checked once at the end."""
    require_gpu()
    shape = S(B=6, H=4, P=32, N=64, G=2, L=5, T_max=3, seed=34)
    gen = synth.make_generator(shape.seed)
    S0 = synth.initial_state(shape, gen)
    orc = oracle.ReplayOracle(f64(S0), L=shape.L, R=shape.R, G=shape.G)
    model = ReplaySSM(layer_shape(shape), dev(S0))
    ops = np.random.default_rng(7).integers(0, 3, size=60)
    for i, op in enumerate(ops):
        if op < 2:  # decode
            a, v, k, q = synth.decode_step_inputs(shape, gen)
            o = model.decode_step(dev(a), dev(v), dev(k), dev(q)).cpu()
            o_ref, _ = orc.decode(f64(a), f64(v), f64(k), f64(q))
            assert slice_rel_err(o, o_ref, 1) <= REL_TOL, f"call {i}: decode"
        else:  # verify, commit, flush at L
            T = 1 + i % shape.T_max
            a, v, k, q = synth.verify_round_inputs(shape, T, gen)
            O = model.verify(dev(a), dev(v), dev(k), dev(q)).cpu()
            assert slice_rel_err(O, orc.verify(f64(a), f64(v), f64(k), f64(q)), 1) <= REL_TOL, f"call {i}: verify"
            acc = synth.accepted_lengths(shape.B, T, gen)
            model.commit(dev(acc))
            orc.commit(acc.numpy())
            model.flush(shape.L)
            orc.flush(shape.L)
    start, count, err = model.read_pointers()
    assert err == 0
    assert np.array_equal(start.numpy(), orc.start) and np.array_equal(count.numpy(), orc.count)
    assert slice_rel_err(model.ckpt.cpu(), orc.ckpt, 2) <= REL_TOL

"""GPU parity of the tensor-core verify (tcgen05 kind::tf32 MMAs, split checkpoint).

The checkpoint product S_ckpt Q runs on the tensor cores with the checkpoint
split into a TF32-exact high part and the remainder, so the outputs must meet
the FP32 path's tolerance (1e-4 per (sequence, head)) against the float64
oracle: verify rounds with commits, flushes and decode steps in between, every
draft count from 1 to 16, items of one, two and four heads (P = 128, 64, 32),
both key sizes (N = 128, 64), batches that split unevenly over the CTAs, and the
largest ring (R = 32). The drafts' records must land in the ring bit for bit,
and rejected drafts must not change anything that follows.
"""
import numpy as np
import pytest
import torch

import synth
from hybrid_model_ssm_gb300 import LayerShape, ReplaySSM, RssmError, launch_plan
from tests.gpu_helpers import dev, layer_shape, require_gpu
from tests.test_gpu_verify import run_verify_parity

pytestmark = pytest.mark.gpu

S = synth.Shape
TC_CASES = [
    # name, shape, rounds
    ("p64_n128_l16_t16", S(B=5, H=16, P=64, N=128, G=2, L=16, T_max=16, seed=60), 34),
    ("p128_n128_l8_t12", S(B=3, H=4, P=128, N=128, G=2, L=8, T_max=12, seed=61), 26),
    ("p32_n64_l6_t9", S(B=7, H=8, P=32, N=64, G=2, L=6, T_max=9, seed=62), 20),
    ("p64_n64_l4_t16", S(B=3, H=4, P=64, N=64, G=1, L=4, T_max=16, seed=63), 20),
    ("largest_ring_l17_t16", S(B=2, H=2, P=64, N=128, G=1, L=17, T_max=16, seed=64), 20),
]


@pytest.mark.parametrize("name,shape,rounds", TC_CASES, ids=[c[0] for c in TC_CASES])
def test_tensor_core_verify_matches_oracle(name, shape, rounds):
    run_verify_parity(shape, rounds, verify_kernel="tensor_cores", check_ring=True)


def test_tensor_core_verify_at_small_t_matches_oracle():
    """Draft counts 1..4 forced onto the tensor cores (zero-padded query columns)."""
    shape = S(B=4, H=16, P=64, N=128, G=2, L=16, T_max=4, seed=65)
    run_verify_parity(shape, 24, verify_kernel="tensor_cores")


def test_kernel_choice():
    require_gpu()
    shape = S(B=2, H=4, P=64, N=128, G=2, L=8, T_max=16, seed=66)
    model = ReplaySSM(layer_shape(shape), dev(synth.initial_state(shape, synth.make_generator(66))))
    assert model.verify_kernel(4) == "cuda_cores" and model.verify_kernel(8) == "cuda_cores"
    assert model.verify_kernel(9) == "tensor_cores" and model.verify_kernel(16) == "tensor_cores"
    model.set_verify_kernel("cuda_cores")
    assert model.verify_kernel(8) == "cuda_cores" and model.verify_kernel(9) == "tensor_cores"
    model.set_verify_kernel("tensor_cores")
    assert model.verify_kernel(1) == "tensor_cores"
    f32 = S(B=2, H=4, P=64, N=128, G=2, L=8, T_max=8, in_dtype="f32", seed=67)
    fmodel = ReplaySSM(layer_shape(f32), dev(synth.initial_state(f32, synth.make_generator(67))))
    assert fmodel.verify_kernel(8) == "cuda_cores"
    with pytest.raises(RssmError):
        fmodel.set_verify_kernel("tensor_cores")
    plan = launch_plan(LayerShape(B=512, H=128, P=64, N=128, G=8, L=16, T_max=16), "verify_tc")
    assert plan["smem_bytes"] <= 227 * 1024 and plan["layouts"][0]["stages"] >= 4


def test_tensor_core_and_cuda_core_verify_agree():
    """Both kernels on the same state and drafts (T = 8): within 1e-5 of each other (1.9e-6
    measured). The tensor-core kernel reads the checkpoint tile as stored and lets kind::tf32
    ignore the low 13 mantissa bits (its hi part); a conversion that rounded instead would
    leave about 1e-4 here."""
    require_gpu()
    shape = S(B=6, H=16, P=64, N=128, G=2, L=16, T_max=8, seed=68)
    gen = synth.make_generator(shape.seed)
    S0 = dev(synth.initial_state(shape, gen))
    ma, mb = ReplaySSM(layer_shape(shape), S0.clone()), ReplaySSM(layer_shape(shape), S0.clone())
    ma.set_verify_kernel("cuda_cores")
    mb.set_verify_kernel("tensor_cores")
    for r in range(6):
        a, v, k, q = (dev(x) for x in synth.verify_round_inputs(shape, 8, gen))
        oa, ob = ma.verify(a, v, k, q).cpu().double(), mb.verify(a, v, k, q).cpu().double()
        rel = ((oa - ob).abs().amax(-1) / ob.abs().amax(-1).clamp_min(1e-30)).max().item()
        assert rel <= 1e-5, f"round {r}: {rel:.3g}"
        acc = dev(synth.accepted_lengths(shape.B, 8, gen))
        for m in (ma, mb):
            m.commit(acc)
            m.flush(shape.L)
    # the pointer blocks agree bit for bit (ring slots never written hold uninitialised bytes)
    assert torch.equal(ma.ptrs, mb.ptrs)


def test_rejected_drafts_do_not_matter_on_tensor_cores():
    require_gpu()
    shape = S(B=4, H=8, P=64, N=128, G=2, L=8, T_max=16, seed=69)
    results = []
    for garbage in (False, True):
        gen = synth.make_generator(shape.seed)
        model = ReplaySSM(layer_shape(shape), dev(synth.initial_state(shape, gen)))
        model.set_verify_kernel("tensor_cores")
        outs = []
        for r in range(10):
            T = 16 if r % 2 else 7
            a, v, k, q = synth.verify_round_inputs(shape, T, gen)
            acc = synth.accepted_lengths(shape.B, T, gen)
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
        start, count, _ = model.read_pointers()
        results.append((outs, model.ckpt.cpu(), start, count))
    (o0, c0, s0, n0), (o1, c1, s1, n1) = results
    assert torch.equal(c0, c1) and torch.equal(s0, s1) and torch.equal(n0, n1)
    for x, y in zip(o0, o1):
        assert torch.equal(x, y)

"""The decode step that allocates nothing (rssm_decode_step_static_scratch).

This is for callers that cannot give the library more device memory while
decoding runs: an engine that carves one fixed arena at start-up and hands
out nothing else, code running while another component owns the device
allocator, or a stream under graph capture, where cudaMalloc is not allowed.
The variant keeps the kernel's per-sequence ticket counters in a static device
array of the library instead of the caller's pointer block.

The tests call it through the C ABI. They check it against rssm_decode_step
on the same state and inputs for two calls in a row (the second is a flush
step, so both kernel paths run), against the float64 oracle over a full
window and a flush with a batch that does not fill the CTA tiling, and they
check its two refusals. The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from hybrid_model_ssm_gb300 import LayerShape, ReplaySSM, lib
from hybrid_model_ssm_gb300.rssm import RSSM_EUNSUPPORTED, RSSM_OK
from tests.gpu_helpers import REL_TOL, dev, f64, layer_shape, require_gpu, slice_rel_err

pytestmark = pytest.mark.gpu


def _static_step(model, a, v, k, q, o) -> int:
    stream = torch.cuda.current_stream().cuda_stream
    return lib().rssm_decode_step_static_scratch(model._h, a.data_ptr(), v.data_ptr(), k.data_ptr(), q.data_ptr(),
                                                 o.data_ptr(), ctypes.c_void_p(stream))


def test_static_scratch_decode_matches_decode_step():
    require_gpu()
    shape = synth.Shape(B=5, H=8, P=64, N=128, G=2, L=2, seed=90)
    gen = synth.make_generator(shape.seed)
    S0 = synth.initial_state(shape, gen)
    ref = ReplaySSM(layer_shape(shape), dev(S0))
    alt = ReplaySSM(layer_shape(shape), dev(S0))
    for call in range(2):
        a, v, k, q = (dev(x) for x in synth.decode_step_inputs(shape, gen))
        o_ref = ref.decode_step(a, v, k, q)
        o_alt = torch.full_like(o_ref, float("nan"))
        status = _static_step(alt, a, v, k, q, o_alt)
        assert status == RSSM_OK, lib().rssm_last_error().decode()
        assert slice_rel_err(o_alt.cpu(), o_ref.cpu().double().numpy(), 1) <= REL_TOL, f"call {call}"
        s_ref, c_ref, e_ref = ref.read_pointers()
        s_alt, c_alt, e_alt = alt.read_pointers()
        assert e_ref == 0 and e_alt == 0
        assert torch.equal(s_ref, s_alt) and torch.equal(c_ref, c_alt), f"call {call}: pointers differ"
        assert slice_rel_err(alt.ckpt.cpu(), ref.ckpt.cpu().double().numpy(), 2) <= REL_TOL
    assert np.array_equal(c_alt.numpy(), np.zeros(shape.B, np.int32))  # the second call flushed


def test_static_scratch_decode_matches_oracle_over_a_window():
    """17 steps at L = 16 (15 non-flush, one flush, one more non-flush) with B = 7, whose
    7 x 8 heads split unevenly over the persistent CTAs: outputs at 1e-4, pointers bit-exact,
    the checkpoint at the flush at 1e-4."""
    require_gpu()
    shape = synth.Shape(B=7, H=8, P=64, N=128, G=2, L=16, seed=91)
    gen = synth.make_generator(shape.seed)
    S0 = synth.initial_state(shape, gen)
    model = ReplaySSM(layer_shape(shape), dev(S0))
    orc = oracle.ReplayOracle(f64(S0), L=shape.L, R=shape.R, G=shape.G)
    out = torch.empty((shape.B, shape.H, shape.P), dtype=torch.float32, device="cuda")
    for t in range(shape.L + 1):
        a, v, k, q = synth.decode_step_inputs(shape, gen)
        status = _static_step(model, dev(a), dev(v), dev(k), dev(q), out)
        assert status == RSSM_OK, lib().rssm_last_error().decode()
        o_ref, flushed = orc.decode(f64(a), f64(v), f64(k), f64(q))
        rel = slice_rel_err(out.cpu(), o_ref, 1)
        assert rel <= REL_TOL, f"step {t}: {rel:.3g}"
        start, count, err = model.read_pointers()
        assert err == 0
        assert np.array_equal(start.numpy(), orc.start) and np.array_equal(count.numpy(), orc.count), f"step {t}"
        if flushed.any():
            assert slice_rel_err(model.ckpt.cpu(), orc.ckpt, 2) <= REL_TOL


def test_static_scratch_refusals():
    """More sequences than the static array holds, and a delta-rule layer, are refused on the host."""
    require_gpu()
    big = LayerShape(B=8193, H=1, P=8, N=16, G=1, L=2, in_dtype="f32")
    model = ReplaySSM(big, torch.zeros((big.B, 1, 8, 16), dtype=torch.float32, device="cuda"))
    a = torch.ones((big.B, 1), device="cuda")
    v = torch.zeros((big.B, 1, 8), device="cuda")
    k = torch.zeros((big.B, 1, 16), device="cuda")
    o = torch.empty((big.B, 1, 8), device="cuda")
    assert _static_step(model, a, v, k, k, o) == RSSM_EUNSUPPORTED
    assert "8192" in lib().rssm_last_error().decode()
    ds = LayerShape(B=2, H=2, P=8, N=64, G=1, L=2, in_dtype="f32", recurrence="delta")
    dmodel = ReplaySSM(ds, torch.zeros((2, 2, 8, 64), dtype=torch.float32, device="cuda"))
    a = torch.ones((2, 2), device="cuda")
    v = torch.zeros((2, 2, 8), device="cuda")
    k = torch.zeros((2, 1, 64), device="cuda")
    o = torch.empty((2, 2, 8), device="cuda")
    assert _static_step(dmodel, a, v, k, k, o) == RSSM_EUNSUPPORTED
    assert "outer-product" in lib().rssm_last_error().decode()
    torch.cuda.synchronize()


def test_static_scratch_binding_read_copy_two_kernels():
    """Through the Python binding, on an E4M3 read-copy layer with bf16 inputs (the
    warp-per-head kernel, then the head kernel): a window, a flush and two more steps, with
    outputs, pointers and checkpoint identical bit for bit to rssm_decode_step on a twin layer
    (the two calls differ only in where the tickets live)."""
    require_gpu()
    shape = synth.Shape(B=6, H=8, P=64, N=128, G=2, L=4, in_dtype="bf16", seed=92)
    gen = synth.make_generator(shape.seed)
    S0 = synth.initial_state(shape, gen)
    ref = ReplaySSM(layer_shape(shape, "e4m3"), dev(S0))
    alt = ReplaySSM(layer_shape(shape, "e4m3"), dev(S0))
    assert alt.decode_kernel() == "warp_per_head"
    for t in range(shape.L + 2):
        a, v, k, q = (dev(x) for x in synth.decode_step_inputs(shape, gen))
        o_ref = ref.decode_step(a, v, k, q)
        o_alt = alt.decode_step_static_scratch(a, v, k, q)
        assert torch.equal(o_alt, o_ref), f"step {t}"
        s_ref, c_ref, e_ref = ref.read_pointers()
        s_alt, c_alt, e_alt = alt.read_pointers()
        assert e_ref == 0 and e_alt == 0
        assert torch.equal(s_ref, s_alt) and torch.equal(c_ref, c_alt), f"step {t}: pointers differ"
    assert torch.equal(alt.ckpt, ref.ckpt)

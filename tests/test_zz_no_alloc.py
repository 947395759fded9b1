"""The decode step that allocates nothing (rssm_decode_step_static_scratch).

This is for callers that cannot give the library more device memory while
decoding runs: a fixed arena planned at start-up, an allocator owned by
another component, a stream under capture. The variant keeps the kernel's
per-sequence ticket counters in a static device array of the library. This
test calls it through the C ABI and checks it against rssm_decode_step on the
same state and inputs, for two calls in a row. The second call is a flush step,
so both kernel paths run. The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from hybrid_model_ssm_gb300 import ReplaySSM, lib
from hybrid_model_ssm_gb300.rssm import RSSM_OK
from tests.gpu_helpers import REL_TOL, dev, layer_shape, require_gpu, slice_rel_err

pytestmark = pytest.mark.gpu


def test_static_scratch_decode_matches_decode_step():
    require_gpu()
    shape = synth.Shape(B=5, H=8, P=64, N=128, G=2, L=2, seed=90)
    gen = synth.make_generator(shape.seed)
    S0 = synth.initial_state(shape, gen)
    ref = ReplaySSM(layer_shape(shape), dev(S0))
    alt = ReplaySSM(layer_shape(shape), dev(S0))
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        a, v, k, q = (dev(x) for x in synth.decode_step_inputs(shape, gen))
        o_ref = ref.decode_step(a, v, k, q)
        o_alt = torch.full_like(o_ref, float("nan"))
        status = lib().rssm_decode_step_static_scratch(alt._h, a.data_ptr(), v.data_ptr(), k.data_ptr(),
                                                       q.data_ptr(), o_alt.data_ptr(), ctypes.c_void_p(stream))
        assert status == RSSM_OK, lib().rssm_last_error().decode()
        assert slice_rel_err(o_alt.cpu(), o_ref.cpu().double().numpy(), 1) <= REL_TOL, f"call {call}"
        s_ref, c_ref, e_ref = ref.read_pointers()
        s_alt, c_alt, e_alt = alt.read_pointers()
        assert e_ref == 0 and e_alt == 0
        assert torch.equal(s_ref, s_alt) and torch.equal(c_ref, c_alt), f"call {call}: pointers differ"
        assert slice_rel_err(alt.ckpt.cpu(), ref.ckpt.cpu().double().numpy(), 2) <= REL_TOL
    assert np.array_equal(c_alt.numpy(), np.zeros(shape.B, np.int32))  # the second call flushed

"""Error paths: host-side argument checks and device-side per-sequence errors.

Device errors never trap. A sequence whose request would overflow its ring,
or that commits an accepted length outside 0..T, is skipped. A bit is set
in the error word. The other sequences proceed, and the context stays usable.
"""
import numpy as np
import pytest
import torch

import synth
from hybrid_model_ssm_gb300 import ReplaySSM, RssmError
from hybrid_model_ssm_gb300.rssm import ERR_ACCEPT, ERR_CAPACITY, RSSM_ECAPACITY, RSSM_EINVAL
from tests.gpu_helpers import dev, layer_shape, require_gpu

pytestmark = pytest.mark.gpu

S = synth.Shape


def _model(shape):
    gen = synth.make_generator(shape.seed)
    return ReplaySSM(layer_shape(shape), dev(synth.initial_state(shape, gen))), gen


def test_host_argument_errors():
    require_gpu()
    shape = S(B=2, H=4, P=16, N=32, G=2, L=4, T_max=2, seed=40)
    model, gen = _model(shape)
    a, v, k, q = (dev(x) for x in synth.decode_step_inputs(shape, gen))
    with pytest.raises(ValueError):
        model.decode_step(a, v, k[:, :1], q)  # wrong shape, caught by the binding
    # misaligned pointer: caught by the C ABI
    raw = torch.empty(a.numel() + 1, device="cuda")
    bad = raw[1:].view_as(a)
    bad.copy_(a)
    with pytest.raises(RssmError) as ei:
        model.decode_step(bad, v, k, q)
    assert ei.value.status == RSSM_EINVAL
    with pytest.raises(RssmError) as ei:  # commit without a pending verify
        model.commit(torch.zeros(2, dtype=torch.int32, device="cuda"))
    assert ei.value.status == RSSM_EINVAL
    with pytest.raises(RssmError):
        model.flush(0)
    va, vv, vk, vq = (dev(x) for x in synth.verify_round_inputs(shape, 3, gen))
    with pytest.raises(RssmError):  # T = 3 > T_max = 2
        model.verify(va, vv, vk, vq)
    # the handle still works afterwards
    model.decode_step(a, v, k, q)
    assert model.read_pointers()[2] == 0


def test_bad_accepted_length_sets_error_and_skips_sequence():
    require_gpu()
    shape = S(B=3, H=4, P=16, N=32, G=2, L=4, T_max=3, seed=41)
    model, gen = _model(shape)
    a, v, k, q = (dev(x) for x in synth.verify_round_inputs(shape, 2, gen))
    model.verify(a, v, k, q)
    model.commit(torch.tensor([1, 3, -1], dtype=torch.int32, device="cuda"))  # 3 > T = 2, -1 < 0
    start, count, err = model.read_pointers(check=False)
    assert err & ERR_ACCEPT
    assert count.tolist() == [1, 0, 0]
    with pytest.raises(RssmError) as ei:
        model.read_pointers()
    assert ei.value.status == RSSM_ECAPACITY
    model.clear_error()
    assert model.read_pointers()[2] == 0


def test_ring_overflow_sets_error_and_leaves_sequence_untouched():
    """Commit without flushing until the ring is full, then decode: the full
    sequence is skipped (no output, no state change), the other one proceeds."""
    require_gpu()
    shape = S(B=2, H=4, P=16, N=32, G=2, L=4, T_max=3, seed=42)  # R = 6
    model, gen = _model(shape)
    for acc in ([3, 1], [3, 1]):
        a, v, k, q = (dev(x) for x in synth.verify_round_inputs(shape, 3, gen))
        model.verify(a, v, k, q)
        model.commit(torch.tensor(acc, dtype=torch.int32, device="cuda"))
    start, count, err = model.read_pointers()
    assert count.tolist() == [6, 2] and err == 0
    ck = model.ckpt.clone()
    a, v, k, q = (dev(x) for x in synth.decode_step_inputs(shape, gen))
    o = torch.full((2, 4, 16), 7.0, device="cuda")
    model.decode_step(a, v, k, q, out=o)
    start2, count2, err2 = model.read_pointers(check=False)
    assert err2 & ERR_CAPACITY
    assert count2.tolist() == [6, 3]
    assert torch.all(o[0] == 7.0)  # skipped sequence: output untouched
    assert not torch.all(o[1] == 7.0)
    assert torch.equal(model.ckpt[0], ck[0])
    # verify beyond capacity is refused the same way
    model.clear_error()
    a, v, k, q = (dev(x) for x in synth.verify_round_inputs(shape, 3, gen))
    model.verify(a, v, k, q)
    assert model.read_pointers(check=False)[2] & ERR_CAPACITY
    # a forced flush recovers the full sequence
    model.clear_error()
    model.commit(torch.zeros(2, dtype=torch.int32, device="cuda"))
    model.flush(1)
    start3, count3, err3 = model.read_pointers()
    assert count3.tolist() == [0, 0] and err3 == 0
    assert start3.tolist() == [6 % 6, 3]


def test_bounded_wait_expires_and_reports():
    """A wait that nothing completes gives up after its limit, sets the timeout
    bit in the error word and returns; the context keeps working afterwards."""
    import ctypes
    import time

    from hybrid_model_ssm_gb300 import lib
    from hybrid_model_ssm_gb300.rssm import ERR_TIMEOUT, RSSM_OK

    require_gpu()
    word = torch.zeros(4, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    st = lib().rssm_selftest_bounded_wait(word.data_ptr(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == RSSM_OK
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(word[0]) & ERR_TIMEOUT
    assert 0.5 < elapsed < 10.0
    shape = S(B=2, H=4, P=16, N=32, G=2, L=4, seed=43)
    model, gen = _model(shape)
    a, v, k, q = (dev(x) for x in synth.decode_step_inputs(shape, gen))
    model.decode_step(a, v, k, q)
    assert model.read_pointers()[2] == 0



def test_clear_error_resets_part_counted_tickets():
    """A launch that gives up on a wait leaves its sequences' tickets part-counted.
    The host plants that state (nonzero tickets and the timeout bit) in the pointer
    block; after rssm_clear_error the next decode steps must advance the pointers
    exactly as the oracle's bookkeeping does."""
    require_gpu()
    from hybrid_model_ssm_gb300.rssm import ERR_TIMEOUT
    from tests.gpu_helpers import PointerShadow, check_pointers

    shape = S(B=5, H=6, P=16, N=32, G=2, L=3, seed=44)
    model, gen = _model(shape)
    shadow = PointerShadow(shape.B, shape.L, shape.R)
    nb = -(-shape.B * 4 // 256) * 256  # each pointer-block array is 256-byte aligned
    tickets = model.ptrs[2 * nb: 2 * nb + 4 * shape.B].view(torch.int32)
    err = model.ptrs[3 * nb: 3 * nb + 4].view(torch.int32)
    tickets.copy_(torch.tensor([3, 0, 5, 1, 2], dtype=torch.int32, device="cuda"))
    err.fill_(ERR_TIMEOUT)
    model.clear_error()
    torch.cuda.synchronize()
    assert torch.count_nonzero(tickets).item() == 0 and int(err.item()) == 0
    for _ in range(2 * shape.L + 1):
        a, v, k, q = (dev(x) for x in synth.decode_step_inputs(shape, gen))
        model.decode_step(a, v, k, q)
        shadow.decode()
        check_pointers(model, shadow)
    assert torch.count_nonzero(tickets).item() == 0

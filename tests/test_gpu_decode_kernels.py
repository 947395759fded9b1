"""GPU parity of the two decode kernels of small head tiles.

With an E4M3 or E2M1 read copy, or an FP16 checkpoint, a decode step runs a
warp-per-head kernel for the non-flush sequences and then the head kernel for
the flushing ones (which also advances every pointer); the head kernel alone
is the other choice. Sequences are staggered (a verify and a commit of random
accepted lengths) so that single steps mix flushing and non-flushing
sequences.

Bit-exact between the two choices: pointers, checkpoints, read copies and the
live ring records (the appends are raw copies of the inputs, and the fold is
the same kernel). Outputs agree to 1e-5 per (sequence, head) (FP32 summation
order). Against the oracle (read copies): each non-flush output equals the
oracle's output-only form on the device copy and the buffered records, and
each flush output the exact recurrence, both within 1e-4.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from hybrid_model_ssm_gb300 import ReplaySSM, RssmError
from hybrid_model_ssm_gb300.rssm import RSSM_EUNSUPPORTED
from tests.gpu_helpers import REL_TOL, dev, f64, layer_shape, require_gpu, slice_rel_err
from tests.test_gpu_readcopy import _dequantized_copy

pytestmark = pytest.mark.gpu

S = synth.Shape
# (format, N, input dtype, P): tiles from 0.5 KiB (E4M3 P=8 N=64) to 16 KiB (FP16), and head
# dimensions that are no power of two (a row pass over 24 or 120 rows, one ragged
# group of chunk rows, value rows of 48 or 240 bytes)
CASES = [("e4m3", 64, "bf16", 32), ("e4m3", 128, "f32", 32), ("e4m3", 128, "bf16", 64), ("e2m1", 64, "f32", 32),
         ("e2m1", 128, "bf16", 64), ("e2m1", 128, "bf16", 128), ("f16_sr", 128, "bf16", 32), ("f16_rn", 64, "f32", 32),
         ("e4m3", 64, "f32", 8), ("e4m3", 128, "bf16", 24), ("e2m1", 64, "bf16", 120), ("e2m1", 128, "f32", 40),
         ("f16_rn", 64, "bf16", 24)]


def _model(shape, fmt, S0, kernel):
    if fmt.startswith("f16"):
        ls = dataclasses.replace(layer_shape(shape), ckpt=fmt, seed=77)
        m = ReplaySSM(ls, dev(S0.to(torch.float16)))
    else:
        m = ReplaySSM(layer_shape(shape, fmt), dev(S0))
    m.set_decode_kernel(kernel)
    return m


def _live_ring(model, shape):
    """The committed records of every sequence: (alpha [H], v [H,P], k [G,N]) per (b, j), raw bytes."""
    a, V, K = model.ring_views()
    start, count, _ = model.read_pointers()
    out = []
    for b in range(shape.B):
        for j in range(int(count[b])):
            s = (int(start[b]) + j) % shape.R
            out.append((a[b, :, s].cpu().view(torch.int32), V[b, :, s].cpu().contiguous().view(torch.uint8),
                        K[b, :, s].cpu().contiguous().view(torch.uint8)))
    return out


def _assert_same_state(m1, m2, shape, where):
    s1, c1, e1 = m1.read_pointers()
    s2, c2, e2 = m2.read_pointers()
    assert e1 == 0 and e2 == 0, f"{where}: error word {e1} / {e2}"
    assert torch.equal(s1, s2) and torch.equal(c1, c2), f"{where}: pointers differ"
    assert torch.equal(m1.ckpt.view(torch.uint8), m2.ckpt.view(torch.uint8)), f"{where}: checkpoints differ"
    if m1.copy is not None:
        assert torch.equal(m1.copy, m2.copy), f"{where}: read copies differ"
    for i, (x, y) in enumerate(zip(_live_ring(m1, shape), _live_ring(m2, shape))):
        for part, name in zip(range(3), ("decays", "values", "keys")):
            assert torch.equal(x[part], y[part]), f"{where}: live record {i}: {name} differ"


def test_kernel_choice_and_refusal():
    require_gpu()
    shape = S(B=2, H=4, P=16, N=64, G=2, L=4, seed=90)
    S0 = synth.initial_state(shape, synth.make_generator(shape.seed))
    m = ReplaySSM(layer_shape(shape, "e4m3"), dev(S0))
    assert m.decode_kernel() == "warp_per_head"
    m.set_decode_kernel("head_kernel")
    assert m.decode_kernel() == "head_kernel"
    m.set_decode_kernel("auto")
    assert m.decode_kernel() == "warp_per_head"
    f16 = _model(shape, "f16_sr", S0, "auto")
    assert f16.decode_kernel() == "head_kernel"  # automatic: FP16 checkpoints keep the head kernel
    f16.set_decode_kernel("warp_per_head")
    assert f16.decode_kernel() == "warp_per_head"
    plain = ReplaySSM(layer_shape(shape), dev(S0))
    assert plain.decode_kernel() == "head_kernel"
    with pytest.raises(RssmError) as ei:
        plain.set_decode_kernel("warp_per_head")
    assert ei.value.status == RSSM_EUNSUPPORTED
    assert plain.decode_kernel() == "head_kernel"


@pytest.mark.parametrize("fmt,N,in_dtype,P", CASES)
def test_staggered_steps_agree(fmt, N, in_dtype, P):
    require_gpu()
    shape = S(B=5, H=8, P=P, N=N, G=2, L=6, T_max=3, in_dtype=in_dtype, seed=91)
    gen = synth.make_generator(shape.seed)
    S0 = synth.initial_state(shape, gen)
    mh = _model(shape, fmt, S0, "head_kernel")
    mw = _model(shape, fmt, S0, "warp_per_head")
    assert mh.decode_kernel() == "head_kernel" and mw.decode_kernel() == "warp_per_head"
    rc = not fmt.startswith("f16")
    orc = oracle.ReplayOracle(f64(S0), L=shape.L, R=shape.R, G=shape.G) if rc else None
    mixed = 0
    for rnd in range(3):
        # stagger: a verify of T = 3 drafts and a commit of random accepted lengths
        a, v, k, q = synth.verify_round_inputs(shape, 3, gen)
        acc = synth.accepted_lengths(shape.B, 3, gen)
        start, count, _ = mw.read_pointers()
        if np.any(count.numpy() + 3 > shape.R):  # flush first where the drafts would not fit
            for m in (mh, mw):
                m.flush(1)
            if orc is not None:
                orc.flush(1)
        for m in (mh, mw):  # then fold the sequences that now hold L or more records
            m.verify(dev(a), dev(v), dev(k), dev(q))
            m.commit(dev(acc))
            m.flush(shape.L)
        if orc is not None:
            orc.verify(f64(a), f64(v), f64(k), f64(q))
            orc.commit(acc.numpy())
            orc.flush(shape.L)
        _assert_same_state(mh, mw, shape, f"round {rnd} after commit")
        for t in range(shape.L + 1):
            a, v, k, q = synth.decode_step_inputs(shape, gen)
            torch.cuda.synchronize()
            copy_vals = _dequantized_copy(mw.copy, shape, fmt) if rc else None
            recs_before = [list(r) for r in orc.records] if rc else None
            oh = mh.decode_step(dev(a), dev(v), dev(k), dev(q)).cpu().numpy().astype(np.float64)
            ow = mw.decode_step(dev(a), dev(v), dev(k), dev(q)).cpu().numpy().astype(np.float64)
            where = f"round {rnd} step {t}"
            assert slice_rel_err(ow, oh, 1) <= 1e-5, f"{where}: the two kernels' outputs differ"
            _assert_same_state(mh, mw, shape, where)
            if orc is None:
                continue
            o_ref, flushed = orc.decode(f64(a), f64(v), f64(k), f64(q))
            mixed += int(flushed.any() and not flushed.all())
            for b in range(shape.B):
                if flushed[b]:
                    assert slice_rel_err(ow[b], o_ref[b], 1) <= REL_TOL, f"{where} seq {b}: flush output"
                    continue
                alphas = np.stack([r[0] for r in recs_before[b]] + [f64(a)[b]])
                vs = np.stack([r[1] for r in recs_before[b]] + [f64(v)[b]])
                ks = np.stack([r[2] for r in recs_before[b]] + [f64(k)[b]])
                o_copy = oracle.replay_output(copy_vals[b], alphas, vs, ks, f64(q)[b])
                assert slice_rel_err(ow[b], o_copy, 1) <= REL_TOL, f"{where} seq {b}: non-flush output"
    if orc is not None:
        assert mixed > 0, "no step mixed flushing and non-flushing sequences"


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1", "f16_rn"])
@pytest.mark.parametrize("qscale", [2.0 ** -100, 2.0 ** -60, 1.0, 2.0 ** 40, 2.0 ** 100, "spread"])
def test_query_scales(fmt, qscale):
    """bf16 queries from 2^-100 to 2^100: the warp-per-head step scales each group's query by a power
    of two before its binary16 tile dot and back after, so its outputs agree with the head
    kernel's FP32 dot (1e-5) and, for read copies, with the oracle's read-copy output (1e-4)."""
    require_gpu()
    shape = S(B=2, H=4, P=16, N=128, G=2, L=4, seed=92)
    gen = synth.make_generator(shape.seed)
    S0 = synth.initial_state(shape, gen)
    mh = _model(shape, fmt, S0, "head_kernel")
    mw = _model(shape, fmt, S0, "warp_per_head")
    rc = not fmt.startswith("f16")
    orc = oracle.ReplayOracle(f64(S0), L=shape.L, R=shape.R, G=shape.G) if rc else None
    for t in range(shape.L - 1):  # non-flush steps only
        a, v, k, q = synth.decode_step_inputs(shape, gen)
        if qscale == "spread":  # elements from 2^-20 to 2^20 of each other in every group
            mag = 2.0 ** torch.linspace(-20, 20, shape.N)
            q = (q.float() * mag).to(q.dtype)
        else:
            q = (q.float() * qscale).to(q.dtype)
        torch.cuda.synchronize()
        copy_vals = _dequantized_copy(mw.copy, shape, fmt) if rc else None
        recs_before = [list(r) for r in orc.records] if rc else None
        oh = mh.decode_step(dev(a), dev(v), dev(k), dev(q)).cpu().numpy().astype(np.float64)
        ow = mw.decode_step(dev(a), dev(v), dev(k), dev(q)).cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(ow))
        assert slice_rel_err(ow, oh, 1) <= 1e-5, f"step {t}: the two kernels' outputs differ"
        _assert_same_state(mh, mw, shape, f"step {t}")
        if orc is None:
            continue
        o_ref, flushed = orc.decode(f64(a), f64(v), f64(k), f64(q))
        assert not flushed.any()
        for b in range(shape.B):
            alphas = np.stack([r[0] for r in recs_before[b]] + [f64(a)[b]])
            vs = np.stack([r[1] for r in recs_before[b]] + [f64(v)[b]])
            ks = np.stack([r[2] for r in recs_before[b]] + [f64(k)[b]])
            o_copy = oracle.replay_output(copy_vals[b], alphas, vs, ks, f64(q)[b])
            assert slice_rel_err(ow[b], o_copy, 1) <= REL_TOL, f"step {t} seq {b}"


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
def test_read_copy_step_replayed_from_a_cuda_graph(fmt):
    """A read-copy decode step (the warp-per-head kernel, then the head kernel) captured once
    in a CUDA graph and replayed across flush boundaries: every output against the oracle's
    read-copy form on the device copy (non-flush) or the exact recurrence (flush)."""
    require_gpu()
    shape = S(B=3, H=8, P=32, N=128, G=2, L=6, seed=93)
    gen = synth.make_generator(shape.seed)
    S0 = synth.initial_state(shape, gen)
    model = ReplaySSM(layer_shape(shape, fmt), dev(S0))
    assert model.decode_kernel() == "warp_per_head"
    orc = oracle.ReplayOracle(f64(S0), L=shape.L, R=shape.R, G=shape.G)
    buf = tuple(dev(x) for x in synth.decode_step_inputs(shape, synth.make_generator(0)))
    out = torch.empty((shape.B, shape.H, shape.P), device="cuda")
    graph, flushes = None, 0
    for t in range(4 * shape.L):
        a, v, k, q = synth.decode_step_inputs(shape, gen)
        for d, h in zip(buf, (a, v, k, q)):
            d.copy_(h)
        torch.cuda.synchronize()
        copy_vals = _dequantized_copy(model.copy, shape, fmt)
        recs_before = [list(r) for r in orc.records]
        if t < shape.L + 2:
            model.decode_step(*buf, out=out)
        else:
            if graph is None:
                graph = torch.cuda.CUDAGraph()
                side = torch.cuda.Stream()
                side.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(side):
                    with torch.cuda.graph(graph, stream=side):  # records the launches only
                        model.decode_step(*buf, out=out)
                torch.cuda.current_stream().wait_stream(side)
            graph.replay()
        o = out.cpu().numpy().astype(np.float64)
        o_ref, flushed = orc.decode(f64(a), f64(v), f64(k), f64(q))
        flushes += int(flushed.any())
        for b in range(shape.B):
            if flushed[b]:
                assert slice_rel_err(o[b], o_ref[b], 1) <= REL_TOL, f"step {t} seq {b}: flush output"
                continue
            alphas = np.stack([r[0] for r in recs_before[b]] + [f64(a)[b]])
            vs = np.stack([r[1] for r in recs_before[b]] + [f64(v)[b]])
            ks = np.stack([r[2] for r in recs_before[b]] + [f64(k)[b]])
            o_copy = oracle.replay_output(copy_vals[b], alphas, vs, ks, f64(q)[b])
            assert slice_rel_err(o[b], o_copy, 1) <= REL_TOL, f"step {t} seq {b}: non-flush output"
    assert flushes == 4
    start, count, err = model.read_pointers()
    assert err == 0
    assert np.array_equal(start.numpy(), orc.start) and np.array_equal(count.numpy(), orc.count)

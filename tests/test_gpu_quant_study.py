"""Quantized reads over a long decode: output error against the exact recurrence, step by step.

Workload: B=64, H=32, P=64, N=128, G=2, L=16, bf16 inputs, 8192 decode steps
from an N(0, 0.1^2) state, with the mandated decays (u ~ N(0, 1)) and with a
long-memory variant (u ~ N(-4, 1), decays near 0.98). Every arm sees the same
inputs:

* replay with FP32 reads (no copy), on the GPU;
* replay with the E4M3 row-scaled read copy, on the GPU;
* replay with the E2M1 block-scaled read copy, on the GPU;
* fully quantized states (E4M3, E2M1) in the oracle: the state itself is
  stored quantized and fed back every step, so rounding re-enters the
  recurrence (the failure mode that keeping the recurrence in FP32 avoids:
  ReplaySSM pages, quantization sections).

The exact reference is the float64 oracle on sequence 0 (all heads); the fully
quantized arms run on two heads of it. Checks:

* the FP32 arm stays within 1e-4 of the exact output at every step;
* the read-copy arms stay within the per-format bound at every non-flush step
  (the bound of test_gpu_readcopy, from the device checkpoint of the last
  flush) and within 1e-4 at flush steps, so their error cannot grow with the
  step count;
* with long memory, the fully quantized arms end with a larger error than the
  read-copy arms.

The error-vs-step table (per-step normwise relative error, mean and max over
windows of steps) is printed; run with ``-s`` to see it.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import quant
from hybrid_model_ssm_gb300 import ReplaySSM
from tests.gpu_helpers import REL_TOL, dev, f64, layer_shape, require_gpu, slice_rel_err

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

STEPS = 8192
WINDOWS = [(1, 16), (17, 256), (257, 1024), (1025, 4096), (4097, 8192)]
FQ_HEADS = 2  # heads 0..1 of sequence 0, both in group 0


def _window_table(errs: dict) -> str:
    lines = ["arm".ljust(12) + "".join(f"steps {a}-{b}".rjust(24) for a, b in WINDOWS)]
    for arm, e in errs.items():
        e = np.asarray(e)
        cells = []
        for a, b in WINDOWS:
            w = e[a - 1: b]
            cells.append(f"{w.mean():.2e} / {w.max():.2e}".rjust(24))
        lines.append(arm.ljust(12) + "".join(cells))
    return "\n".join(lines)


@pytest.mark.parametrize("variant,mu", [("mandated", 0.0), ("long_memory", -4.0)])
def test_error_vs_step(variant, mu):
    require_gpu()
    shape = synth.PRESETS["quant_b64_h32_l16"]
    gen = synth.make_generator(shape.seed)
    S0 = synth.initial_state(shape, gen)
    models = {fmt: ReplaySSM(layer_shape(shape, fmt), dev(S0)) for fmt in (None, "e4m3", "e2m1")}
    exact = f64(S0[:1])  # [1, H, P, N]
    fq = {fmt: quant.FullyQuantizedState(exact[:, :FQ_HEADS], fmt) for fmt in ("e4m3", "e2m1")}
    g = oracle.head_groups(shape.H, shape.G)
    # per-element bounds of each copy, from the fp32 checkpoint it was made from (sequence 0)
    ebound = {fmt: quant.element_error_bound(fmt, S0[0].numpy()) for fmt in ("e4m3", "e2m1")}  # [H, P, N]
    gam = np.ones(shape.H)  # decays since the last flush, sequence 0
    names = {None: "fp32 replay", "e4m3": "e4m3 read", "e2m1": "e2m1 read"}
    errs = {k: [] for k in ["fp32 replay", "e4m3 read", "e2m1 read", "e4m3 full-q", "e2m1 full-q"]}
    ratio = {"e4m3": 0.0, "e2m1": 0.0}
    for t in range(STEPS):
        a, v, k, q = synth.decode_step_inputs(shape, gen, mu)
        da, dv, dk, dq = dev(a), dev(v), dev(k), dev(q)
        outs = {fmt: m.decode_step(da, dv, dk, dq)[0].cpu().numpy().astype(np.float64) for fmt, m in models.items()}
        a0, v0, k0, q0 = f64(a[:1]), f64(v[:1]), f64(k[:1]), f64(q[:1])
        exact, o_ref = oracle.conventional_step(exact, a0, v0, k0, q0)
        o_ref = o_ref[0]  # [H, P]
        flush = (t + 1) % shape.L == 0
        gam = gam * a0[0]
        for fmt, o in outs.items():
            e = slice_rel_err(o, o_ref, 1)
            errs[names[fmt]].append(e)
            if fmt is None or flush:
                assert e <= REL_TOL, f"{variant} step {t}: {names[fmt]} rel err {e:.3g}"
                continue
            qg = np.abs(q0[0][g])  # [H, N]
            bound = gam[:, None] * np.einsum("hpn,hn->hp", ebound[fmt], qg)
            slack = 1e-5 * np.abs(o_ref).max(axis=-1, keepdims=True)
            err = np.abs(o - o_ref)
            assert np.all(err <= 1.05 * bound + slack), f"{variant} step {t}: {fmt} read above its bound"
            ratio[fmt] = max(ratio[fmt], float((err / (bound + slack)).max()))
        for fmt, st in fq.items():
            o_fq = st.step(a0[:, :FQ_HEADS], v0[:, :FQ_HEADS], k0[:, :1], q0[:, :1])[0]
            errs[f"{fmt} full-q"].append(slice_rel_err(o_fq, o_ref[:FQ_HEADS], 1))
        if flush:
            gam = np.ones(shape.H)
            ebound = {fmt: quant.element_error_bound(fmt, models[fmt].ckpt[0].cpu().numpy()) for fmt in ("e4m3", "e2m1")}
    for fmt, m in models.items():
        assert m.read_pointers()[2] == 0
    print(f"\nquantized reads, {variant} decays (B=64 H=32 P=64 N=128 L=16, {STEPS} steps); "
          f"per-step max-over-heads normwise rel error, mean / max per window")
    print(_window_table(errs))
    print("largest error / bound over all non-flush steps: " + ", ".join(f"{k} {v:.3f}" for k, v in ratio.items()))
    if variant == "long_memory":
        for fmt in ("e4m3", "e2m1"):
            read_last = np.mean(errs[f"{fmt} read"][-1024:])
            fq_last = np.mean(errs[f"{fmt} full-q"][-1024:])
            assert fq_last > 2.0 * read_last, f"{fmt}: fully quantized {fq_last:.3g} vs read copy {read_last:.3g}"

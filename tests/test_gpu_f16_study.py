"""FP16 recurrent checkpoint over a long decode: error against the exact recurrence, step by step.

Workload: B=64, H=32, P=64, N=128, G=2, L=16, bf16 inputs, 8192 decode steps,
with the mandated decays (u ~ N(0, 1)) and a long-memory variant (u ~ N(-4, 1)).
Three GPU arms see the same inputs: replay with the FP32 checkpoint, and with an
FP16 checkpoint stored with stochastic rounding or with rounding to nearest.
The reference is the float64 conventional recurrence on sequence 0 from the
FP32 initial state (the FP16 arms start from its binary16 rounding). The FP32
arm must stay within 1e-4 at every step; the FP16 arms' error must not grow
(the last 1024 steps' mean within 4x of steps 17-256). The error-vs-step table
is printed (run with ``-s``).
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from hybrid_model_ssm_gb300 import ReplaySSM
from tests.gpu_helpers import REL_TOL, dev, f64, layer_shape, require_gpu, slice_rel_err

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

STEPS = 8192
WINDOWS = [(1, 16), (17, 256), (257, 1024), (1025, 4096), (4097, 8192)]


@pytest.mark.parametrize("variant,mu", [("mandated", 0.0), ("long_memory", -4.0)])
def test_f16_checkpoint_error_vs_step(variant, mu):
    require_gpu()
    shape = synth.PRESETS["quant_b64_h32_l16"]
    gen = synth.make_generator(shape.seed)
    S0 = synth.initial_state(shape, gen)
    base = layer_shape(shape)
    models = {"fp32": ReplaySSM(base, dev(S0))}
    for m in ("f16_sr", "f16_rn"):
        models[m] = ReplaySSM(dataclasses.replace(base, ckpt=m, seed=4242), dev(S0.to(torch.float16)))
    exact = f64(S0[:1])
    errs = {k: [] for k in models}
    for t in range(STEPS):
        a, v, k, q = synth.decode_step_inputs(shape, gen, mu)
        da, dv, dk, dq = dev(a), dev(v), dev(k), dev(q)
        outs = {m: md.decode_step(da, dv, dk, dq)[0].cpu().numpy() for m, md in models.items()}
        exact, o_ref = oracle.conventional_step(exact, f64(a[:1]), f64(v[:1]), f64(k[:1]), f64(q[:1]))
        for m, o in outs.items():
            e = slice_rel_err(o, o_ref[0], 1)
            errs[m].append(e)
            if m == "fp32":
                assert e <= REL_TOL, f"{variant} step {t}: fp32 rel err {e:.3g}"
    for md in models.values():
        assert md.read_pointers()[2] == 0
    lines = ["arm".ljust(8) + "".join(f"steps {a}-{b}".rjust(24) for a, b in WINDOWS)]
    for m, e in errs.items():
        e = np.asarray(e)
        lines.append(m.ljust(8) + "".join(f"{e[a - 1:b].mean():.2e} / {e[a - 1:b].max():.2e}".rjust(24)
                                          for a, b in WINDOWS))
    print(f"\nFP16 checkpoint, {variant} decays (B=64 H=32 P=64 N=128 L=16, {STEPS} steps); "
          "per-step max-over-heads normwise rel error, mean / max per window")
    print("\n".join(lines))
    for m in ("f16_sr", "f16_rn"):
        e = np.asarray(errs[m])
        assert e[-1024:].mean() <= 4 * e[16:256].mean(), f"{variant}: {m} error grows"

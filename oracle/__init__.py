"""Float64 CPU oracle for the ReplaySSM decode path.

TEST INFRASTRUCTURE ONLY. Nothing in the product package imports, calls or
links this package. Three places may use it: ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline arm of ``bench.py``. The oracle
and the CUDA path share no code. Both receive the same seeded inputs from the
separate ``synth`` package.

Sources. Citations give the page and its section:
  [RU] aikraft.ru, "ReplaySSM: Революция в декодировании гибридных моделей",
       sections 01-07 (01 = recurrence, 03 = unrolled window and flush,
       05 = rollback and output-only evaluation, 06 = split precision).
  [AR] sitech.ge, "NVIDIA و Dao AI Lab يقدّمان ReplaySSM لتسريع فك ترميز النماذج الهجينة",
       sections "كيف يعمل ReplaySSM" (how it works),
       "تقليل حركة الحالة وتبسيط rollback" (traffic and rollback),
       "الحد من خطأ التكميم" (quantization error).
  [ZH] ai.cheesepanini.fun, "知识卡片：ReplaySSM——重新思考混合模型解码的状态存储",
       section "方法/产品要点" (core representation, two step kinds,
       output-only evaluation formula).
Format definitions for the quantizers come from the OCP 8-bit floating point
specification (E4M3) and the OCP Microscaling specification (E2M1). The
stochastic rounding of the FP16 checkpoint draws from Philox4x32-10 (Salmon et
al., SC'11), written from its published definition.

Each function here is pinned by ``tests/test_oracle_pins.py``,
``tests/test_oracle_quant.py``, ``tests/test_oracle_sround.py`` and ``tests/test_oracle_delta.py`` to something other than itself: closed forms,
hand-computed golden cases, brute force, library conversions and
invariants. No function is left with unpinned parity.
"""
from .recurrence import (  # noqa: F401
    head_groups,
    to_f64,
    conventional_step,
    unrolled_state,
    replay_output,
    verify_outputs,
)
from .replay import ReplayOracle, CapacityError  # noqa: F401
from .quant import (  # noqa: F401
    E4M3_MAX,
    E2M1_MAX,
    e4m3_value,
    e2m1_value,
    e4m3_encode,
    e2m1_encode,
    quantize_rows_e4m3,
    dequantize_rows_e4m3,
    quantize_rows_e2m1,
    dequantize_rows_e2m1,
    element_error_bound,
    FullyQuantizedState,
)
from .sround import (  # noqa: F401
    philox4x32_10,
    sr_words,
    stochastic_round_f16,
    nearest_f16,
    f16_toward_zero,
    ReplayOracleF16,
)
from .delta import (  # noqa: F401
    delta_step,
    delta_pseudo_value,
    delta_replay_output,
    delta_fold,
    DeltaReplayOracle,
)

"""ReplaySSM decode path for GB300 (sm_103a): a C-ABI CUDA library plus a ctypes binding.

The kernels live in ``csrc/`` and are built into ``librssm.so`` by
``hybrid_model_ssm_gb300.build``. The public C interface is ``include/rssm.h``.
This package only marshals arguments. It has no CPU implementation of the path.
"""
from .rssm import (  # noqa: F401
    ConventionalVerifier,
    LayerShape,
    ReplaySSM,
    RssmError,
    conventional_step,
    launch_plan,
    read_copy_layout,
    round_f16,
    ring_offsets,
    workspace_size,
    lib,
    LIB_PATH,
)

"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This package draws random numbers and nothing else: it holds none of the
ReplaySSM arithmetic (no decays, no outer products, no outputs). Both the CUDA
path and the CPU oracle receive the tensors it produces.
"""
from .inputs import (  # noqa: F401
    Shape,
    PRESETS,
    make_generator,
    initial_state,
    decode_step_inputs,
    delta_step_inputs,
    delta_verify_round_inputs,
    verify_round_inputs,
    accepted_lengths,
)

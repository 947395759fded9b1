"""Helpers shared by the GPU parity tests.

Tolerances. The FP32 path must match the float64 oracle within a relative
error of 1e-4. The error is taken normwise per slice, because elementwise
relative error is undefined near zero: for every (sequence, head) the largest
absolute output error, divided by the largest absolute oracle output of that
slice. The same applies to the checkpoint, per (sequence, head) P x N matrix.
Integers (pointers, flush events, ring contents) must match bit for bit.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from hybrid_model_ssm_gb300 import LayerShape, ReplaySSM

REL_TOL = 1e-4


def require_gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")


def layer_shape(s: synth.Shape, read_fmt=None) -> LayerShape:
    return LayerShape(B=s.B, H=s.H, P=s.P, N=s.N, G=s.G, L=s.L, T_max=s.T_max, in_dtype=s.in_dtype,
                      read_fmt=read_fmt)


def slice_rel_err(got: np.ndarray, ref: np.ndarray, slice_dims: int) -> float:
    """max over slices of max|got-ref| / max|ref|; the last slice_dims axes form a slice."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    axes = tuple(range(ref.ndim - slice_dims, ref.ndim))
    num = np.abs(got - ref).max(axis=axes)
    den = np.maximum(np.abs(ref).max(axis=axes), 1e-30)
    return float((num / den).max())


def f64(x) -> np.ndarray:
    return oracle.to_f64(x)


def dev(x: torch.Tensor) -> torch.Tensor:
    return x.to("cuda", non_blocking=False).contiguous()


class PointerShadow:
    """Pointer bookkeeping of the oracle for every sequence (1 x 1 x 1 x 1 dummy state).

    The oracle's integer policy does not depend on the state's size, so a
    ReplayOracle on a 1-element state gives (start, count) for the whole batch.
    """

    def __init__(self, B: int, L: int, R: int):
        self.orc = oracle.ReplayOracle(np.zeros((B, 1, 1, 1)), L=L, R=R, G=1)
        self.B = B

    def decode(self):
        z = np.zeros
        return self.orc.decode(np.ones((self.B, 1)), z((self.B, 1, 1)), z((self.B, 1, 1)), z((self.B, 1, 1)))[1]

    def verify(self, T):
        z = np.zeros
        self.orc.verify(np.ones((self.B, T, 1)), z((self.B, T, 1, 1)), z((self.B, T, 1, 1)), z((self.B, T, 1, 1)))

    def commit(self, a):
        self.orc.commit(np.asarray(a))

    def flush(self, m):
        return self.orc.flush(m)

    @property
    def start(self):
        return self.orc.start

    @property
    def count(self):
        return self.orc.count


def check_pointers(model: ReplaySSM, shadow: PointerShadow):
    start, count, err = model.read_pointers()
    assert err == 0
    assert np.array_equal(start.numpy(), shadow.start), "start pointers differ"
    assert np.array_equal(count.numpy(), shadow.count), "count pointers differ"

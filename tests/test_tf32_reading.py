"""The numeric premise behind keeping the checkpoint contractions on FP32 FMAs.

The verify dots and the flush fold run on CUDA-core FP32 FMAs, not on TF32
tensor cores, because one TF32 product S q misses the 1e-4 normwise tolerance
of the FP32 path. A two-term split of the checkpoint (S = hi + lo, hi with its
low 13 mantissa bits cleared) meets it, because bf16 queries are exact in TF32.
This CPU model checks both statements: TF32 operands by truncation of the
mantissa to 10 bits (a conversion that rounds to nearest behaves the same
within a factor of two), products accumulated in fp32 over K-steps of 8, on
seeded tiles at the workload's scales. It tests no library code.
"""
import numpy as np


def _tf32(x):
    b = np.asarray(x, np.float32).view(np.uint32)
    return (b & np.uint32(0xFFFFE000)).view(np.float32)


def _bf16(x):
    b = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    b = b + 0x7FFF + ((b >> 16) & 1)
    return (b & 0xFFFF0000).astype(np.uint32).view(np.float32)


def _mma(A, B):
    acc = np.zeros((A.shape[0], B.shape[1]), np.float32)
    for k0 in range(0, A.shape[1], 8):
        part = (A[:, k0:k0 + 8].astype(np.float64) @ B[k0:k0 + 8].astype(np.float64)).astype(np.float32)
        acc = (acc + part).astype(np.float32)
    return acc


def _worst(fn, trials=40):
    rng = np.random.default_rng(0)
    worst = 0.0
    for _ in range(trials):
        S = (rng.standard_normal((64, 128)) * 0.1 * rng.uniform(0.2, 5)).astype(np.float32)
        q = _bf16(rng.standard_normal((128, 16)) / np.sqrt(128))
        ref = S.astype(np.float64) @ q.astype(np.float64)
        err = np.abs(fn(S, q) - ref).max(axis=0) / np.abs(ref).max(axis=0)
        worst = max(worst, float(err.max()))
    return worst


def test_bf16_queries_are_exact_in_tf32():
    q = _bf16(np.random.default_rng(1).standard_normal(4096))
    assert np.array_equal(_tf32(q), q)


def test_one_tf32_product_misses_the_tolerance():
    assert _worst(lambda S, q: _mma(_tf32(S), q)) > 1e-4


def test_split_checkpoint_meets_the_tolerance():
    def split(S, q):
        hi = _tf32(S)
        lo = _tf32(S - hi)
        return (_mma(hi, q) + _mma(lo, q)).astype(np.float32)
    assert _worst(split) < 1e-5

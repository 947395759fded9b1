"""Batch-level oracle for ReplaySSM decoding: exact state plus pointer bookkeeping.

TEST INFRASTRUCTURE ONLY (see the package docstring for who may use it).

The exact target is the conventional recurrence: replay decoding reaches the
same outputs up to floating point ([RU] §03, last paragraph; [AR] "كيف يعمل
ReplaySSM"; [ZH] 方法/产品要点). This class therefore advances the float64
state with ``conventional_step``. Next to it, it keeps the integers that a
replay implementation must reproduce bit for bit:

* ``start[b]``: ring slot of the first record not yet folded into the checkpoint;
* ``count[b]``: committed records in the ring;
* the flush events.

Policy (readings where the pages leave it open):

* decode: the step's record is appended. The step whose append brings the record
  count to L (or more) is a flush step. It folds all records into the
  checkpoint and clears the buffer ([RU] §03 item 2; [ZH] 两类步骤). The fold
  is eager: the flush step's own output uses the folded state.
* verify: T draft records are appended after the committed ones. The pointers
  do not move. Each draft's output uses the committed records plus the drafts
  up to and including itself ([RU] §05; [ZH] 方法/产品要点).
* commit(a): count += a, with 0 <= a <= T. Drafts past the pointer are
  ignored and are overwritten by the next appends. Nothing is snapshotted or
  restored ([RU] §05; [AR] traffic and rollback section).
* flush(min_count): every sequence with count >= min_count folds all of its
  records. Then start = (start + count) mod R and count = 0.

With a read copy (``read_fmt`` = "e4m3" or "e2m1"), the checkpoint is also
quantized at every flush (and at creation), from its fp32 rounding. Non-flush
decode outputs then use the dequantized copy in the output-only formula.
Verify outputs and flush-step outputs use the FP32 checkpoint.
The recurrence itself stays exact ([RU] §06; [AR] quantization section).
"""
from __future__ import annotations

import numpy as np

from .recurrence import conventional_step, head_groups, replay_output
from . import quant


class CapacityError(RuntimeError):
    """A request would hold more records than the ring has slots, or commit more than was drafted
    (no passage: the ring capacity R = L + T_max - 1 is this build's reading)."""


class ReplayOracle:
    """Exact float64 state of every (sequence, head) plus the window bookkeeping
    of replay decoding: start, count and the records since the last flush
    ([RU] §03 unrolled window; [ZH] 方法/产品要点, core representation), the
    checkpoint at each flush, and the read copy made from it ([RU] §06)."""

    def __init__(self, S0, L: int, R: int, G: int, read_fmt: str | None = None):
        S0 = np.asarray(S0, np.float64)
        self.B, self.H, self.P, self.N = S0.shape
        self.G, self.L, self.R = G, L, R
        if R < L or L < 1:
            raise ValueError("need R >= L >= 1")
        head_groups(self.H, G)
        self.S = S0.copy()  # exact state (conventional recurrence)
        self.ckpt = S0.copy()  # exact state as of each sequence's last flush
        self.start = np.zeros(self.B, np.int64)
        self.count = np.zeros(self.B, np.int64)
        self.flush_log: list[tuple[int, np.ndarray]] = []  # (event index, flushed sequences)
        self.events = 0
        # Records since each sequence's last flush (float64): alpha [H], v [H,P], k [G,N].
        self.records: list[list[tuple[np.ndarray, np.ndarray, np.ndarray]]] = [[] for _ in range(self.B)]
        self._drafts = None
        self.read_fmt = read_fmt
        self.copy = None  # dequantized read copy per sequence, float64 [B,H,P,N]
        if read_fmt is not None:
            self.copy = self._quantize(self.ckpt)

    # ---------------------------------------------------------------- helpers
    def _quantize(self, X):
        """Read copy of an exact state: round to fp32, quantize rows, dequantize ([RU] §06)."""
        X32 = np.asarray(X, np.float64).astype(np.float32)
        if self.read_fmt == "e4m3":
            codes, scale = quant.quantize_rows_e4m3(X32)
            return quant.dequantize_rows_e4m3(codes, scale)
        if self.read_fmt == "e2m1":
            codes, bcodes, rscale = quant.quantize_rows_e2m1(X32)
            return quant.dequantize_rows_e2m1(codes, bcodes, rscale)
        raise ValueError(self.read_fmt)

    def _fold(self, mask: np.ndarray, n_records: np.ndarray):
        """Flush the sequences in mask: checkpoint := exact state, pointers advance."""
        idx = np.nonzero(mask)[0]
        if len(idx) == 0:
            return idx
        self.ckpt[idx] = self.S[idx]
        self.start[idx] = (self.start[idx] + n_records[idx]) % self.R
        self.count[idx] = 0
        for b in idx:
            self.records[b] = []
        if self.read_fmt is not None:
            self.copy[idx] = self._quantize(self.S[idx])
        self.flush_log.append((self.events, idx.copy()))
        return idx

    # ------------------------------------------------------------------ steps
    def decode(self, alpha, v, k, q):
        """One decode step ([RU] §03: a non-flush step appends its record and
        outputs only; the step that fills the window folds and writes the
        checkpoint). Returns (o [B,H,P], flushed mask [B])."""
        h = self.count + 1
        if np.any(h > self.R):
            raise CapacityError("decode would exceed the ring capacity")
        S_prev_copy = self.copy
        self.S, o_exact = conventional_step(self.S, alpha, v, k, q)
        flush = h >= self.L
        o = o_exact
        if self.read_fmt is not None:
            o = o_exact.copy()
            for b in np.nonzero(~flush)[0]:
                recs = self.records[b] + [(alpha[b], v[b], k[b])]
                a_, v_, k_ = (np.stack(x) for x in zip(*recs))
                o[b] = replay_output(S_prev_copy[b], a_, v_, k_, q[b])
        for b in range(self.B):
            self.records[b].append((alpha[b].copy(), v[b].copy(), k[b].copy()))
        self.count = h
        self._fold(flush, h)
        self.events += 1
        self._drafts = None
        return o, flush

    def verify(self, alpha, v, k, q):
        """Speculative verify of T drafts: alpha [B,T,H], v [B,T,H,P], k,q [B,T,G,N].

        Output-only: the drafts run on a scratch copy of the exact state, so
        the real state and the pointers stay unchanged. Verify reads the FP32
        checkpoint even when a read copy exists (reading: the pages tie the
        copy to non-flush decode reads, [RU] §06). Returns O [B,T,H,P].
        """
        T = alpha.shape[1]
        if np.any(self.count + T > self.R):
            raise CapacityError("verify would exceed the ring capacity")
        O = np.empty((self.B, T, self.H, self.P))
        Sc = self.S.copy()
        for t in range(T):
            Sc, O[:, t] = conventional_step(Sc, alpha[:, t], v[:, t], k[:, t], q[:, t])
        self._drafts = (alpha.copy(), v.copy(), k.copy(), q.copy(), T)
        self.events += 1
        return O

    def commit(self, accepted):
        """Commit the first accepted[b] drafts of the last verify (count += a):
        rollback is a pointer move ([RU] §05; [AR] "تقليل حركة الحالة وتبسيط rollback")."""
        if self._drafts is None:
            raise CapacityError("commit without a preceding verify")
        alpha, v, k, q, T = self._drafts
        a = np.asarray(accepted, np.int64)
        if np.any(a < 0) or np.any(a > T):
            raise CapacityError("accepted length outside 0..T")
        for t in range(T):
            m = t < a
            if not np.any(m):
                continue
            S_m, _ = conventional_step(self.S[m], alpha[m, t], v[m, t], k[m, t], q[m, t])
            self.S[m] = S_m
            for b in np.nonzero(m)[0]:
                self.records[b].append((alpha[b, t].copy(), v[b, t].copy(), k[b, t].copy()))
        self.count = self.count + a
        self._drafts = None
        self.events += 1

    def flush(self, min_count: int):
        """Fold every sequence holding at least min_count (>= 1) records ([RU] §03
        flush; after a commit, this build's reading of where the flush goes).
        Returns the mask."""
        if min_count < 1:
            raise ValueError("min_count must be >= 1")
        mask = self.count >= min_count
        self._fold(mask, self.count.copy())
        self.events += 1
        return mask

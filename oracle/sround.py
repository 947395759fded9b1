"""FP16 checkpoint storage with stochastic rounding, and the counter-based generator it draws from.

TEST INFRASTRUCTURE ONLY (see the package docstring for who may use it).

The pages report that keeping the recurrent checkpoint in FP16 with stochastic
rounding stays close to FP32 ([RU] §06, last paragraph; [AR] "الحد من خطأ
التكميم": "FP16 or FP8 recurrence"). They define neither the rounding nor the
random numbers. Readings used by this build:

Generator: Philox4x32 with 10 rounds (Salmon, Moraes, Dror and Shaw, "Parallel
random numbers: as easy as 1, 2, 3", SC'11). State: a 128-bit counter
(c0, c1, c2, c3) and a 64-bit key (k0, k1). One round takes the full 64-bit
products c0 * 0xD2511F53 = (hi0, lo0) and c2 * 0xCD9E8D57 = (hi1, lo1) and sets
    (c0, c1, c2, c3) <- (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0);
between rounds the key advances by the Weyl increments (0x9E3779B9, 0xBB67AE85).
The four output words are the counter after ten rounds.

Counters: element group g = flat index into [B,H,P,N] // 4 (four consecutive
elements along N share one call, word e for element 4 g + e);
counter = (g mod 2^32, g div 2^32, epoch, 0) with epoch the sequence's number of
earlier flushes; key = (seed mod 2^32, seed div 2^32).

Stochastic rounding of a binary32 value x to binary16 with a 32-bit word r:
    NaN stays NaN; |x| >= 65504 gives +-65504 (saturation);
    lo = x rounded toward zero to binary16, hi = the next binary16 away from zero;
    frac = (|x| - |lo|) / (|hi| - |lo|), exact in binary32 (the difference is
           exact because |lo| <= |x| < 2|lo| or lo = 0, and the divisor is a
           power of two);
    t = floor(frac * 2^32), exact whenever frac has no bits below 2^-32;
    result = hi if r < t else lo, with the sign of x.
So P(result = hi) = t / 2^32 = frac: the rounding is unbiased (below 2^-32 of an
ulp off for values under 2^-48, where frac has more bits than the word).
Round-to-nearest (ties to even) storage is the comparison mode.
"""
from __future__ import annotations

import numpy as np

PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
F16_MAX = 65504.0
_MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(counter, key):
    """Philox4x32-10 (Salmon et al., SC'11), the rounds as the module docstring states them.

    counter: uint32 array [..., 4]; key: uint32 array [..., 2] (broadcast). Returns uint32 [..., 4]."""
    c = np.asarray(counter, dtype=np.uint64)
    k = np.broadcast_to(np.asarray(key, dtype=np.uint64), c.shape[:-1] + (2,)).copy()
    c0, c1, c2, c3 = (c[..., i].copy() for i in range(4))
    k0, k1 = k[..., 0].copy(), k[..., 1].copy()
    for rnd in range(10):
        p0 = c0 * np.uint64(PHILOX_M0)  # < 2^64: exact in uint64
        p1 = c2 * np.uint64(PHILOX_M1)
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
        if rnd < 9:
            k0 = (k0 + np.uint64(PHILOX_W0)) & _MASK32
            k1 = (k1 + np.uint64(PHILOX_W1)) & _MASK32
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def sr_words(n_elements: int, base_index: int, epoch: int, seed: int) -> np.ndarray:
    """The 32-bit words of elements base_index .. base_index + n - 1 (base_index a multiple of 4),
    from this build's counter layout (module docstring; the pages name no generator)."""
    assert base_index % 4 == 0 and n_elements % 4 == 0
    g = np.arange(base_index // 4, (base_index + n_elements) // 4, dtype=np.uint64)
    ctr = np.stack([g & _MASK32, g >> np.uint64(32), np.full_like(g, epoch), np.zeros_like(g)], axis=-1)
    key = np.array([seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF], dtype=np.uint64)
    return philox4x32_10(ctr, key).reshape(-1)


def f16_toward_zero(x32) -> np.ndarray:
    """binary32 -> binary16 rounded toward zero (finite inputs with |x| < 65520), as float32 values
    (IEEE 754 binary16; the lower neighbour of the stochastic rounding)."""
    x = np.asarray(x32, dtype=np.float32)
    near = x.astype(np.float16)  # round to nearest even
    over = np.abs(near.astype(np.float32)) > np.abs(x)
    toward = np.where(over, np.nextafter(near, np.float16(0)), near)
    return toward.astype(np.float32)


def stochastic_round_f16(x32, words) -> np.ndarray:
    """Stochastic rounding of binary32 values to binary16 with one 32-bit word per value: the
    FP16 checkpoint store of [RU] §06, with the rounding rule read in the module docstring."""
    x = np.asarray(x32, dtype=np.float32)
    r = np.asarray(words, dtype=np.uint64)
    ax = np.abs(x)
    big = ax >= np.float32(F16_MAX)
    axc = np.where(big, np.float32(0), ax)  # keep the arithmetic finite; saturated below
    lo = f16_toward_zero(axc)
    hi = np.nextafter(lo.astype(np.float16), np.float16(np.inf)).astype(np.float32)
    diff = (axc.astype(np.float64) - lo.astype(np.float64))  # exact
    ulp = hi.astype(np.float64) - lo.astype(np.float64)      # a power of two
    frac = np.where(np.isnan(diff), 0.0, diff / ulp)
    t = np.floor(frac * 2.0 ** 32).astype(np.uint64)
    mag = np.where(r < t, hi, lo)
    mag = np.where(big, np.float32(F16_MAX), mag)
    out = np.where(np.signbit(x), -mag, mag).astype(np.float16)
    return np.where(np.isnan(x), np.float16(np.nan), out)


def nearest_f16(x32) -> np.ndarray:
    """Round-to-nearest-even binary16 storage with saturation (the comparison mode; IEEE 754 binary16)."""
    x = np.asarray(x32, dtype=np.float32)
    y = np.clip(x, -F16_MAX, F16_MAX).astype(np.float16)
    return np.where(np.isnan(x), np.float16(np.nan), y)


class ReplayOracleF16:
    """ReplaySSM decoding with the checkpoint stored in FP16 (float64 arithmetic otherwise).

    The checkpoint holds binary16 values. Non-flush outputs, verify outputs and
    folds read it as it is stored: the unrolled window formula on the FP16
    checkpoint ([RU] §03 and §05). A fold computes the new state
    gamma_h S_ckpt + sum_j gamma_{j+1:h} v_j k_j^T in float64, gives the step
    its output S_new q from that unrounded state (reading: the fold has the
    full-precision state in hand), and stores rn32(S_new) rounded to binary16,
    stochastically (``mode="sr"``, generator words of this module) or to
    nearest (``mode="rn"``). Flush policy and pointers follow ``ReplayOracle``.
    Each flush of a sequence advances its epoch, which enters the counter.
    ``S`` is the exact conventional recurrence from the initial checkpoint,
    kept for error studies.
    """

    def __init__(self, S0_f16, L: int, R: int, G: int, seed: int, mode: str = "sr"):
        from .recurrence import head_groups

        self.ckpt = np.asarray(S0_f16, np.float64)
        self.B, self.H, self.P, self.N = self.ckpt.shape
        if not np.array_equal(self.ckpt.astype(np.float16).astype(np.float64), self.ckpt):
            raise ValueError("the initial checkpoint must hold binary16 values")
        self.G, self.L, self.R, self.seed, self.mode = G, L, R, seed, mode
        self.g = head_groups(self.H, G)
        self.S = self.ckpt.copy()
        self.start = np.zeros(self.B, np.int64)
        self.count = np.zeros(self.B, np.int64)
        self.epoch = np.zeros(self.B, np.int64)
        self.records = [[] for _ in range(self.B)]
        self._drafts = None

    def _store(self, b: int, S_new):
        x32 = np.asarray(S_new, np.float64).astype(np.float32)
        if self.mode == "sr":
            n = self.H * self.P * self.N
            words = sr_words(n, b * n, int(self.epoch[b]), self.seed).reshape(x32.shape)
            self.ckpt[b] = stochastic_round_f16(x32, words).astype(np.float64)
        else:
            self.ckpt[b] = nearest_f16(x32).astype(np.float64)
        self.epoch[b] += 1

    def _fold(self, b: int, recs):
        from .recurrence import unrolled_state

        a_, v_, k_ = (np.stack(x) for x in zip(*recs))
        return unrolled_state(self.ckpt[b], a_, v_, k_)

    def decode(self, alpha, v, k, q):
        """One decode step over the FP16 checkpoint ([RU] §03 non-flush / flush steps;
        §06 FP16 storage). Returns (o [B,H,P], flushed mask [B])."""
        from .recurrence import conventional_step, replay_output

        h = self.count + 1
        if np.any(h > self.R):
            raise ValueError("decode would exceed the ring capacity")
        flush = h >= self.L
        o = np.empty((self.B, self.H, self.P))
        for b in range(self.B):
            recs = self.records[b] + [(alpha[b].copy(), v[b].copy(), k[b].copy())]
            if flush[b]:
                S_new = self._fold(b, recs)
                o[b] = np.einsum("hpn,hn->hp", S_new, q[b][self.g])
                self._store(b, S_new)
                self.records[b] = []
                self.start[b] = (self.start[b] + h[b]) % self.R
                self.count[b] = 0
            else:
                a_, v_, k_ = (np.stack(x) for x in zip(*recs))
                o[b] = replay_output(self.ckpt[b], a_, v_, k_, q[b])
                self.records[b] = recs
                self.count[b] = h[b]
        self.S, _ = conventional_step(self.S, alpha, v, k, q)
        self._drafts = None
        return o, flush

    def verify(self, alpha, v, k, q):
        """Output-only evaluation of T drafts from the stored checkpoint ([RU] §05;
        [ZH] 方法/产品要点, verify formula). Returns O [B,T,H,P]."""
        from .recurrence import verify_outputs

        T = alpha.shape[1]
        if np.any(self.count + T > self.R):
            raise ValueError("verify would exceed the ring capacity")
        O = np.empty((self.B, T, self.H, self.P))
        for b in range(self.B):
            recs = self.records[b] + [(alpha[b, t], v[b, t], k[b, t]) for t in range(T)]
            a_, v_, k_ = (np.stack(x) for x in zip(*recs))
            O[b] = verify_outputs(self.ckpt[b], a_, v_, k_, q[b], int(self.count[b]))
        self._drafts = (alpha.copy(), v.copy(), k.copy(), q.copy(), T)
        return O

    def commit(self, accepted):
        """Keep the first accepted[b] drafts as records (count += a; [RU] §05)."""
        from .recurrence import conventional_step

        alpha, v, k, q, T = self._drafts
        a = np.asarray(accepted, np.int64)
        if np.any(a < 0) or np.any(a > T):
            raise ValueError("accepted length outside 0..T")
        for b in range(self.B):
            for t in range(int(a[b])):
                self.records[b].append((alpha[b, t].copy(), v[b, t].copy(), k[b, t].copy()))
        for t in range(T):
            m = t < a
            if np.any(m):
                self.S[m], _ = conventional_step(self.S[m], alpha[m, t], v[m, t], k[m, t], q[m, t])
        self.count = self.count + a
        self._drafts = None

    def flush(self, min_count: int):
        """Fold and store (rounded) every sequence holding at least min_count records ([RU] §03, §06)."""
        mask = (self.count >= min_count) & (self.count > 0)
        for b in np.nonzero(mask)[0]:
            self._store(b, self._fold(b, self.records[b]))
            self.records[b] = []
            self.start[b] = (self.start[b] + self.count[b]) % self.R
            self.count[b] = 0
        return mask

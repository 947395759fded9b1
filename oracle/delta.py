"""Gated delta-rule layers (Gated DeltaNet) under replay decoding: float64 oracle.

TEST INFRASTRUCTURE ONLY (see the package docstring for who may use it).

The pages name Gated DeltaNet among the SSM layers of hybrid models and say
that the same replay form applies to it ([ZH] 方法/产品要点 and the open
questions list; [RU] introduction), but give no formula. Readings:

Recurrence (the gated delta rule), per (sequence, value head), with the key and
query of the head's group:
    S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = S_t q_t
S is P x N, alpha_t in (0, 1] the decay, beta_t the write strength.

Replay form derived here. With A_t = alpha_t (I - beta_t k_t k_t^T), h records
after a checkpoint S_0 give
    S_h = S_0 A_1 ... A_h + sum_j beta_j v_j k_j^T A_{j+1} ... A_h,
so the output needs the query carried backwards through the records:
    u_h = q,   c_j = beta_j (k_j^T u_j),   u_{j-1} = alpha_j (u_j - c_j k_j),
    o = S_0 u_0 + sum_j c_j v_j.
The checkpoint is read once per step, as for the outer-product recurrence;
the extra work is O(h N) per head. A fold applies the records in order:
    S <- alpha_j S + beta_j (v_j - alpha_j S k_j) k_j^T.
Flush policy and pointers are those of ``replay.ReplayOracle``, and so are
speculative verify (T drafts evaluated on a copy of the exact state, nothing
changed) and commit (the first a drafts applied, count += a): the pages state
rollback and output-only evaluation for the replay form in general ([RU] 05),
and nothing in them is specific to the outer-product rule.

The write term of step j, w_j = beta_j (v_j - alpha_j S_{j-1} k_j) with
S_{j-1} the state just before it (``delta_pseudo_value``), makes every step
S_j = alpha_j S_{j-1} + w_j k_j^T: the outer-product recurrence with v_j
replaced by w_j. A replay may therefore keep w_j per record instead of v_j.
``tests/test_oracle_delta.py`` pins w_j to the step's own write term.
"""
from __future__ import annotations

import numpy as np

from .recurrence import head_groups
from .replay import CapacityError


def delta_step(S, alpha, beta, v, k, q):
    """One step of the definition for every (sequence, head): the gated delta rule,
    this build's reading of the Gated DeltaNet layers the pages name ([RU]
    introduction; [ZH] 事件概述或研究问题).

    S [B,H,P,N], alpha and beta [B,H], v [B,H,P], k and q [B,G,N] (float64).
    Returns (S_t, o_t [B,H,P]).
    """
    S = np.asarray(S, np.float64)
    B, H, P, N = S.shape
    g = head_groups(H, k.shape[1])
    kh, qh = k[:, g, :], q[:, g, :]  # [B,H,N]
    Sk = np.einsum("bhpn,bhn->bhp", S, kh)
    a = alpha[:, :, None, None]
    bt = beta[:, :, None, None]
    # alpha S (I - beta k k^T) + beta v k^T
    S_new = a * (S - bt * Sk[..., None] * kh[:, :, None, :]) + bt * v[..., None] * kh[:, :, None, :]
    return S_new, np.einsum("bhpn,bhn->bhp", S_new, qh)


def delta_pseudo_value(S, alpha, beta, v, k):
    """The write term of one step: w = beta (v - alpha S k), so that
    S_t = alpha S + w k^T (derived here for the pages' claim that GDN can use the
    same replay form, [ZH] 待核实 list). S [B,H,P,N] is the state before the step, alpha and
    beta [B,H], v [B,H,P], k [B,G,N]. Returns w [B,H,P]."""
    S = np.asarray(S, np.float64)
    g = head_groups(S.shape[1], k.shape[1])
    Sk = np.einsum("bhpn,bhn->bhp", S, k[:, g, :])
    return beta[:, :, None] * (v - alpha[:, :, None] * Sk)


def delta_replay_output(S_ckpt, alphas, betas, vs, ks, q):
    """Output-only evaluation for one sequence after h records (form above): the
    pages' output-only evaluation ([RU] §05; [ZH] 方法/产品要点) carried to the
    delta rule.

    S_ckpt [H,P,N]; alphas, betas [h,H]; vs [h,H,P]; ks [h,G,N]; q [G,N].
    Returns o [H,P].
    """
    S_ckpt = np.asarray(S_ckpt, np.float64)
    H, P, N = S_ckpt.shape
    g = head_groups(H, q.shape[0])
    h = len(alphas)
    o = np.empty((H, P))
    for head in range(H):
        u = np.array(q[g[head]], np.float64)
        val = np.zeros(P)
        for j in range(h - 1, -1, -1):
            kj = ks[j, g[head]]
            c = betas[j, head] * float(kj @ u)
            val += c * vs[j, head]
            u = alphas[j, head] * (u - c * kj)
        o[head] = S_ckpt[head] @ u + val
    return o


def delta_fold(S_ckpt, alphas, betas, vs, ks):
    """The state after h records, applied in order (one sequence): the flush fold ([RU] §03)."""
    S = np.array(S_ckpt, np.float64)
    H = S.shape[0]
    g = head_groups(H, ks.shape[1])
    for j in range(len(alphas)):
        for head in range(H):
            kj = ks[j, g[head]]
            y = S[head] @ kj
            S[head] = alphas[j, head] * S[head] + np.outer(betas[j, head] * (vs[j, head] - alphas[j, head] * y), kj)
    return S


class DeltaReplayOracle:
    """Replay decoding (and speculative verify / commit) of a gated delta-rule layer
    ([RU] §03 and §05, with the delta rule in place of the outer product).

    The exact target is the definition, so ``S`` advances by ``delta_step``
    and the outputs are its outputs; ``ckpt`` is the exact state at each
    sequence's last flush. The integers (start, count, flush events) follow the
    eager policy of ``ReplayOracle``: the step whose append brings the count to
    L folds all records.
    """

    def __init__(self, S0, L: int, R: int, G: int):
        self.S = np.array(S0, np.float64)
        self.ckpt = self.S.copy()
        self.B = self.S.shape[0]
        self.L, self.R, self.G = L, R, G
        self.start = np.zeros(self.B, np.int64)
        self.count = np.zeros(self.B, np.int64)
        self._drafts = None

    def decode(self, alpha, beta, v, k, q):
        """One decode step ([RU] §03 non-flush / flush policy). Returns (o [B,H,P], flushed mask [B])."""
        h = self.count + 1
        if np.any(h > self.R):
            raise CapacityError("decode would exceed the ring capacity")
        self._drafts = None
        self.S, o = delta_step(self.S, alpha, beta, v, k, q)
        flush = h >= self.L
        self.ckpt[flush] = self.S[flush]
        self.start = np.where(flush, (self.start + h) % self.R, self.start)
        self.count = np.where(flush, 0, h)
        return o, flush

    def verify(self, alpha, beta, v, k, q):
        """Speculative verify of T drafts: alpha, beta [B,T,H], v [B,T,H,P], k, q [B,T,G,N].

        Output-only: the drafts run on a scratch copy of the exact state, so the
        real state and the pointers stay unchanged ([RU] §05). Returns O [B,T,H,P].
        """
        T = alpha.shape[1]
        if np.any(self.count + T > self.R):
            raise CapacityError("verify would exceed the ring capacity")
        O = np.empty(v.shape)
        Sc = self.S.copy()
        for t in range(T):
            Sc, O[:, t] = delta_step(Sc, alpha[:, t], beta[:, t], v[:, t], k[:, t], q[:, t])
        self._drafts = (alpha.copy(), beta.copy(), v.copy(), k.copy(), q.copy(), T)
        return O

    def commit(self, accepted):
        """Apply the first accepted[b] drafts of the last verify (count += a; [RU] §05)."""
        if self._drafts is None:
            raise CapacityError("commit without a preceding verify")
        alpha, beta, v, k, q, T = self._drafts
        a = np.asarray(accepted, np.int64)
        if np.any(a < 0) or np.any(a > T):
            raise CapacityError("accepted length outside 0..T")
        for t in range(T):
            m = t < a
            if np.any(m):
                self.S[m], _ = delta_step(self.S[m], alpha[m, t], beta[m, t], v[m, t], k[m, t], q[m, t])
        self.count = self.count + a
        self._drafts = None

    def flush(self, min_count: int):
        """Fold every sequence holding at least min_count records ([RU] §03). Returns the mask."""
        mask = (self.count >= min_count) & (self.count > 0)
        self.ckpt[mask] = self.S[mask]
        self.start = np.where(mask, (self.start + self.count) % self.R, self.start)
        self.count = np.where(mask, 0, self.count)
        return mask

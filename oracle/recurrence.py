"""The gated outer-product recurrence and its unrolled forms, in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring for who may use it).

Notation (pages [RU] §01, §03 and [ZH] 方法/产品要点):
  S      state of one value head, P x N (rows follow v, columns follow k and q)
  alpha  data-dependent scalar decay per step and value head
  v      value vector (length P), per value head
  k, q   key / query vectors (length N), shared by the value heads of a group
Records are numbered 1..h after the checkpoint S_ckpt. The cumulative decay is
gamma_{a:b} = prod_{i=a..b} alpha_i. An empty product is 1 and gamma_h means
gamma_{1:h}. This indexing is a reading: the pages call gamma only the
"cumulative decay".
"""
from __future__ import annotations

import numpy as np


def to_f64(x) -> np.ndarray:
    """Exact up-cast of a torch tensor (fp32/bf16) or array to a float64 ndarray
    (no passage: the oracle works in float64 on the stored inputs)."""
    try:
        import torch

        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu")
            if x.dtype in (torch.bfloat16, torch.float16):
                x = x.to(torch.float32)  # exact: both embed in fp32
            return x.numpy().astype(np.float64)
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def head_groups(H: int, G: int) -> np.ndarray:
    """Group index of every value head.

    The pages only say that k and q are shared by the value heads of a group
    ([ZH] 方法/产品要点, "KᵀQ shared across a group's value heads"). Reading:
    contiguous blocks of H/G heads form a group (the Mamba-2 convention), so
    head h uses group h // (H/G).
    """
    if G <= 0 or H % G:
        raise ValueError(f"H={H} must be a positive multiple of G={G}")
    return np.arange(H) // (H // G)


def conventional_step(S, alpha, v, k, q):
    """One decode step for every (sequence, head). This is the definition the
    oracle follows ([RU] §01, recurrence):

        S_t = alpha_t S_{t-1} + v_t k_t^T,    o_t = S_t q_t

    S [B,H,P,N], alpha [B,H], v [B,H,P], k and q [B,G,N], all float64.
    Returns (S_t, o_t) with o_t of shape [B,H,P].
    """
    S = np.asarray(S, np.float64)
    B, H, P, N = S.shape
    g = head_groups(H, k.shape[1])
    kh = k[:, g, :]  # [B,H,N]: each value head's key
    qh = q[:, g, :]  # [B,H,N]
    S_new = alpha[:, :, None, None] * S + v[:, :, :, None] * kh[:, :, None, :]
    o = (S_new * qh[:, :, None, :]).sum(axis=-1)
    return S_new, o


def _gamma(alphas_head, a: int, b: int) -> float:
    """gamma_{a:b} for one head: product of alpha_i for i = a..b (1-based, inclusive)."""
    out = 1.0
    for i in range(a, b + 1):
        out *= float(alphas_head[i - 1])
    return out


def unrolled_state(S_ckpt, alphas, vs, ks):
    """State after h records, written as the unrolled window sum
    ([RU] §03, unrolled equation; [ZH] 方法/产品要点, core representation):

        S_h = gamma_h S_ckpt + sum_{j=1..h} gamma_{j+1:h} v_j k_j^T

    One sequence: S_ckpt [H,P,N], alphas [h,H], vs [h,H,P], ks [h,G,N].
    The loops and direct products are written out on purpose. This function
    computes the sum independently of ``conventional_step``.
    """
    S_ckpt = np.asarray(S_ckpt, np.float64)
    H, P, N = S_ckpt.shape
    h = len(alphas)
    g = head_groups(H, ks.shape[1] if h else 1) if h else np.zeros(H, int)
    out = np.empty_like(S_ckpt)
    for head in range(H):
        acc = _gamma(alphas[:, head], 1, h) * S_ckpt[head]
        for j in range(1, h + 1):
            acc = acc + _gamma(alphas[:, head], j + 1, h) * np.outer(vs[j - 1, head], ks[j - 1, g[head]])
        out[head] = acc
    return out


def replay_output(S_ckpt, alphas, vs, ks, q):
    """Output-only evaluation for one query ([RU] §05; [ZH] 方法/产品要点):

        o = gamma_h (S_ckpt q) + V (w ⊙ K^T q),   w_j = gamma_{j+1:h}

    One sequence. S_ckpt [H,P,N] is the checkpoint (or its dequantized read
    copy). alphas [h,H], vs [h,H,P] and ks [h,G,N] are the records since the
    checkpoint, the current one last. q is [G,N]. Returns o [H,P].
    """
    S_ckpt = np.asarray(S_ckpt, np.float64)
    H, P, N = S_ckpt.shape
    G = q.shape[0]
    g = head_groups(H, G)
    h = len(alphas)
    o = np.empty((H, P))
    for head in range(H):
        qg = q[g[head]]
        term = _gamma(alphas[:, head], 1, h) * (S_ckpt[head] @ qg)
        for j in range(1, h + 1):
            w_j = _gamma(alphas[:, head], j + 1, h)
            s_j = float(ks[j - 1, g[head]] @ qg)  # k_j^T q
            term = term + (w_j * s_j) * vs[j - 1, head]
        o[head] = term
    return o


def verify_outputs(S_ckpt, alphas, vs, ks, Q, h: int):
    """Outputs for T draft queries in one pass ([ZH] 方法/产品要点, verify form):

        O = S_ckpt Q D + V (W ⊙ (K^T Q))

    One sequence. The records are the h committed ones followed by the T
    drafts: alphas [h+T,H], vs [h+T,H,P], ks [h+T,G,N]. Q is [T,G,N].
    Reading of the undefined symbols: D = diag(gamma_{1:h+tau}) and
    W[j,tau] = gamma_{j+1:h+tau} for j <= h+tau, else 0, with tau = 1..T.
    Returns O [T,H,P].
    """
    S_ckpt = np.asarray(S_ckpt, np.float64)
    H, P, N = S_ckpt.shape
    T, G, _ = Q.shape
    J = h + T
    g = head_groups(H, G)
    O = np.empty((T, H, P))
    for head in range(H):
        a = alphas[:, head]
        D = np.diag([_gamma(a, 1, h + t) for t in range(1, T + 1)])  # [T,T]
        W = np.zeros((J, T))
        for t in range(1, T + 1):
            for j in range(1, h + t + 1):
                W[j - 1, t - 1] = _gamma(a, j + 1, h + t)
        Qm = Q[:, g[head], :].T  # [N,T], columns are the queries
        Km = ks[:, g[head], :].T  # [N,J], columns are the keys
        Vm = vs[:, head, :].T  # [P,J], columns are the values
        Oh = S_ckpt[head] @ Qm @ D + Vm @ (W * (Km.T @ Qm))  # [P,T]
        O[:, head, :] = Oh.T
    return O

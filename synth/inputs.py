"""Seeded input recipes for the ReplaySSM decode workloads.

Every tensor comes from one ``torch.Generator`` on the CPU, so a given
(shape, seed) pair yields the same bytes on any machine. Draw order:

1. the initial FP32 checkpoint ``S0 ~ N(0, 0.1^2)`` of shape [B, H, P, N];
2. per decode step, in this order: ``u ~ N(mu, 1)`` [B, H] turned into the
   decay ``alpha = exp(-softplus(u))`` (fp32), ``v ~ N(0,1)/sqrt(N)`` [B, H, P],
   ``k ~ N(0,1)/sqrt(N)`` [B, G, N], ``q ~ N(0,1)/sqrt(N)`` [B, G, N];
   v, k and q are then cast to the storage dtype (bf16 or fp32);
3. per speculative round, the same four draws with a draft axis T after B,
   then (separately, see ``accepted_lengths``) the accepted length per sequence
   drawn uniformly from 0..T.

The decay recipe and the 1/sqrt(N) scaling are the tiny-case recipe of the
workload list; the larger layer shapes reuse it. ``mu`` shifts u to produce
long-memory decays (mu = -4 gives alpha ~ 0.98).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Shape:
    """Sizes of one SSM layer's decode problem.

    B sequences, H value heads, P head dim of v/o, N state dim of k/q,
    G groups (k and q are shared by H/G consecutive value heads),
    L flush window, T_max largest speculative draft count (1 for plain decode).
    """

    B: int
    H: int
    P: int
    N: int
    G: int
    L: int
    T_max: int = 1
    in_dtype: str = "bf16"  # storage dtype of v, k, q: "bf16" or "f32"
    seed: int = 0

    @property
    def R(self) -> int:
        """Ring slots: the window plus room for T_max - 1 speculative drafts."""
        return self.L + self.T_max - 1

    @property
    def torch_dtype(self) -> torch.dtype:
        return {"bf16": torch.bfloat16, "f32": torch.float32}[self.in_dtype]

    def with_(self, **kw) -> "Shape":
        return replace(self, **kw)


# Named workloads (sizes from the workload list of the method's evaluation).
PRESETS = {
    # 2 sequences, 2 heads, P=N=16, one group, window 4, fp32 inputs.
    "tiny_b2_h2_p16_n16_l4": Shape(B=2, H=2, P=16, N=16, G=1, L=4, in_dtype="f32", seed=0),
    # One Mamba-2-shaped layer: 4 MiB FP32 state per sequence, batch 256, window 16.
    "mamba2_layer_b256_l16": Shape(B=256, H=128, P=64, N=128, G=8, L=16, seed=1),
    # Same layer, batch 512, four drafts per speculative round.
    "mamba2_verify_b512_t4": Shape(B=512, H=128, P=64, N=128, G=8, L=16, T_max=4, seed=2),
    # Quantized-read study: batch 64, 32 heads, two groups.
    "quant_b64_h32_l16": Shape(B=64, H=32, P=64, N=128, G=2, L=16, seed=3),
    # Alternative layer shape: 32 value heads of dim 128 sharing 16 k/q heads.
    "alt_h32_p128_n128_g16": Shape(B=256, H=32, P=128, N=128, G=16, L=16, seed=4),
}


def make_generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def initial_state(shape: Shape, gen: torch.Generator, std: float = 0.1) -> torch.Tensor:
    """FP32 initial checkpoint [B, H, P, N] with entries N(0, std^2)."""
    s = torch.randn((shape.B, shape.H, shape.P, shape.N), generator=gen, dtype=torch.float32)
    return s.mul_(std)


def _decay_from_normal(u: torch.Tensor) -> torch.Tensor:
    # alpha = exp(-softplus(u)) in fp32 (the decay recipe of the tiny workload).
    return torch.exp(-torch.nn.functional.softplus(u)).to(torch.float32)


def decode_step_inputs(shape: Shape, gen: torch.Generator, mu: float = 0.0):
    """One decode step's inputs (alpha [B,H] fp32, v [B,H,P], k [B,G,N], q [B,G,N])."""
    B, H, P, N, G = shape.B, shape.H, shape.P, shape.N, shape.G
    sc = 1.0 / math.sqrt(N)
    u = torch.randn((B, H), generator=gen, dtype=torch.float32) + mu
    alpha = _decay_from_normal(u)
    v = (torch.randn((B, H, P), generator=gen, dtype=torch.float32) * sc).to(shape.torch_dtype)
    k = (torch.randn((B, G, N), generator=gen, dtype=torch.float32) * sc).to(shape.torch_dtype)
    q = (torch.randn((B, G, N), generator=gen, dtype=torch.float32) * sc).to(shape.torch_dtype)
    return alpha, v, k, q


def verify_round_inputs(shape: Shape, T: int, gen: torch.Generator, mu: float = 0.0):
    """T draft records and queries: alpha [B,T,H], v [B,T,H,P], k,q [B,T,G,N]."""
    B, H, P, N, G = shape.B, shape.H, shape.P, shape.N, shape.G
    sc = 1.0 / math.sqrt(N)
    u = torch.randn((B, T, H), generator=gen, dtype=torch.float32) + mu
    alpha = _decay_from_normal(u)
    v = (torch.randn((B, T, H, P), generator=gen, dtype=torch.float32) * sc).to(shape.torch_dtype)
    k = (torch.randn((B, T, G, N), generator=gen, dtype=torch.float32) * sc).to(shape.torch_dtype)
    q = (torch.randn((B, T, G, N), generator=gen, dtype=torch.float32) * sc).to(shape.torch_dtype)
    return alpha, v, k, q


def accepted_lengths(B: int, T: int, gen: torch.Generator) -> torch.Tensor:
    """Accepted draft count per sequence, uniform on 0..T, int32 [B]."""
    return torch.randint(0, T + 1, (B,), generator=gen, dtype=torch.int32)


def delta_step_inputs(shape: Shape, gen: torch.Generator, mu: float = 0.0):
    """One decode step's inputs for a gated delta-rule layer.

    Draw order: u ~ N(mu, 1) [B,H] -> alpha = exp(-softplus(u)); z ~ N(0, 1)
    [B,H] -> beta = sigmoid(z) (write strength in (0, 1)); v ~ N(0,1)/sqrt(N)
    [B,H,P]; k and q ~ N(0, 1) [B,G,N], each scaled to unit L2 norm per
    (sequence, group) as delta-rule layers normalize their keys and queries.
    v, k and q are then cast to the storage dtype. Returns (alpha, beta, v, k, q).
    """
    B, H, P, N, G = shape.B, shape.H, shape.P, shape.N, shape.G
    u = torch.randn((B, H), generator=gen, dtype=torch.float32) + mu
    alpha = _decay_from_normal(u)
    beta = torch.sigmoid(torch.randn((B, H), generator=gen, dtype=torch.float32))
    v = (torch.randn((B, H, P), generator=gen, dtype=torch.float32) / math.sqrt(N)).to(shape.torch_dtype)
    k = torch.randn((B, G, N), generator=gen, dtype=torch.float32)
    q = torch.randn((B, G, N), generator=gen, dtype=torch.float32)
    k = (k / k.norm(dim=-1, keepdim=True)).to(shape.torch_dtype)
    q = (q / q.norm(dim=-1, keepdim=True)).to(shape.torch_dtype)
    return alpha, beta, v, k, q


def delta_verify_round_inputs(shape: Shape, T: int, gen: torch.Generator, mu: float = 0.0):
    """T draft records and queries of a gated delta-rule layer: the recipe of
    ``delta_step_inputs`` with a draft axis T after B, drawn in the same order.
    Returns (alpha [B,T,H], beta [B,T,H], v [B,T,H,P], k [B,T,G,N], q [B,T,G,N])."""
    B, H, P, N, G = shape.B, shape.H, shape.P, shape.N, shape.G
    u = torch.randn((B, T, H), generator=gen, dtype=torch.float32) + mu
    alpha = _decay_from_normal(u)
    beta = torch.sigmoid(torch.randn((B, T, H), generator=gen, dtype=torch.float32))
    v = (torch.randn((B, T, H, P), generator=gen, dtype=torch.float32) / math.sqrt(N)).to(shape.torch_dtype)
    k = torch.randn((B, T, G, N), generator=gen, dtype=torch.float32)
    q = torch.randn((B, T, G, N), generator=gen, dtype=torch.float32)
    k = (k / k.norm(dim=-1, keepdim=True)).to(shape.torch_dtype)
    q = (q / q.norm(dim=-1, keepdim=True)).to(shape.torch_dtype)
    return alpha, beta, v, k, q

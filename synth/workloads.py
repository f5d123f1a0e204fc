"""Workload table and seeded tensor generators (no attention arithmetic here).

The shapes follow the diffusers context-parallelism pages' FLUX.1-dev examples:
a 1024x1024 image gives 512 text + (1024/16)^2 = 4096 image tokens, 24 heads of
width 128, run in bf16. Those weights and prompts are not needed: N(0, 1)
tensors of the same shapes stand in for the attention inputs.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    S: int
    D: int
    dtype: str            # "bf16" or "f32": the dtype of q, k, v
    ring_degree: int
    ulysses_degree: int
    uneven_ok: bool
    seed: int
    q_mult: float = 1.0   # 8.0 for the logit-stress variant
    description: str = ""

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def flops(self) -> int:
        """Algorithmic FLOPs of one full attention: QK^T plus PV, 2 FLOP per MAC."""
        return 4 * self.B * self.H * self.S * self.S * self.D


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_ring", B=1, H=2, S=256, D=64, dtype="f32", ring_degree=2,
                 ulysses_degree=1, uneven_ok=False, seed=0,
                 description="tiny ring: two 128-token K/V blocks merged by LSE"),
        Workload("flux_ring4", B=1, H=24, S=4608, D=128, dtype="bf16", ring_degree=4,
                 ulysses_degree=1, uneven_ok=False, seed=1,
                 description="FLUX-like joint attention (512 text + 4096 image tokens), ring of 4 x 1152"),
        Workload("flux_ulysses4", B=1, H=24, S=4608, D=128, dtype="bf16", ring_degree=1,
                 ulysses_degree=4, uneven_ok=False, seed=2,
                 description="FLUX-like shapes, Ulysses degree 4 (4 x [1152 tokens, 24 heads] -> 4 x [4608 tokens, 6 heads])"),
        Workload("flux_ulysses4_qx8", B=1, H=24, S=4608, D=128, dtype="bf16", ring_degree=1,
                 ulysses_degree=4, uneven_ok=False, seed=2, q_mult=8.0,
                 description="logit-stress variant: q scaled by 8"),
        Workload("ring_anything3", B=2, H=24, S=4607, D=128, dtype="bf16", ring_degree=3,
                 ulysses_degree=1, uneven_ok=True, seed=3,
                 description="Ring Anything: S not divisible, shards 1536/1536/1535"),
        Workload("flux1008_ulysses_anything4", B=1, H=24, S=4481, D=128, dtype="bf16", ring_degree=1,
                 ulysses_degree=4, uneven_ok=True, seed=5,
                 description="Ulysses Anything at a 1008x1008 image (512 + 63^2 = 4481 tokens): shards 1121/1120/1120/1120"),
        Workload("ulysses_anything5_heads", B=1, H=24, S=4608, D=128, dtype="bf16", ring_degree=1,
                 ulysses_degree=5, uneven_ok=True, seed=6,
                 description="Ulysses Anything with 24 heads over 5 groups (5/5/5/5/4) and 4608 tokens (922/922/922/921/921)"),
        Workload("video_unified", B=1, H=24, S=32768, D=128, dtype="bf16", ring_degree=2,
                 ulysses_degree=4, uneven_ok=False, seed=4,
                 description="video-length unified grid: ring 2 x Ulysses 4 (16384-token ring blocks, 6-head groups)"),
    ]
}


def _torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def make_qkv(B: int, H: int, S: int, D: int, dtype: str, seed: int, q_mult: float = 1.0,
             Skv: int | None = None):
    """Draw q [B,S,H,D] and k, v [B,Skv,H,D] on the CPU, in the order q, k, v."""
    Skv = S if Skv is None else Skv
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, S, H, D), generator=g, dtype=torch.float32)
    k = torch.randn((B, Skv, H, D), generator=g, dtype=torch.float32)
    v = torch.randn((B, Skv, H, D), generator=g, dtype=torch.float32)
    dt = _torch_dtype(dtype)
    q, k, v = q.to(dt), k.to(dt), v.to(dt)
    if q_mult != 1.0:
        q = q * q_mult
    return q, k, v


def make_dout(B: int, S: int, H: int, D: int, dtype: str, seed: int):
    """The upstream gradient dout [B,S,H,D] of a backward check: float32 N(0, 1)
    from its own CPU generator (seed + 1000), rounded to the workload dtype."""
    g = torch.Generator().manual_seed(seed + 1000)
    return torch.randn((B, S, H, D), generator=g, dtype=torch.float32).to(_torch_dtype(dtype))


def make_merge_operands(B: int, H: int, S: int, D: int, seed: int, neg_inf_rows: int = 0):
    """Two fp32 (out, lse) partials of the shapes a ring step produces.

    out_* are N(0,1) float32 [B,S,H,D]; lse_* are float32 [B,H,S] drawn as
    8 + 2*N(0,1) (the range of log-sum-exps over ~10^3 unit logits). The first
    token rows [0, n) of operand a get lse = -inf and out = 0 (an empty
    block); operand b is empty on rows [0, n/2) and [n, n + n/2), so rows with
    both empty, only a empty and only b empty all occur.
    """
    g = torch.Generator().manual_seed(seed)
    out_a = torch.randn((B, S, H, D), generator=g, dtype=torch.float32)
    out_b = torch.randn((B, S, H, D), generator=g, dtype=torch.float32)
    lse_a = 8.0 + 2.0 * torch.randn((B, H, S), generator=g, dtype=torch.float32)
    lse_b = 8.0 + 2.0 * torch.randn((B, H, S), generator=g, dtype=torch.float32)
    if neg_inf_rows:
        n = min(neg_inf_rows, S)
        half = n // 2
        lse_a[:, :, :n] = float("-inf")
        out_a[:, :n] = 0.0
        for lo, hi in ((0, half), (n, min(S, n + half))):
            lse_b[:, :, lo:hi] = float("-inf")
            out_b[:, lo:hi] = 0.0
    return out_a, lse_a, out_b, lse_b

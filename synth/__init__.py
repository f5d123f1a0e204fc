"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and bench.py.

This module holds no attention arithmetic: it only draws tensors and names the
workloads. Both sides of every parity check (the float64 CPU oracle and the
CUDA library) are fed from here, so they see bit-identical inputs.

Recipe (the same for every workload):
  * a CPU ``torch.Generator`` seeded with the workload's seed;
  * ``q``, ``k``, ``v`` drawn in that order as float32 N(0, 1), each of shape
    ``[B, S, H, D]`` (BSHD, D contiguous);
  * for bf16 workloads each tensor is then rounded to bfloat16 with
    round-to-nearest-even (``Tensor.to(torch.bfloat16)``);
  * the logit-stress variant multiplies ``q`` by 8 after rounding, which is
    exact in bf16 (a power of two);
  * a backward check draws ``dout`` N(0, 1) from its own generator
    (seed + 1000), rounded like q, k, v.
"""
from .workloads import WORKLOADS, Workload, make_dout, make_merge_operands, make_qkv

__all__ = ["WORKLOADS", "Workload", "make_dout", "make_qkv", "make_merge_operands"]

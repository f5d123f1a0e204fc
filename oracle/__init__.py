"""Float64 CPU oracle for context-parallel attention.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The CUDA library
never calls it and shares no code with it.

Every function is the plain definition (or the pages' decomposition of it)
written out in numpy float64; see ``cp_oracle`` for the passage each one
follows. All functions are pinned by ``tests/test_oracle_pins.py`` against
brute force, closed forms, invariants and library special cases.
"""
from .cp_oracle import (
    NotDivisibleError,
    UnsupportedComboError,
    attention,
    attention_bwd,
    attention_delta,
    attention_rows,
    head2seq,
    lse_merge,
    ring_attention,
    ring_shard_table,
    seq2head,
    ulysses_attention,
    unified_attention,
    cp_attention,
    cp_attention_bwd,
    ring_attention_bwd,
)

__all__ = [
    "NotDivisibleError",
    "UnsupportedComboError",
    "attention",
    "attention_bwd",
    "attention_delta",
    "cp_attention_bwd",
    "ring_attention_bwd",
    "attention_rows",
    "head2seq",
    "lse_merge",
    "ring_attention",
    "ring_shard_table",
    "seq2head",
    "ulysses_attention",
    "unified_attention",
    "cp_attention",
]

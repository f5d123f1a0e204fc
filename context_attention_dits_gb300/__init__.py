"""Context-parallel attention (forward and backward) for diffusion transformers on one GB300.

The computation lives in libcpattn.so (hand-written CUDA for sm_103a, C ABI in
include/cp_attn.h); this package is its build script and a thin torch binding.
"""
from .api import (  # noqa: F401
    CpError,
    cp_attention_bwd,
    cp_attention_bwd_launch_count,
    cp_attention_bwd_workspace_size,
    cp_attention_fwd,
    cp_attention_fwd_host,
    cp_attention_fwd_no_alloc,
    cp_attention_host_buffer_size,
    cp_attention_launch_count,
    cp_attention_validate,
    cp_attention_workspace_size,
    cp_block_attn_fwd,
    cp_check_device_status,
    cp_debug_bounded_wait_probe,
    cp_lse_merge,
    cp_ring_shard_table,
    cp_status_string,
    cp_ulysses_anything_head2seq,
    cp_ulysses_anything_seq2head,
    cp_ulysses_head2seq,
    cp_ulysses_seq2head,
    cp_version,
)
from ._lib import LIB_PATH, lib  # noqa: F401

"""Python binding of the C ABI with the same names (argument marshalling only).

Every call takes CUDA torch tensors, checks shapes and dtypes, and passes raw
device pointers, sizes and the current torch stream to libcpattn.so. All
computation happens in the library's kernels; PyTorch only supplies device
memory and the stream.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import CP_BF16, CP_F32, CP_LAP_FUSED, CP_LAP_STEPWISE, CpError, check, lib

_DT = {torch.bfloat16: CP_BF16, torch.float32: CP_F32}
_MODES = {"fused": CP_LAP_FUSED, "stepwise": CP_LAP_STEPWISE}


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _dt(t: torch.Tensor) -> int:
    if t.dtype not in _DT:
        raise TypeError(f"unsupported dtype {t.dtype}: q/k/v must be bfloat16 or float32")
    return _DT[t.dtype]


def _cuda(*ts):
    for t in ts:
        if not t.is_cuda:
            raise ValueError("tensors must live on a CUDA device")


def _mode(mode) -> int:
    return _MODES[mode] if isinstance(mode, str) else int(mode)


def cp_block_attn_fwd(q, k, v, out, lse, scale: float, stream=None):
    """Block attention of q [B,Sq,H,D] against k, v [B,Skv,H,D] -> out [B,Sq,H,D] f32, lse [B,H,Sq] f32.

    q, k, v may be views with a batch stride (the inner [S, H, D] must be dense);
    out likewise; lse must be dense.
    """
    _cuda(q, k, v, out, lse)
    B, Sq, H, D = q.shape
    Skv = k.shape[1]
    if k.shape != (B, Skv, H, D) or v.shape != k.shape or out.shape != (B, Sq, H, D) or lse.shape != (B, H, Sq):
        raise ValueError("shape mismatch")
    if q.dtype != k.dtype or q.dtype != v.dtype or out.dtype != torch.float32 or lse.dtype != torch.float32:
        raise TypeError("q, k, v must share a dtype; out and lse must be float32")
    for t in (q, k, v, out):
        if t.stride()[1:] != (H * D, D, 1):
            raise ValueError("the [S, H, D] part of each tensor must be dense")
    if not lse.is_contiguous():
        raise ValueError("lse must be dense")
    st = lib().cp_block_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                 B, H, Sq, Skv, D, float(scale), q.stride(0), k.stride(0), out.stride(0),
                                 _dt(q), _stream(stream))
    check(st, "cp_block_attn_fwd")


def cp_lse_merge(out_acc, lse_acc, out_blk, lse_blk, stream=None):
    """In place: (out_acc, lse_acc) <- merge((out_acc, lse_acc), (out_blk, lse_blk)); all float32 dense."""
    _cuda(out_acc, lse_acc, out_blk, lse_blk)
    B, S, H, D = out_acc.shape
    if out_blk.shape != out_acc.shape or lse_acc.shape != (B, H, S) or lse_blk.shape != (B, H, S):
        raise ValueError("shape mismatch")
    for t in (out_acc, lse_acc, out_blk, lse_blk):
        if t.dtype != torch.float32 or not t.is_contiguous():
            raise TypeError("merge operands must be dense float32")
    st = lib().cp_lse_merge(out_acc.data_ptr(), lse_acc.data_ptr(), out_blk.data_ptr(), lse_blk.data_ptr(),
                            B, H, S, D, _stream(stream))
    check(st, "cp_lse_merge")


def cp_ulysses_seq2head(x_in, x_out, stream=None):
    """[U, B, S/U, H, D] -> [U, B, S, H/U, D] (any dtype, dense)."""
    _cuda(x_in, x_out)
    U, B, Sl, H, D = x_in.shape
    if x_out.shape != (U, B, Sl * U, H // U, D) or x_out.dtype != x_in.dtype:
        raise ValueError("shape/dtype mismatch")
    if not (x_in.is_contiguous() and x_out.is_contiguous()):
        raise ValueError("tensors must be dense")
    st = lib().cp_ulysses_seq2head(x_in.data_ptr(), x_out.data_ptr(), U, B, Sl * U, H, D, x_in.element_size(),
                                   _stream(stream))
    check(st, "cp_ulysses_seq2head")


def cp_ulysses_head2seq(x_in, x_out, stream=None):
    """[U, B, S, H/U, D] -> [U, B, S/U, H, D] (any dtype, dense)."""
    _cuda(x_in, x_out)
    U, B, S, Hg, D = x_in.shape
    if x_out.shape != (U, B, S // U, Hg * U, D) or x_out.dtype != x_in.dtype:
        raise ValueError("shape/dtype mismatch")
    if not (x_in.is_contiguous() and x_out.is_contiguous()):
        raise ValueError("tensors must be dense")
    st = lib().cp_ulysses_head2seq(x_in.data_ptr(), x_out.data_ptr(), U, B, S, Hg * U, D, x_in.element_size(),
                                   _stream(stream))
    check(st, "cp_ulysses_head2seq")


def _anything(name, x_in, x_out, U, B, S, H, D, stream):
    _cuda(x_in, x_out)
    n = B * S * H * D
    if x_in.numel() != n or x_out.numel() != n or x_out.dtype != x_in.dtype:
        raise ValueError("both buffers must hold B*S*H*D elements of one dtype")
    if not (x_in.is_contiguous() and x_out.is_contiguous()):
        raise ValueError("buffers must be dense")
    st = getattr(lib(), name)(x_in.data_ptr(), x_out.data_ptr(), U, B, S, H, D, x_in.element_size(),
                              _stream(stream))
    check(st, name)


def cp_ulysses_anything_seq2head(x_in, x_out, U, B, S, H, D, stream=None):
    """Ragged regroup: rank blocks [B, S_u, H, D] back to back -> head-group blocks [B, S, H_g, D]
    back to back (balanced splits of S and H into U; any dtype; flat dense buffers)."""
    _anything("cp_ulysses_anything_seq2head", x_in, x_out, U, B, S, H, D, stream)


def cp_ulysses_anything_head2seq(x_in, x_out, U, B, S, H, D, stream=None):
    """Inverse of cp_ulysses_anything_seq2head."""
    _anything("cp_ulysses_anything_head2seq", x_in, x_out, U, B, S, H, D, stream)


def cp_attention_validate(B, H, S, D, ring_degree=1, ulysses_degree=1, uneven_ok=False, dtype=torch.bfloat16) -> int:
    """Status code cp_attention_fwd would return on validation (0 = ok). Host only."""
    return lib().cp_attention_validate(B, H, S, D, ring_degree, ulysses_degree, int(bool(uneven_ok)), _DT[dtype])


def cp_ring_shard_table(S: int, n: int, uneven_ok: bool = False):
    """[(offset, length)] of the n ring shards. Host only."""
    off = (ctypes.c_int * n)()
    ln = (ctypes.c_int * n)()
    check(lib().cp_ring_shard_table(S, n, int(bool(uneven_ok)), off, ln), "cp_ring_shard_table")
    return [(off[i], ln[i]) for i in range(n)]


def cp_attention_workspace_size(B, H, S, D, ring_degree=1, ulysses_degree=1, dtype=torch.bfloat16,
                                mode="fused") -> int:
    return int(lib().cp_attention_workspace_size(B, H, S, D, ring_degree, ulysses_degree, _DT[dtype], _mode(mode)))


def cp_attention_launch_count(B, H, S, D, ring_degree=1, ulysses_degree=1, dtype=torch.bfloat16,
                              mode="fused") -> int:
    return int(lib().cp_attention_launch_count(B, H, S, D, ring_degree, ulysses_degree, _DT[dtype], _mode(mode)))


def cp_attention_fwd(q, k, v, out, lse, scale: float, ring_degree: int = 1, ulysses_degree: int = 1,
                     uneven_ok: bool = False, workspace=None, mode="fused", stream=None, key_mask=None):
    """Context-parallel attention over global q, k, v [B,S,H,D] -> out [B,S,H,D] f32, lse [B,H,S] f32.

    workspace: a CUDA uint8 tensor of at least cp_attention_workspace_size(...)
    bytes; allocated here through torch when None. key_mask: optional CUDA
    bool/uint8 tensor [B, S] (True/nonzero = the key takes part); calls
    cp_attention_fwd_masked.
    """
    _cuda(q, k, v, out, lse)
    B, S, H, D = q.shape
    if k.shape != q.shape or v.shape != q.shape or out.shape != q.shape or lse.shape != (B, H, S):
        raise ValueError("shape mismatch")
    if q.dtype != k.dtype or q.dtype != v.dtype or out.dtype != torch.float32 or lse.dtype != torch.float32:
        raise TypeError("q, k, v must share a dtype; out and lse must be float32")
    for t in (q, k, v, out, lse):
        if not t.is_contiguous():
            raise ValueError("tensors must be dense")
    m = _mode(mode)
    need = cp_attention_workspace_size(B, H, S, D, ring_degree, ulysses_degree, q.dtype, m)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    if key_mask is not None:
        _cuda(key_mask)
        if key_mask.shape != (B, S) or key_mask.dtype not in (torch.bool, torch.uint8) or not key_mask.is_contiguous():
            raise ValueError("key_mask must be a dense bool or uint8 tensor [B, S]")
        st = lib().cp_attention_fwd_masked(q.data_ptr(), k.data_ptr(), v.data_ptr(), key_mask.data_ptr(),
                                           out.data_ptr(), lse.data_ptr(), B, H, S, D, float(scale), ring_degree,
                                           ulysses_degree, int(bool(uneven_ok)), ws_ptr, ws_bytes, _dt(q), m,
                                           _stream(stream))
        check(st, "cp_attention_fwd_masked")
        return
    st = lib().cp_attention_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                B, H, S, D, float(scale), ring_degree, ulysses_degree, int(bool(uneven_ok)),
                                ws_ptr, ws_bytes, _dt(q), m, _stream(stream))
    check(st, "cp_attention_fwd")


def cp_attention_host_buffer_size(B, H, S, D, ring_degree=1, ulysses_degree=1, dtype=torch.bfloat16,
                                  mode="fused") -> int:
    return int(lib().cp_attention_host_buffer_size(B, H, S, D, ring_degree, ulysses_degree, _DT[dtype], _mode(mode)))


def cp_attention_fwd_host(q, k, v, out, lse, scale: float, ring_degree: int = 1, ulysses_degree: int = 1,
                          uneven_ok: bool = False, dev_buffer=None, mode="fused", head_chunks: int = 5,
                          stream=None):
    """cp_attention_fwd over host (CPU, ideally pinned) tensors q, k, v [B,S,H,D], out [B,S,H,D] f32 and
    lse [B,H,S] f32, with transfers overlapping compute over head chunks. dev_buffer: a CUDA uint8 tensor
    of at least cp_attention_host_buffer_size(...) bytes (allocated here through torch when None).
    Returns without waiting; the results are in out, lse once `stream` reaches this point."""
    for t in (q, k, v, out, lse):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v, out, lse must be dense host tensors")
    B, S, H, D = q.shape
    if k.shape != q.shape or v.shape != q.shape or out.shape != (B, S, H, D) or lse.shape != (B, H, S):
        raise ValueError("shape mismatch")
    if k.dtype != q.dtype or v.dtype != q.dtype or out.dtype != torch.float32 or lse.dtype != torch.float32:
        raise ValueError("dtype mismatch")
    need = cp_attention_host_buffer_size(B, H, S, D, ring_degree, ulysses_degree, q.dtype, mode)
    if dev_buffer is None:
        dev_buffer = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    _cuda(dev_buffer)
    st = lib().cp_attention_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                     B, H, S, D, float(scale), ring_degree, ulysses_degree, int(bool(uneven_ok)),
                                     dev_buffer.data_ptr(), dev_buffer.numel(), _dt(q), _mode(mode), head_chunks,
                                     _stream(stream))
    check(st, "cp_attention_fwd_host")
    return dev_buffer


def cp_attention_fwd_no_alloc(q, k, v, out, lse, scale: float, ring_degree: int = 1, ulysses_degree: int = 1,
                              uneven_ok: bool = False, mode="fused", stream=None):
    """cp_attention_fwd with the library's built-in 64 MiB device workspace (no allocation).

    For callers that cannot allocate device memory. All calls share the
    built-in workspace: calls that overlap on the GPU race.
    """
    _cuda(q, k, v, out, lse)
    B, S, H, D = q.shape
    if k.shape != q.shape or v.shape != q.shape or out.shape != q.shape or lse.shape != (B, H, S):
        raise ValueError("shape mismatch")
    if q.dtype != k.dtype or q.dtype != v.dtype or out.dtype != torch.float32 or lse.dtype != torch.float32:
        raise TypeError("q, k, v must share a dtype; out and lse must be float32")
    for t in (q, k, v, out, lse):
        if not t.is_contiguous():
            raise ValueError("tensors must be dense")
    st = lib().cp_attention_fwd_no_alloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                         B, H, S, D, float(scale), ring_degree, ulysses_degree, int(bool(uneven_ok)),
                                         _dt(q), _mode(mode), _stream(stream))
    check(st, "cp_attention_fwd_no_alloc")


def cp_attention_bwd_workspace_size(B, H, S, D, ring_degree=1, ulysses_degree=1, dtype=torch.bfloat16) -> int:
    return int(lib().cp_attention_bwd_workspace_size(B, H, S, D, ring_degree, ulysses_degree, _DT[dtype]))


def cp_attention_bwd_launch_count(B, H, S, D, ring_degree=1, ulysses_degree=1, dtype=torch.bfloat16) -> int:
    return int(lib().cp_attention_bwd_launch_count(B, H, S, D, ring_degree, ulysses_degree, _DT[dtype]))


def cp_attention_bwd(q, k, v, out, dout, lse, dq, dk, dv, scale: float, ring_degree: int = 1,
                     ulysses_degree: int = 1, uneven_ok: bool = False, workspace=None, stream=None):
    """Backward of cp_attention_fwd: q, k, v, dout [B,S,H,D] (one dtype), out [B,S,H,D] f32 and
    lse [B,H,S] f32 from the forward -> dq, dk, dv [B,S,H,D] f32 (written).

    Ring, Ulysses, unified, and Ulysses Anything (uneven_ok with ulysses_degree > 1); Ring
    Anything is inference only and raises. workspace: a CUDA uint8 tensor of at least
    cp_attention_bwd_workspace_size(...) bytes; allocated here through torch when None.
    """
    _cuda(q, k, v, out, dout, lse, dq, dk, dv)
    B, S, H, D = q.shape
    for t in (k, v, dout, out, dq, dk, dv):
        if t.shape != q.shape:
            raise ValueError("shape mismatch")
    if lse.shape != (B, H, S):
        raise ValueError("lse must be [B, H, S]")
    if k.dtype != q.dtype or v.dtype != q.dtype or dout.dtype != q.dtype:
        raise TypeError("q, k, v and dout must share a dtype")
    for t in (out, lse, dq, dk, dv):
        if t.dtype != torch.float32:
            raise TypeError("out, lse, dq, dk and dv must be float32")
    for t in (q, k, v, out, dout, lse, dq, dk, dv):
        if not t.is_contiguous():
            raise ValueError("tensors must be dense")
    need = cp_attention_bwd_workspace_size(B, H, S, D, ring_degree, ulysses_degree, q.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _cuda(workspace)
    st = lib().cp_attention_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), dout.data_ptr(),
                                lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, S, D,
                                float(scale), ring_degree, ulysses_degree, int(bool(uneven_ok)),
                                workspace.data_ptr(), workspace.numel(), _dt(q), _stream(stream))
    check(st, "cp_attention_bwd")


def cp_check_device_status(stream=None) -> int:
    """Synchronizes the stream; returns 0, or CP_ERR_TIMEOUT if a kernel's bounded wait expired."""
    return int(lib().cp_check_device_status(_stream(stream)))


def cp_debug_bounded_wait_probe(timeout_us: int, stream=None):
    check(lib().cp_debug_bounded_wait_probe(int(timeout_us), _stream(stream)), "cp_debug_bounded_wait_probe")


def cp_status_string(status: int) -> str:
    return _lib.status_string(status)


def cp_version() -> int:
    return int(lib().cp_version())


__all__ = [
    "CpError", "cp_block_attn_fwd", "cp_lse_merge", "cp_ulysses_seq2head", "cp_ulysses_head2seq",
    "cp_ulysses_anything_seq2head", "cp_ulysses_anything_head2seq",
    "cp_attention_validate", "cp_ring_shard_table", "cp_attention_workspace_size", "cp_attention_launch_count",
    "cp_attention_bwd", "cp_attention_bwd_workspace_size", "cp_attention_bwd_launch_count",
    "cp_attention_fwd", "cp_attention_fwd_no_alloc", "cp_attention_fwd_host", "cp_attention_host_buffer_size", "cp_check_device_status", "cp_debug_bounded_wait_probe", "cp_status_string", "cp_version",
]

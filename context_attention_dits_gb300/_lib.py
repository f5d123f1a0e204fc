"""ctypes declarations of libcpattn.so (the C ABI in include/cp_attn.h).

Loading fails loudly when the library has not been built: there is no other
implementation of these calls.
"""
from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libcpattn.so")

# status codes (cp_status)
CP_OK = 0
CP_ERR_INVALID_ARG = -1
CP_ERR_NOT_DIVISIBLE = -2
CP_ERR_UNSUPPORTED_COMBO = -3
CP_ERR_ALIGNMENT = -4
CP_ERR_CUDA = -5
CP_ERR_TIMEOUT = -6
CP_ERR_WORKSPACE = -7
CP_ERR_UNSUPPORTED_DEVICE = -8

CP_BF16 = 0
CP_F32 = 1
CP_LAP_FUSED = 0
CP_LAP_STEPWISE = 1

# every symbol include/cp_attn.h declares, with (restype, argtypes)
_vp, _i, _i64, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
_ip = ctypes.POINTER(ctypes.c_int)
SIGNATURES = {
    "cp_status_string": (ctypes.c_char_p, [_i]),
    "cp_version": (_i, []),
    "cp_block_attn_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i64, _i64, _i64, _i, _vp]),
    "cp_lse_merge": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp]),
    "cp_ulysses_seq2head": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _i, _vp]),
    "cp_ulysses_head2seq": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _i, _vp]),
    "cp_ulysses_anything_seq2head": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _i, _vp]),
    "cp_ulysses_anything_head2seq": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _i, _vp]),
    "cp_attention_validate": (_i, [_i, _i, _i, _i, _i, _i, _i, _i]),
    "cp_ring_shard_table": (_i, [_i, _i, _i, _ip, _ip]),
    "cp_attention_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i, _i, _i]),
    "cp_attention_launch_count": (_i, [_i, _i, _i, _i, _i, _i, _i, _i]),
    "cp_attention_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _i, _i, _vp, _sz, _i, _i, _vp]),
    "cp_check_device_status": (_i, [_vp]),
    "cp_debug_bounded_wait_probe": (_i, [_i, _vp]),
    "cp_attention_fwd_no_alloc": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _i, _i, _i, _i, _vp]),
    "cp_attention_host_buffer_size": (_sz, [_i, _i, _i, _i, _i, _i, _i, _i]),
    "cp_attention_fwd_masked": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _i, _i, _vp, _sz, _i, _i,
                                     _vp]),
    "cp_attention_fwd_host": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _i, _i, _vp, _sz, _i, _i, _i,
                                   _vp]),
    "cp_attention_bwd_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i, _i]),
    "cp_attention_bwd_launch_count": (_i, [_i, _i, _i, _i, _i, _i, _i]),
    "cp_attention_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _i, _i, _vp, _sz,
                              _i, _vp]),
}
CP_NO_ALLOC_WORKSPACE_BYTES = 64 * 1024 * 1024

_lock = threading.Lock()
_lib = None


class CpError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"libcpattn.so is not built ({LIB_PATH}); run "
                        "`python -m context_attention_dits_gb300.build`")
                L = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    fn = getattr(L, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().cp_status_string(int(status)).decode()


def check(status: int, where: str) -> None:
    if status != CP_OK:
        raise CpError(status, where)

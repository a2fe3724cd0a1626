"""ctypes binding of the C ABI in ``include/sp_api.h``.

Argument marshalling only: every step of the sequence-parallel path runs in
the CUDA library.  PyTorch supplies device memory and the current stream.
There is no fallback: if the shared library is missing, importing the
binding fails with instructions to build it.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libsp_gb300.so")

SP_OK = 0
SP_ERR_NOT_DIVISIBLE = 1
SP_ERR_HEADS_NOT_DIVISIBLE = 2
SP_ERR_INVALID_ARG = 3
SP_ERR_ALIGNMENT = 4
SP_ERR_UNSUPPORTED = 5
SP_ERR_TIMEOUT = 6
SP_ERR_BARRIER = 7
SP_ERR_CUDA = 8

SP_F32, SP_BF16 = 0, 1
SP_MASK_NONE, SP_MASK_KEY, SP_MASK_FULL = 0, 1, 2
SP_MAX_RANKS = 8
SP_WORKSPACE_HEADER_BYTES = 256
SP_WORKSPACE_KV_STALL_OFFSET = 80  # test hook word of the workspace header
SP_SHARD_KV, SP_SHARD_Q = 1, 2

# Symbols declared in include/sp_api.h, with (restype, argtypes).
_P, _I, _I64, _Z, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
_PP = ctypes.POINTER(ctypes.c_void_p)
_IP = ctypes.POINTER(ctypes.c_int)
_I64P = ctypes.POINTER(ctypes.c_int64)
SIGNATURES = {
    "sp_status_string": (ctypes.c_char_p, [_I]),
    "sp_last_error": (ctypes.c_char_p, []),
    "sp_version": (_I, []),
    "sp_launch_count": (ctypes.c_uint64, []),
    "sp_padded_len": (_I, [_I, _I, _IP]),
    "sp_pad": (_I, [_P, _P, _I, _I, _I, _I64, _P]),
    "sp_pad_mask": (_I, [_P, _P, _I, _I, _I, _P]),
    "sp_partition": (_I, [_I, _I, _IP, _IP]),
    "sp_tile": (_I, [_P, _PP, _I, _I, _I, _I64, _P]),
    "sp_optimal_split": (_I, [_I, _IP, _IP]),
    "sp_tile_2d": (_I, [_P, _PP, _I, _I, _I, _I, _I, _I, _I64, _P]),
    "sp_gather_2d": (_I, [_PP, _P, _I, _I, _I, _I, _I, _I, _I64, _P]),
    "sp_send_recv_heads": (_I, [_PP, _PP, _I, _I, _I, _I, _I, _I, _P, _P]),
    "sp_gather_heads": (_I, [_PP, _PP, _I, _I, _I, _I, _I, _I, _P, _P]),
    "sp_send_recv_heads_noalloc": (_I, [_PP, _PP, _I, _I, _I, _I, _I, _I, _IP, _P]),
    "sp_pad_send_heads": (_I, [_P, _PP, _I, _I, _I, _I, _I, _I, _I, _P, _P]),
    "sp_gather_heads_output": (_I, [_PP, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P]),
    "sp_workspace_status": (_I, [_P, _IP, _IP, _IP, _I, _P]),
    "sp_sm_rotation_counts": (_I, [_I, _I, _IP]),
    "sp_exchange_grid": (_I, [_IP]),
    "sp_attention": (_I, [_PP, _PP, _PP, _PP, _I, _I, _I, _I, _I, _I, _I, _I64P, _I64P, _I64P, _I, _P, _F,
                          _P, _Z, _P]),
    "sp_attention_shards": (_I, [_PP, _PP, _PP, _PP, _I, _I, _I, _I, _I, _I, _I, _I, _I64P, _I64P, _I64P, _I, _P,
                                 _F, _P, _Z, _P]),
    "sp_attention_workspace_bytes": (_Z, [_I, _I, _I, _I, _I, _I, _I]),
    "sp_gather_output": (_I, [_PP, _P, _I, _I, _I, _I, _I64, _P]),
    "sp_unpad": (_I, [_P, _P, _I, _I, _I, _I64, _P]),
}

_lock = threading.Lock()
_lib = None


class SPError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{_name(code)}: {msg}")
        self.code = code


class SPValueError(SPError, ValueError):
    """Argument errors (including the partition's not-divisible rule)."""


def _name(code: int) -> str:
    try:
        return lib().sp_status_string(code).decode()
    except Exception:  # pragma: no cover - only while the library is unusable
        return f"status {code}"


def lib() -> ctypes.CDLL:
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(
                    f"{LIB_PATH} is missing: build the CUDA library first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def check(rc: int) -> None:
    if rc == SP_OK:
        return
    msg = lib().sp_last_error().decode(errors="replace")
    if rc in (SP_ERR_NOT_DIVISIBLE, SP_ERR_HEADS_NOT_DIVISIBLE, SP_ERR_INVALID_ARG, SP_ERR_ALIGNMENT,
              SP_ERR_UNSUPPORTED):
        raise SPValueError(rc, msg)
    raise SPError(rc, msg)


def ptr_array(tensors) -> ctypes.Array:
    return (ctypes.c_void_p * len(tensors))(*[int(t.data_ptr()) for t in tensors])


def stream_handle(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(int(s.cuda_stream))

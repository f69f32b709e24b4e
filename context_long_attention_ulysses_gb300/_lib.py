"""ctypes view of libusp.so (declared in include/usp.h).

Loading fails loudly if the library has not been built: there is no CPU or
PyTorch fallback for any entry point.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB

USP_OK = 0
USP_ERR_INVALID_ARG = 1
USP_ERR_UNSUPPORTED = 2
USP_ERR_MISALIGNED = 3
USP_ERR_WORKSPACE = 4
USP_ERR_CUDA = 5
USP_ERR_TIMEOUT = 6

NOALLOC_SCRATCH_BYTES = 64 << 20  # USP_NOALLOC_SCRATCH_BYTES

USP_F32 = 0
USP_BF16 = 1

# every symbol include/usp.h declares
SYMBOLS = (
    "usp_a2a_seq2head", "usp_a2a_head2seq", "usp_attn_fwd", "usp_attn_bwd_workspace_size", "usp_attn_bwd",
    "usp_ring_workspace_size", "usp_ring_attn_fwd", "usp_ring_merge", "usp_device_status", "usp_status_string",
    "usp_build_info", "usp_trace_enable", "usp_trace_reset", "usp_trace_report", "usp_attn_bwd_noalloc",
    "usp_ring_bwd_workspace_size", "usp_ring_attn_bwd", "usp_allgather_workspace_size", "usp_allgather_attn_fwd",
    "usp_allgather_bwd_workspace_size", "usp_allgather_attn_bwd", "usp_zigzag_shard", "usp_zigzag_unshard",
    "usp_zigzag_workspace_size", "usp_zigzag_bwd_workspace_size", "usp_zigzag_attn_fwd", "usp_zigzag_attn_bwd",
    "usp_fused_attn_fwd", "usp_fused_attn_bwd_workspace_size", "usp_fused_attn_bwd", "usp_hybrid_seq2head",
    "usp_hybrid_head2seq", "usp_hybrid_workspace_size", "usp_hybrid_bwd_workspace_size", "usp_hybrid_attn_fwd",
    "usp_hybrid_attn_bwd", "usp_diag_wait_timeout", "usp_diag_raise_status",
    "usp_attn_bwd_deterministic_workspace_size", "usp_attn_bwd_deterministic",
)


class UspProblem(ctypes.Structure):
    """Mirror of ``usp_problem``."""
    _fields_ = [("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("N", ctypes.c_int),
                ("d", ctypes.c_int), ("P", ctypes.c_int), ("causal", ctypes.c_int), ("scale", ctypes.c_float),
                ("dtype", ctypes.c_int)]


class UspTraceEntry(ctypes.Structure):
    """Mirror of ``usp_trace_entry``."""
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int64), ("total_ms", ctypes.c_double)]


class UspError(RuntimeError):
    """A libusp entry point returned a non-OK status."""

    def __init__(self, fn: str, status: int, name: str):
        super().__init__(f"{fn} failed: {name} ({status})")
        self.status = status
        self.fn = fn


_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    """Load libusp.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB):
            raise ImportError(
                f"libusp.so not found at {LIB}; build it first "
                "(python -m context_long_attention_ulysses_gb300.build)")
        lib = ctypes.CDLL(LIB)
        P = ctypes.POINTER(UspProblem)
        vp, i64, sz, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int
        sig = {
            "usp_a2a_seq2head": (ci, [P, ci, vp, vp, vp]),
            "usp_a2a_head2seq": (ci, [P, ci, vp, vp, vp]),
            "usp_attn_fwd": (ci, [P, vp, vp, vp, vp, vp, vp]),
            "usp_attn_bwd_workspace_size": (sz, [P]),
            "usp_attn_bwd": (ci, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
            "usp_ring_workspace_size": (sz, [P]),
            "usp_ring_attn_fwd": (ci, [P, vp, vp, vp, vp, vp, vp, sz, vp]),
            "usp_ring_merge": (ci, [i64, ci, vp, vp, vp, vp, vp, vp, vp]),
            "usp_device_status": (ci, [vp]),
            "usp_status_string": (ctypes.c_char_p, [ci]),
            "usp_build_info": (ctypes.c_char_p, []),
            "usp_trace_enable": (ci, [ci]),
            "usp_trace_reset": (ci, []),
            "usp_trace_report": (ci, [ctypes.POINTER(UspTraceEntry), ci]),
            "usp_attn_bwd_noalloc": (ci, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
            "usp_ring_bwd_workspace_size": (sz, [P]),
            "usp_ring_attn_bwd": (ci, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
            "usp_allgather_workspace_size": (sz, [P]),
            "usp_allgather_attn_fwd": (ci, [P, vp, vp, vp, vp, vp, vp, sz, vp]),
            "usp_allgather_bwd_workspace_size": (sz, [P]),
            "usp_allgather_attn_bwd": (ci, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
            "usp_zigzag_shard": (ci, [P, ci, vp, vp, vp]),
            "usp_zigzag_unshard": (ci, [P, ci, vp, vp, vp]),
            "usp_zigzag_workspace_size": (sz, [P]),
            "usp_zigzag_bwd_workspace_size": (sz, [P]),
            "usp_zigzag_attn_fwd": (ci, [P, vp, vp, vp, vp, vp, vp, sz, vp]),
            "usp_zigzag_attn_bwd": (ci, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
            "usp_fused_attn_fwd": (ci, [P, vp, vp, vp, vp, vp, vp]),
            "usp_fused_attn_bwd_workspace_size": (sz, [P]),
            "usp_fused_attn_bwd": (ci, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
            "usp_hybrid_seq2head": (ci, [P, ci, ci, vp, vp, vp]),
            "usp_hybrid_head2seq": (ci, [P, ci, ci, vp, vp, vp]),
            "usp_hybrid_workspace_size": (sz, [P, ci]),
            "usp_hybrid_bwd_workspace_size": (sz, [P, ci]),
            "usp_hybrid_attn_fwd": (ci, [P, ci, vp, vp, vp, vp, vp, vp, sz, vp]),
            "usp_hybrid_attn_bwd": (ci, [P, ci, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
            "usp_diag_wait_timeout": (ci, [vp]),
            "usp_diag_raise_status": (ci, [vp]),
            "usp_attn_bwd_deterministic_workspace_size": (sz, [P]),
            "usp_attn_bwd_deterministic": (ci, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        }
        for name, (res, args) in sig.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
        return lib


def check(fn: str, status: int) -> None:
    if status != USP_OK:
        name = load().usp_status_string(status).decode()
        raise UspError(fn, status, name)

"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

The generator is Philox4x32-10 (Salmon et al., SC'11) with float64
Box-Muller, written in C in ``philox.c`` and loaded here with ctypes.  It holds
none of the attention arithmetic: it only maps (seed, stream, element index)
to a reproducible N(0,1) sample, rounded to float32 and optionally to bf16
(round to nearest even).

Streams used for the attention inputs (seed 0 by default): Q = 0, K = 1,
V = 2, dO = 3; other streams are free for test-only tensors.

bf16 arrays are returned as ``numpy.uint16`` holding the raw bf16 bits.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "philox.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libsynth.so")
_lock = threading.Lock()
_lib = None

STREAM_Q, STREAM_K, STREAM_V, STREAM_DO = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile ``philox.c`` into ``_build/libsynth.so`` (gcc, -O2, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
             "-pthread", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.synth_normal.restype = ctypes.c_int
            lib.synth_normal.argtypes = [
                ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_uint64,
                ctypes.c_int, ctypes.c_double, ctypes.c_void_p, ctypes.c_int]
            lib.synth_philox4x32_10.restype = None
            lib.synth_philox4x32_10.argtypes = [ctypes.c_void_p] * 3
            _lib = lib
    return _lib


def _threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def philox4x32_10(counter, key) -> np.ndarray:
    """Raw Philox4x32-10 block: four uint32 words for a counter and a key."""
    c = np.ascontiguousarray(np.asarray(counter, dtype=np.uint32).reshape(4))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32).reshape(2))
    out = np.zeros(4, dtype=np.uint32)
    _load().synth_philox4x32_10(c.ctypes.data, k.ctypes.data, out.ctypes.data)
    return out


def normal(shape, seed: int = 0, stream: int = 0, dtype: str = "f32",
           scale: float = 1.0, offset: int = 0, out: np.ndarray | None = None) -> np.ndarray:
    """N(0,1) * scale samples of the (seed, stream) sequence in row-major order.

    dtype "f32" returns float32; "bf16" returns uint16 bf16 bits.
    ``offset`` skips that many elements of the sequence.
    """
    shape = tuple(int(s) for s in (shape if isinstance(shape, (tuple, list)) else (shape,)))
    n = int(np.prod(shape)) if shape else 1
    if dtype == "f32":
        code, npdt = 0, np.float32
    elif dtype == "bf16":
        code, npdt = 1, np.uint16
    else:
        raise ValueError(f"dtype must be 'f32' or 'bf16', got {dtype!r}")
    if out is None:
        out = np.empty(shape, dtype=npdt)
    elif out.dtype != npdt or not out.flags.c_contiguous or out.size != n:
        raise ValueError("out must be a C-contiguous array of the right dtype and size")
    rc = _load().synth_normal(int(seed), int(stream), int(offset), n, code, float(scale),
                              out.ctypes.data, _threads())
    if rc != 0:
        raise RuntimeError(f"synth_normal failed with code {rc}")
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of raw bf16 bits (uint16) to float32."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bits, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)

"""ORACLE -- TEST INFRASTRUCTURE ONLY.

Plain float64 CPU definitions of the Ulysses sequence-parallel attention path
(layout maps, causal/GQA attention forward, its gradients, the partial merge
of ring attention).  The arithmetic lives in ``attn_oracle.c`` (plain C,
float64, threads only split independent rows); this module compiles it with
gcc and marshals numpy arrays to it.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package.  It shares no code with the CUDA path.

``rows_blas`` restates the attention rows and gradients with numpy matrix
products as the library step, for sampled rows of long sequences.

Parity pins: every function here is checked by ``tests/test_oracle.py``
against closed forms, library special cases, brute force and finite
differences (see that file); no function is unpinned.

Tensors are numpy arrays: float32, or uint16 holding raw bf16 bits.  The
logical layout is [B][H][N][d] (sequence at dimension 2, as in the code
example of the "Context Parallelism" glossary page).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_c_long = ctypes.c_long
_c_int = ctypes.c_int
_vp = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-pthread", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            for name in ("orc_shard_seq", "orc_unshard_seq", "orc_seq2head", "orc_head2seq"):
                f = getattr(lib, name)
                f.restype = _c_int
                f.argtypes = [_c_int, _c_int, _c_long, _c_int, _c_int, _c_int, _vp, _vp]
            lib.orc_attn_rows.restype = _c_int
            lib.orc_attn_rows.argtypes = [_c_int, _c_int, _c_int, _c_long, _c_int, _vp, _vp, _vp,
                                          _c_int, _c_int, ctypes.c_double, _c_long, _c_long, _c_long,
                                          _vp, _vp, _vp, _c_int]
            lib.orc_attn_bwd_q_rows.restype = _c_int
            lib.orc_attn_bwd_q_rows.argtypes = [_c_int, _c_int, _c_int, _c_long, _c_int, _vp, _vp, _vp,
                                                _vp, _c_int, _c_int, _c_int, ctypes.c_double, _c_long, _vp,
                                                _vp, _c_int]
            lib.orc_attn_bwd_kv_rows.restype = _c_int
            lib.orc_attn_bwd_kv_rows.argtypes = [_c_int, _c_int, _c_int, _c_long, _c_int, _vp, _vp, _vp,
                                                 _vp, _c_int, _c_int, _c_int, ctypes.c_double, _vp, _vp,
                                                 _c_long, _vp, _vp, _vp, _c_int]
            lib.orc_lse_merge.restype = None
            lib.orc_lse_merge.argtypes = [_c_long, _c_int, _vp, _vp, _vp, _vp, _vp, _vp]
            _lib = lib
    return _lib


def threads() -> int:
    """Host threads the oracle uses (the process affinity mask)."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _dtype_code(x: np.ndarray) -> int:
    if x.dtype == np.float32:
        return 0
    if x.dtype == np.uint16:
        return 1
    raise TypeError(f"oracle inputs are float32 or uint16 (bf16 bits), got {x.dtype}")


def _c(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x)


# ---------------------------------------------------------------- layout maps
def _map(fn_name: str, x: np.ndarray, out_shape, B, H, N, d, P) -> np.ndarray:
    x = _c(x)
    out = np.empty(out_shape, dtype=x.dtype)
    rc = getattr(_load(), fn_name)(B, H, N, d, P, x.itemsize, x.ctypes.data, out.ctypes.data)
    if rc != 0:
        raise ValueError(f"{fn_name}: bad sizes (B={B}, H={H}, N={N}, d={d}, P={P})")
    return out


def shard_seq(x: np.ndarray, P: int) -> np.ndarray:
    """logical [B][H][N][d] -> sequence-sharded [P][B][N/P][H][d]."""
    B, H, N, d = x.shape
    return _map("orc_shard_seq", x, (P, B, N // P, H, d), B, H, N, d, P)


def unshard_seq(x: np.ndarray) -> np.ndarray:
    """sequence-sharded [P][B][N/P][H][d] -> logical [B][H][N][d]."""
    P, B, Np, H, d = x.shape
    return _map("orc_unshard_seq", x, (B, H, Np * P, d), B, H, Np * P, d, P)


def seq2head(x: np.ndarray) -> np.ndarray:
    """All-to-all: sequence-sharded [P][B][N/P][H][d] -> head-sharded [P][B][H/P][N][d]."""
    P, B, Np, H, d = x.shape
    return _map("orc_seq2head", x, (P, B, H // P, Np * P, d), B, H, Np * P, d, P)


def head2seq(x: np.ndarray) -> np.ndarray:
    """All-to-all back: head-sharded [P][B][H/P][N][d] -> sequence-sharded [P][B][N/P][H][d]."""
    P, B, Hl, N, d = x.shape
    return _map("orc_head2seq", x, (P, B, N // P, Hl * P, d), B, Hl * P, N, d, P)


# ------------------------------------------------------------------ attention
def attn_rows(q, k, v, rows=None, causal=True, scale=None, key_lo=0, key_hi=None, nthreads=None):
    """O and LSE (natural log) of the selected query rows, float64.

    q: [B][Hq][N][d]; k, v: [B][Hkv][N][d].  rows: query positions (default
    all).  Keys restricted to [key_lo, key_hi) and, if causal, j <= i.
    Returns (o [B][Hq][nrows][d], lse [B][Hq][nrows]).
    """
    q, k, v = _c(q), _c(k), _c(v)
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (B, Hkv, N, d) or v.shape != k.shape or q.dtype != k.dtype or v.dtype != k.dtype:
        raise ValueError("shape/dtype mismatch")
    rows = np.arange(N, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    key_hi = N if key_hi is None else int(key_hi)
    o = np.empty((B, Hq, len(rows), d), dtype=np.float64)
    lse = np.empty((B, Hq, len(rows)), dtype=np.float64)
    rc = _load().orc_attn_rows(B, Hq, Hkv, N, d, q.ctypes.data, k.ctypes.data, v.ctypes.data,
                               _dtype_code(q), int(bool(causal)), scale, int(key_lo), key_hi,
                               len(rows), rows.ctypes.data, o.ctypes.data, lse.ctypes.data,
                               nthreads or threads())
    if rc != 0:
        raise ValueError("orc_attn_rows: bad arguments")
    return o, lse


def attn_bwd_q_rows(q, k, v, dout, rows=None, causal=True, scale=None, nthreads=None):
    """dQ of the selected query rows for upstream gradient dO, float64 [B][Hq][nrows][d].

    dO may be float32 or bf16 bits independently of Q, K, V.
    """
    q, k, v, dout = _c(q), _c(k), _c(v), _c(dout)
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    if dout.shape != q.shape:
        raise ValueError("dO must match Q in shape")
    rows = np.arange(N, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    dq = np.empty((B, Hq, len(rows), d), dtype=np.float64)
    rc = _load().orc_attn_bwd_q_rows(B, Hq, Hkv, N, d, q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                     dout.ctypes.data, _dtype_code(q), _dtype_code(dout), int(bool(causal)),
                                     scale, len(rows), rows.ctypes.data, dq.ctypes.data, nthreads or threads())
    if rc != 0:
        raise ValueError("orc_attn_bwd_q_rows: bad arguments")
    return dq


def attn_bwd_kv_rows(q, k, v, dout, lse, dvec, rows=None, causal=True, scale=None, nthreads=None):
    """dK, dV of the selected key rows (summed over each KV head's query group).

    lse, dvec: [B][Hq][N] float64 arrays of LSE_i and D_i = dO_i . O_i; only
    rows i that see a selected key are read.  Returns (dk, dv), each
    [B][Hkv][nrows][d] float64.
    """
    q, k, v, dout = _c(q), _c(k), _c(v), _c(dout)
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    lse = np.ascontiguousarray(lse, dtype=np.float64)
    dvec = np.ascontiguousarray(dvec, dtype=np.float64)
    if lse.shape != (B, Hq, N) or dvec.shape != (B, Hq, N):
        raise ValueError("lse/dvec must be [B][Hq][N]")
    rows = np.arange(N, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    dk = np.empty((B, Hkv, len(rows), d), dtype=np.float64)
    dv = np.empty((B, Hkv, len(rows), d), dtype=np.float64)
    rc = _load().orc_attn_bwd_kv_rows(B, Hq, Hkv, N, d, q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                      dout.ctypes.data, _dtype_code(q), _dtype_code(dout), int(bool(causal)),
                                      scale, lse.ctypes.data, dvec.ctypes.data, len(rows), rows.ctypes.data,
                                      dk.ctypes.data, dv.ctypes.data, nthreads or threads())
    if rc != 0:
        raise ValueError("orc_attn_bwd_kv_rows: bad arguments")
    return dk, dv


def attn_bwd_full(q, k, v, dout, causal=True, scale=None, nthreads=None):
    """Every gradient of every row (small problems): (dq, dk, dv, o, lse), float64."""
    B, Hq, N, d = q.shape
    o, lse = attn_rows(q, k, v, None, causal, scale, nthreads=nthreads)
    dof = _as_f64(dout)
    dvec = np.einsum("bhnd,bhnd->bhn", dof, o)
    dq = attn_bwd_q_rows(q, k, v, dout, None, causal, scale, nthreads)
    dk, dv = attn_bwd_kv_rows(q, k, v, dout, lse, dvec, None, causal, scale, nthreads)
    return dq, dk, dv, o, lse


def lse_merge(o_a, lse_a, o_b, lse_b):
    """Exact merge of two partial attentions over disjoint key sets (float64)."""
    o_a = np.ascontiguousarray(o_a, dtype=np.float64)
    o_b = np.ascontiguousarray(o_b, dtype=np.float64)
    lse_a = np.ascontiguousarray(lse_a, dtype=np.float64)
    lse_b = np.ascontiguousarray(lse_b, dtype=np.float64)
    d = o_a.shape[-1]
    rows = lse_a.size
    if o_a.shape != o_b.shape or lse_a.shape != lse_b.shape or o_a.size != rows * d:
        raise ValueError("shape mismatch")
    o = np.empty_like(o_a)
    lse = np.empty_like(lse_a)
    _load().orc_lse_merge(rows, d, o_a.ctypes.data, lse_a.ctypes.data, o_b.ctypes.data,
                          lse_b.ctypes.data, o.ctypes.data, lse.ctypes.data)
    return o, lse


def _as_f64(x: np.ndarray) -> np.ndarray:
    if x.dtype == np.uint16:
        return (np.ascontiguousarray(x).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.asarray(x, dtype=np.float64)


def as_f64(x: np.ndarray) -> np.ndarray:
    """Exact float64 value of a float32 or bf16-bits array."""
    return _as_f64(x)

"""Ulysses sequence-parallel attention on one GB300 -- Python binding of libusp.

The functions named ``usp_*`` mirror the C ABI in ``include/usp.h`` one to
one: they only marshal arguments (torch tensors or raw device pointers, the
current torch stream) and raise :class:`UspError` on a non-OK status.  Every
step of the computation runs in libusp's CUDA kernels; PyTorch provides
device memory and streams.

The helpers ``ulysses_attention_fwd``/``ulysses_attention_bwd`` and
``ring_attention_fwd`` chain those calls the way one sequence-parallel
attention layer does (all-to-all, attention, all-to-all back) and allocate
their outputs with torch.
"""
from __future__ import annotations

import ctypes
import math
from dataclasses import dataclass

import torch

from ._lib import (NOALLOC_SCRATCH_BYTES, SYMBOLS, USP_BF16, USP_F32, USP_OK, UspError, UspProblem,  # noqa: F401
                   UspTraceEntry, check, load)

__all__ = [
    "Problem", "UspError", "SYMBOLS",
    "usp_a2a_seq2head", "usp_a2a_head2seq", "usp_attn_fwd", "usp_attn_bwd_workspace_size", "usp_attn_bwd",
    "usp_ring_workspace_size", "usp_ring_attn_fwd", "usp_ring_merge", "usp_device_status", "usp_status_string",
    "usp_build_info", "usp_trace_enable", "usp_trace_reset", "usp_trace_report", "usp_attn_bwd_noalloc",
    "NOALLOC_SCRATCH_BYTES", "ulysses_attention_fwd", "ulysses_attention_bwd", "ring_attention_fwd", "library_path",
    "usp_ring_bwd_workspace_size", "usp_ring_attn_bwd", "ring_attention_bwd",
    "usp_allgather_workspace_size", "usp_allgather_attn_fwd", "usp_allgather_bwd_workspace_size",
    "usp_allgather_attn_bwd", "allgather_attention_fwd", "allgather_attention_bwd",
    "usp_zigzag_shard", "usp_zigzag_unshard", "usp_zigzag_workspace_size", "usp_zigzag_bwd_workspace_size",
    "usp_zigzag_attn_fwd", "usp_zigzag_attn_bwd", "zigzag_attention_fwd", "zigzag_attention_bwd",
    "usp_fused_attn_fwd", "usp_fused_attn_bwd_workspace_size", "usp_fused_attn_bwd", "fused_attention_fwd",
    "fused_attention_bwd", "usp_hybrid_seq2head", "usp_hybrid_head2seq", "usp_hybrid_workspace_size",
    "usp_hybrid_bwd_workspace_size", "usp_hybrid_attn_fwd", "usp_hybrid_attn_bwd", "hybrid_attention_fwd",
    "hybrid_attention_bwd", "usp_diag_wait_timeout", "usp_diag_raise_status",
    "usp_attn_bwd_deterministic_workspace_size", "usp_attn_bwd_deterministic",
]

_TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Problem:
    """Q: B x Hq x N x d, K/V: B x Hkv x N x d, sequence-parallel degree P."""
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    P: int
    causal: bool = True
    scale: float = 0.0  # 0 selects 1/sqrt(d)
    dtype: str = "bf16"

    def c(self) -> UspProblem:
        if self.dtype not in _TORCH_DTYPE:
            raise ValueError(f"dtype must be 'f32' or 'bf16', got {self.dtype!r}")
        return UspProblem(self.B, self.Hq, self.Hkv, self.N, self.d, self.P, int(bool(self.causal)),
                          float(self.scale), USP_F32 if self.dtype == "f32" else USP_BF16)

    @property
    def torch_dtype(self) -> torch.dtype:
        return _TORCH_DTYPE[self.dtype]

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale else 1.0 / math.sqrt(self.d)

    def seq_shape(self, H: int):
        """Sequence-sharded layout [P][B][N/P][H][d]."""
        return (self.P, self.B, self.N // self.P, H, self.d)

    def head_shape(self, H: int):
        """Head-sharded layout [P][B][H/P][N][d]."""
        return (self.P, self.B, H // self.P, self.N, self.d)

    def lse_head_shape(self):
        return (self.P, self.B, self.Hq // self.P, self.N)

    def lse_seq_shape(self):
        return (self.P, self.B, self.N // self.P, self.Hq)

    def hybrid_shape(self, H: int, Pu: int):
        """2-D layout [P][B][H/Pu][N/Pr][d] (Pr = P/Pu ring groups of Pu Ulysses ranks)."""
        return (self.P, self.B, H // Pu, self.N // (self.P // Pu), self.d)

    def lse_hybrid_shape(self, Pu: int):
        return (self.P, self.B, self.Hq // Pu, self.N // (self.P // Pu))


def library_path() -> str:
    from .build import LIB
    return LIB


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if isinstance(x, torch.Tensor):
        if x.numel() and not x.is_cuda:
            raise ValueError("libusp takes device tensors")
        if not x.is_contiguous():
            raise ValueError("libusp takes contiguous tensors")
        return x.data_ptr()
    raise TypeError(f"expected a torch tensor, a device pointer or None, got {type(x).__name__}")


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else 0
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _prob(p) -> ctypes.POINTER(UspProblem):
    if p is None:
        return None
    return ctypes.byref(p.c() if isinstance(p, Problem) else p)


# --------------------------------------------------------------- C ABI mirror
def usp_a2a_seq2head(p, Hx: int, src, dst, stream=None) -> None:
    check("usp_a2a_seq2head", load().usp_a2a_seq2head(_prob(p), Hx, _ptr(src), _ptr(dst), _stream(stream)))


def usp_a2a_head2seq(p, Hx: int, src, dst, stream=None) -> None:
    check("usp_a2a_head2seq", load().usp_a2a_head2seq(_prob(p), Hx, _ptr(src), _ptr(dst), _stream(stream)))


def usp_attn_fwd(p, q, k, v, o, lse, stream=None) -> None:
    check("usp_attn_fwd", load().usp_attn_fwd(_prob(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                              _stream(stream)))


def usp_attn_bwd_workspace_size(p) -> int:
    return int(load().usp_attn_bwd_workspace_size(_prob(p)))


def usp_attn_bwd(p, q, k, v, o, lse, dout, dq, dk, dv, ws, ws_bytes=None, stream=None) -> None:
    if ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size() if isinstance(ws, torch.Tensor) else 0
    check("usp_attn_bwd", load().usp_attn_bwd(_prob(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
                                              _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), int(ws_bytes),
                                              _stream(stream)))


def usp_attn_bwd_deterministic_workspace_size(p) -> int:
    return int(load().usp_attn_bwd_deterministic_workspace_size(_prob(p)))


def usp_attn_bwd_deterministic(p, q, k, v, o, lse, dout, dq, dk, dv, ws, ws_bytes=None, stream=None) -> None:
    if ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size() if isinstance(ws, torch.Tensor) else 0
    check("usp_attn_bwd_deterministic",
          load().usp_attn_bwd_deterministic(_prob(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
                                            _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), int(ws_bytes), _stream(stream)))


def usp_attn_bwd_noalloc(p, q, k, v, o, lse, dout, dq, dk, dv, stream=None) -> None:
    """usp_attn_bwd_deterministic with the library's built-in scratch instead of a workspace.

    For callers that cannot allocate device memory.  Problems needing more
    than NOALLOC_SCRATCH_BYTES of workspace raise UspError (USP_ERR_WORKSPACE);
    calls that may overlap on the GPU share the scratch and must be serialised.
    """
    check("usp_attn_bwd_noalloc", load().usp_attn_bwd_noalloc(_prob(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                                              _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                                                              _stream(stream)))


def usp_ring_workspace_size(p) -> int:
    return int(load().usp_ring_workspace_size(_prob(p)))


def usp_ring_attn_fwd(p, q, k, v, o, lse, ws, ws_bytes=None, stream=None) -> None:
    if ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size() if isinstance(ws, torch.Tensor) else 0
    check("usp_ring_attn_fwd", load().usp_ring_attn_fwd(_prob(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                                        _ptr(ws), int(ws_bytes), _stream(stream)))


def usp_ring_bwd_workspace_size(p) -> int:
    return int(load().usp_ring_bwd_workspace_size(_prob(p)))


def usp_ring_attn_bwd(p, q, k, v, o, lse, dout, dq, dk, dv, ws, ws_bytes=None, stream=None) -> None:
    if ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size() if isinstance(ws, torch.Tensor) else 0
    check("usp_ring_attn_bwd", load().usp_ring_attn_bwd(_prob(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                                        _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws),
                                                        int(ws_bytes), _stream(stream)))


def usp_allgather_workspace_size(p) -> int:
    return int(load().usp_allgather_workspace_size(_prob(p)))


def usp_allgather_attn_fwd(p, q, k, v, o, lse, ws, ws_bytes=None, stream=None) -> None:
    if ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size() if isinstance(ws, torch.Tensor) else 0
    check("usp_allgather_attn_fwd", load().usp_allgather_attn_fwd(_prob(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                                                  _ptr(lse), _ptr(ws), int(ws_bytes), _stream(stream)))


def usp_allgather_bwd_workspace_size(p) -> int:
    return int(load().usp_allgather_bwd_workspace_size(_prob(p)))


def usp_allgather_attn_bwd(p, q, k, v, o, lse, dout, dq, dk, dv, ws, ws_bytes=None, stream=None) -> None:
    if ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size() if isinstance(ws, torch.Tensor) else 0
    check("usp_allgather_attn_bwd", load().usp_allgather_attn_bwd(_prob(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                                                  _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                                                                  _ptr(ws), int(ws_bytes), _stream(stream)))


def usp_zigzag_shard(p, hx: int, src, dst, stream=None) -> None:
    check("usp_zigzag_shard", load().usp_zigzag_shard(_prob(p), int(hx), _ptr(src), _ptr(dst), _stream(stream)))


def usp_zigzag_unshard(p, hx: int, src, dst, stream=None) -> None:
    check("usp_zigzag_unshard", load().usp_zigzag_unshard(_prob(p), int(hx), _ptr(src), _ptr(dst), _stream(stream)))


def usp_zigzag_workspace_size(p) -> int:
    return int(load().usp_zigzag_workspace_size(_prob(p)))


def usp_zigzag_bwd_workspace_size(p) -> int:
    return int(load().usp_zigzag_bwd_workspace_size(_prob(p)))


def usp_zigzag_attn_fwd(p, q, k, v, o, lse, ws, ws_bytes=None, stream=None) -> None:
    if ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size() if isinstance(ws, torch.Tensor) else 0
    check("usp_zigzag_attn_fwd", load().usp_zigzag_attn_fwd(_prob(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                                            _ptr(ws), int(ws_bytes), _stream(stream)))


def usp_zigzag_attn_bwd(p, q, k, v, o, lse, dout, dq, dk, dv, ws, ws_bytes=None, stream=None) -> None:
    if ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size() if isinstance(ws, torch.Tensor) else 0
    check("usp_zigzag_attn_bwd", load().usp_zigzag_attn_bwd(_prob(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                                            _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws),
                                                            int(ws_bytes), _stream(stream)))


def usp_fused_attn_fwd(p, q, k, v, o, lse, stream=None) -> None:
    check("usp_fused_attn_fwd", load().usp_fused_attn_fwd(_prob(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                                           _stream(stream)))


def usp_fused_attn_bwd_workspace_size(p) -> int:
    return int(load().usp_fused_attn_bwd_workspace_size(_prob(p)))


def usp_fused_attn_bwd(p, q, k, v, o, lse, dout, dq, dk, dv, ws, ws_bytes=None, stream=None) -> None:
    if ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size() if isinstance(ws, torch.Tensor) else 0
    check("usp_fused_attn_bwd", load().usp_fused_attn_bwd(_prob(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                                           _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws),
                                                           int(ws_bytes), _stream(stream)))


def usp_hybrid_seq2head(p, Pu: int, Hx: int, src, dst, stream=None) -> None:
    check("usp_hybrid_seq2head", load().usp_hybrid_seq2head(_prob(p), int(Pu), int(Hx), _ptr(src), _ptr(dst),
                                                             _stream(stream)))


def usp_hybrid_head2seq(p, Pu: int, Hx: int, src, dst, stream=None) -> None:
    check("usp_hybrid_head2seq", load().usp_hybrid_head2seq(_prob(p), int(Pu), int(Hx), _ptr(src), _ptr(dst),
                                                             _stream(stream)))


def usp_hybrid_workspace_size(p, Pu: int) -> int:
    return int(load().usp_hybrid_workspace_size(_prob(p), int(Pu)))


def usp_hybrid_bwd_workspace_size(p, Pu: int) -> int:
    return int(load().usp_hybrid_bwd_workspace_size(_prob(p), int(Pu)))


def usp_hybrid_attn_fwd(p, Pu: int, q, k, v, o, lse, ws, ws_bytes=None, stream=None) -> None:
    if ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size() if isinstance(ws, torch.Tensor) else 0
    check("usp_hybrid_attn_fwd", load().usp_hybrid_attn_fwd(_prob(p), int(Pu), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                                             _ptr(lse), _ptr(ws), int(ws_bytes), _stream(stream)))


def usp_hybrid_attn_bwd(p, Pu: int, q, k, v, o, lse, dout, dq, dk, dv, ws, ws_bytes=None, stream=None) -> None:
    if ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size() if isinstance(ws, torch.Tensor) else 0
    check("usp_hybrid_attn_bwd", load().usp_hybrid_attn_bwd(_prob(p), int(Pu), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                                             _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                                                             _ptr(ws), int(ws_bytes), _stream(stream)))


def usp_ring_merge(rows: int, d: int, o_a, lse_a, o_b, lse_b, o, lse, stream=None) -> None:
    check("usp_ring_merge", load().usp_ring_merge(int(rows), int(d), _ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b),
                                                  _ptr(o), _ptr(lse), _stream(stream)))


def usp_diag_wait_timeout(stream=None) -> None:
    check("usp_diag_wait_timeout", load().usp_diag_wait_timeout(_stream(stream)))


def usp_diag_raise_status(stream=None) -> None:
    check("usp_diag_raise_status", load().usp_diag_raise_status(_stream(stream)))


def usp_device_status(stream=None) -> int:
    return int(load().usp_device_status(_stream(stream)))


def usp_status_string(s: int) -> str:
    return load().usp_status_string(int(s)).decode()


def usp_build_info() -> str:
    return load().usp_build_info().decode()


def usp_trace_enable(on: bool = True) -> None:
    check("usp_trace_enable", load().usp_trace_enable(1 if on else 0))


def usp_trace_reset() -> None:
    check("usp_trace_reset", load().usp_trace_reset())


def usp_trace_report() -> dict:
    """{kernel name: (launches, total milliseconds)} accumulated since the last reset."""
    lib = load()
    n = lib.usp_trace_report(None, 0)
    if n < 0:
        raise UspError("usp_trace_report", n, "event failure")
    buf = (UspTraceEntry * max(n, 1))()
    n = lib.usp_trace_report(buf, n)
    return {buf[i].name.decode(): (int(buf[i].launches), float(buf[i].total_ms)) for i in range(n)}


# ------------------------------------------------------------ layer helpers
def _empty(shape, dtype, device):
    return torch.empty(shape, dtype=dtype, device=device)


def ulysses_attention_fwd(p: Problem, q_seq, k_seq, v_seq, stream=None):
    """One Ulysses attention forward on sequence-sharded Q, K, V.

    seq->head all-to-all of Q, K, V; attention per rank; head->seq all-to-all
    of O.  Returns (o_seq, saved) where ``saved`` holds the head-sharded
    tensors and LSE the backward needs.
    """
    dev, dt = q_seq.device, p.torch_dtype
    qh = _empty(p.head_shape(p.Hq), dt, dev)
    kh = _empty(p.head_shape(p.Hkv), dt, dev)
    vh = _empty(p.head_shape(p.Hkv), dt, dev)
    oh = _empty(p.head_shape(p.Hq), dt, dev)
    lse = _empty(p.lse_head_shape(), torch.float32, dev)
    o_seq = _empty(p.seq_shape(p.Hq), dt, dev)
    usp_a2a_seq2head(p, p.Hq, q_seq, qh, stream)
    usp_a2a_seq2head(p, p.Hkv, k_seq, kh, stream)
    usp_a2a_seq2head(p, p.Hkv, v_seq, vh, stream)
    usp_attn_fwd(p, qh, kh, vh, oh, lse, stream)
    usp_a2a_head2seq(p, p.Hq, oh, o_seq, stream)
    return o_seq, {"q": qh, "k": kh, "v": vh, "o": oh, "lse": lse}


def ulysses_attention_bwd(p: Problem, saved, do_seq, stream=None, deterministic=False):
    """Backward of :func:`ulysses_attention_fwd` for upstream gradient dO (sequence-sharded).

    Returns (dq_seq, dk_seq, dv_seq).  deterministic=True runs the bit-reproducible three-pass
    backward (usp_attn_bwd_deterministic) instead of the one-pass one.
    """
    dev, dt = do_seq.device, p.torch_dtype
    doh = _empty(p.head_shape(p.Hq), dt, dev)
    dqh = _empty(p.head_shape(p.Hq), dt, dev)
    dkh = _empty(p.head_shape(p.Hkv), dt, dev)
    dvh = _empty(p.head_shape(p.Hkv), dt, dev)
    size = usp_attn_bwd_deterministic_workspace_size(p) if deterministic else usp_attn_bwd_workspace_size(p)
    ws = torch.empty(max(size, 256), dtype=torch.uint8, device=dev)
    usp_a2a_seq2head(p, p.Hq, do_seq, doh, stream)
    bwd = usp_attn_bwd_deterministic if deterministic else usp_attn_bwd
    bwd(p, saved["q"], saved["k"], saved["v"], saved["o"], saved["lse"], doh, dqh, dkh, dvh, ws, None, stream)
    dq = _empty(p.seq_shape(p.Hq), dt, dev)
    dk = _empty(p.seq_shape(p.Hkv), dt, dev)
    dv = _empty(p.seq_shape(p.Hkv), dt, dev)
    usp_a2a_head2seq(p, p.Hq, dqh, dq, stream)
    usp_a2a_head2seq(p, p.Hkv, dkh, dk, stream)
    usp_a2a_head2seq(p, p.Hkv, dvh, dv, stream)
    return dq, dk, dv


def ring_attention_fwd(p: Problem, q_seq, k_seq, v_seq, stream=None):
    """Ring attention forward on sequence-sharded buffers: returns (o_seq, lse_seq)."""
    dev, dt = q_seq.device, p.torch_dtype
    o = _empty(p.seq_shape(p.Hq), dt, dev)
    lse = _empty(p.lse_seq_shape(), torch.float32, dev)
    ws = torch.empty(max(usp_ring_workspace_size(p), 256), dtype=torch.uint8, device=dev)
    usp_ring_attn_fwd(p, q_seq, k_seq, v_seq, o, lse, ws, None, stream)
    return o, lse


def allgather_attention_fwd(p: Problem, q_seq, k_seq, v_seq, stream=None):
    """All-gather-KV attention forward on sequence-sharded buffers: returns (o_seq, lse_seq)."""
    dev, dt = q_seq.device, p.torch_dtype
    o = _empty(p.seq_shape(p.Hq), dt, dev)
    lse = _empty(p.lse_seq_shape(), torch.float32, dev)
    ws = torch.empty(max(usp_allgather_workspace_size(p), 256), dtype=torch.uint8, device=dev)
    usp_allgather_attn_fwd(p, q_seq, k_seq, v_seq, o, lse, ws, None, stream)
    return o, lse


def allgather_attention_bwd(p: Problem, q_seq, k_seq, v_seq, o_seq, lse_seq, dout_seq, stream=None):
    """All-gather-KV attention backward on sequence-sharded buffers: returns (dq_seq, dk_seq, dv_seq)."""
    dev = q_seq.device
    dq, dk, dv = torch.empty_like(q_seq), torch.empty_like(k_seq), torch.empty_like(v_seq)
    ws = torch.empty(max(usp_allgather_bwd_workspace_size(p), 256), dtype=torch.uint8, device=dev)
    usp_allgather_attn_bwd(p, q_seq, k_seq, v_seq, o_seq, lse_seq, dout_seq, dq, dk, dv, ws, None, stream)
    return dq, dk, dv


def zigzag_attention_fwd(p: Problem, q_zz, k_zz, v_zz, stream=None):
    """Zigzag ring attention forward on zigzag-sharded buffers: returns (o_zz, lse_zz)."""
    dev, dt = q_zz.device, p.torch_dtype
    o = _empty(p.seq_shape(p.Hq), dt, dev)
    lse = _empty(p.lse_seq_shape(), torch.float32, dev)
    ws = torch.empty(max(usp_zigzag_workspace_size(p), 256), dtype=torch.uint8, device=dev)
    usp_zigzag_attn_fwd(p, q_zz, k_zz, v_zz, o, lse, ws, None, stream)
    return o, lse


def zigzag_attention_bwd(p: Problem, q_zz, k_zz, v_zz, o_zz, lse_zz, dout_zz, stream=None):
    """Zigzag ring attention backward on zigzag-sharded buffers: returns (dq, dk, dv), zigzag-sharded."""
    dev = q_zz.device
    dq, dk, dv = torch.empty_like(q_zz), torch.empty_like(k_zz), torch.empty_like(v_zz)
    ws = torch.empty(max(usp_zigzag_bwd_workspace_size(p), 256), dtype=torch.uint8, device=dev)
    usp_zigzag_attn_bwd(p, q_zz, k_zz, v_zz, o_zz, lse_zz, dout_zz, dq, dk, dv, ws, None, stream)
    return dq, dk, dv


def ring_attention_bwd(p: Problem, q_seq, k_seq, v_seq, o_seq, lse_seq, dout_seq, stream=None):
    """Ring attention backward on sequence-sharded buffers: returns (dq_seq, dk_seq, dv_seq)."""
    dev = q_seq.device
    dq, dk, dv = torch.empty_like(q_seq), torch.empty_like(k_seq), torch.empty_like(v_seq)
    ws = torch.empty(max(usp_ring_bwd_workspace_size(p), 256), dtype=torch.uint8, device=dev)
    usp_ring_attn_bwd(p, q_seq, k_seq, v_seq, o_seq, lse_seq, dout_seq, dq, dk, dv, ws, None, stream)
    return dq, dk, dv


def fused_attention_fwd(p: Problem, q_seq, k_seq, v_seq, stream=None):
    """Ulysses attention with the all-to-all fused into the kernels: sequence-sharded Q, K, V in,
    returns (o_seq, lse_seq) with the LSE as [P][B][N/P][Hq]."""
    dev, dt = q_seq.device, p.torch_dtype
    o = _empty(p.seq_shape(p.Hq), dt, dev)
    lse = _empty(p.lse_seq_shape(), torch.float32, dev)
    usp_fused_attn_fwd(p, q_seq, k_seq, v_seq, o, lse, stream)
    return o, lse


def fused_attention_bwd(p: Problem, q_seq, k_seq, v_seq, o_seq, lse_seq, dout_seq, stream=None):
    """Backward of :func:`fused_attention_fwd`: returns (dq_seq, dk_seq, dv_seq)."""
    dev = q_seq.device
    dq, dk, dv = torch.empty_like(q_seq), torch.empty_like(k_seq), torch.empty_like(v_seq)
    ws = torch.empty(max(usp_fused_attn_bwd_workspace_size(p), 256), dtype=torch.uint8, device=dev)
    usp_fused_attn_bwd(p, q_seq, k_seq, v_seq, o_seq, lse_seq, dout_seq, dq, dk, dv, ws, None, stream)
    return dq, dk, dv


def hybrid_attention_fwd(p: Problem, Pu: int, q_seq, k_seq, v_seq, stream=None):
    """2-D sequence parallelism forward: all-to-all inside each group of Pu ranks, ring attention
    across the P/Pu groups, all-to-all back.  Sequence-sharded in and out; returns (o_seq, saved)
    with the hybrid-layout tensors and LSE the backward needs."""
    dev, dt = q_seq.device, p.torch_dtype
    qh = _empty(p.hybrid_shape(p.Hq, Pu), dt, dev)
    kh = _empty(p.hybrid_shape(p.Hkv, Pu), dt, dev)
    vh = _empty(p.hybrid_shape(p.Hkv, Pu), dt, dev)
    oh = _empty(p.hybrid_shape(p.Hq, Pu), dt, dev)
    lse = _empty(p.lse_hybrid_shape(Pu), torch.float32, dev)
    o_seq = _empty(p.seq_shape(p.Hq), dt, dev)
    ws = torch.empty(max(usp_hybrid_workspace_size(p, Pu), 256), dtype=torch.uint8, device=dev)
    usp_hybrid_seq2head(p, Pu, p.Hq, q_seq, qh, stream)
    usp_hybrid_seq2head(p, Pu, p.Hkv, k_seq, kh, stream)
    usp_hybrid_seq2head(p, Pu, p.Hkv, v_seq, vh, stream)
    usp_hybrid_attn_fwd(p, Pu, qh, kh, vh, oh, lse, ws, None, stream)
    usp_hybrid_head2seq(p, Pu, p.Hq, oh, o_seq, stream)
    return o_seq, {"q": qh, "k": kh, "v": vh, "o": oh, "lse": lse}


def hybrid_attention_bwd(p: Problem, Pu: int, saved, do_seq, stream=None):
    """Backward of :func:`hybrid_attention_fwd` for upstream gradient dO (sequence-sharded).

    Returns (dq_seq, dk_seq, dv_seq)."""
    dev, dt = do_seq.device, p.torch_dtype
    doh = _empty(p.hybrid_shape(p.Hq, Pu), dt, dev)
    dqh = _empty(p.hybrid_shape(p.Hq, Pu), dt, dev)
    dkh = _empty(p.hybrid_shape(p.Hkv, Pu), dt, dev)
    dvh = _empty(p.hybrid_shape(p.Hkv, Pu), dt, dev)
    ws = torch.empty(max(usp_hybrid_bwd_workspace_size(p, Pu), 256), dtype=torch.uint8, device=dev)
    usp_hybrid_seq2head(p, Pu, p.Hq, do_seq, doh, stream)
    usp_hybrid_attn_bwd(p, Pu, saved["q"], saved["k"], saved["v"], saved["o"], saved["lse"], doh, dqh, dkh, dvh, ws,
                        None, stream)
    dq = _empty(p.seq_shape(p.Hq), dt, dev)
    dk = _empty(p.seq_shape(p.Hkv), dt, dev)
    dv = _empty(p.seq_shape(p.Hkv), dt, dev)
    usp_hybrid_head2seq(p, Pu, p.Hq, dqh, dq, stream)
    usp_hybrid_head2seq(p, Pu, p.Hkv, dkh, dk, stream)
    usp_hybrid_head2seq(p, Pu, p.Hkv, dvh, dv, stream)
    return dq, dk, dv

"""ORACLE -- TEST INFRASTRUCTURE ONLY.

The same float64 definitions as ``attn_oracle.c`` for sampled rows of long
sequences, with numpy matrix products (BLAS) as the only library step:
  S = scale * Q[rows] K^T, masked (causal: j <= i), two-pass softmax,
  O = P V, LSE = ln sum exp(S); gradients from the closed forms
  dP = dO V^T, dS = P (dP - D), dQ = scale dS K, dV = P^T dO, dK = scale dS^T Q.
Rows are processed in chunks only to bound memory; each chunk is the plain
definition.  The element-wise steps of a chunk (mask, max, exp, sums) run on
a pool of threads over disjoint row slices, only to use the host's cores:
every slice is the same definition.  Pinned against the C oracle and the
closed forms in tests/test_oracle.py.

Inputs: logical [B][H][N][d] arrays of float32 or uint16 bf16 bits.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_CHUNK = 128
_pool = None


def _threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # not on Linux
        return max(1, os.cpu_count() or 1)


def _rowwise(fn, n: int) -> None:
    """fn(row_slice) over disjoint row slices of range(n), on the thread pool (numpy releases the
    interpreter lock inside its element-wise loops).  About four slices per thread, of 16 rows at
    least (thinner slices cost more in per-call overhead than they gain)."""
    global _pool
    if _pool is None:
        _pool = ThreadPoolExecutor(max_workers=_threads())
    step = max(16, n // (4 * _threads()))
    list(_pool.map(fn, [slice(i, min(n, i + step)) for i in range(0, n, step)]))


def _f64(x: np.ndarray) -> np.ndarray:
    if x.dtype == np.uint16:
        return (np.ascontiguousarray(x).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.asarray(x, dtype=np.float64)


def _softmax_rows(s, rows, causal, m_out=None, l_out=None) -> None:
    """In place on s = scale Q_rows K^T: future keys (j > i) to -inf, then P = exp(s - max_j s)
    (unnormalised).  Row maxima and sums go to m_out / l_out when given.  Threaded over row slices."""
    nk = s.shape[1]

    def work(sl):
        x = s[sl]
        if causal:
            x[np.arange(nk)[None, :] > rows[sl, None]] = -np.inf
        m = x.max(axis=1)
        x -= m[:, None]
        np.exp(x, out=x)
        if m_out is not None:
            m_out[sl] = m
        if l_out is not None:
            l_out[sl] = x.sum(axis=1)

    _rowwise(work, s.shape[0])


def attn_rows(q, k, v, rows, causal=True, scale=None):
    """(o [B][Hq][nrows][d], lse [B][Hq][nrows]) for query positions `rows`."""
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    rows = np.asarray(rows, dtype=np.int64)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    o = np.empty((B, Hq, len(rows), d))
    lse = np.empty((B, Hq, len(rows)))
    for b in range(B):
        for hk in range(Hkv):
            kk, vv = _f64(k[b, hk]), _f64(v[b, hk])
            for h in range(hk * g, (hk + 1) * g):
                for c0 in range(0, len(rows), _CHUNK):
                    r = rows[c0:c0 + _CHUNK]
                    end = int(r.max()) + 1 if causal else N   # keys any of these rows can see
                    s = _f64(q[b, h, r]) @ kk[:end].T
                    s *= scale                                # S
                    m = np.empty(len(r))
                    l_ = np.empty(len(r))
                    _softmax_rows(s, r, causal, m, l_)        # P (unnormalised) in place
                    o[b, h, c0:c0 + len(r)] = (s @ vv[:end]) / l_[:, None]
                    lse[b, h, c0:c0 + len(r)] = m + np.log(l_)
    return o, lse


def attn_bwd_q_rows(q, k, v, dout, rows, causal=True, scale=None):
    """dQ [B][Hq][nrows][d] of query positions `rows` for upstream gradient dO."""
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    rows = np.asarray(rows, dtype=np.int64)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    dq = np.empty((B, Hq, len(rows), d))
    for b in range(B):
        for hk in range(Hkv):
            kk, vv = _f64(k[b, hk]), _f64(v[b, hk])
            for h in range(hk * g, (hk + 1) * g):
                for c0 in range(0, len(rows), _CHUNK):
                    r = rows[c0:c0 + _CHUNK]
                    end = int(r.max()) + 1 if causal else N   # keys any of these rows can see
                    p = _f64(q[b, h, r]) @ kk[:end].T
                    p *= scale                                # S
                    l_ = np.empty(len(r))
                    _softmax_rows(p, r, causal, None, l_)
                    p /= l_[:, None]                          # P_ij
                    oi = p @ vv[:end]                         # O_i
                    doi = _f64(dout[b, h, r])
                    dvec = np.einsum("rd,rd->r", doi, oi)     # D_i
                    ds = doi @ vv[:end].T                     # dP_ij
                    ds -= dvec[:, None]
                    ds *= p                                   # dS_ij = P_ij (dP_ij - D_i)
                    dq[b, h, c0:c0 + len(r)] = scale * (ds @ kk[:end])
    return dq


def attn_lse_dvec(q, k, v, dout, causal=True, scale=None, kv_heads=None, row_lo=0, chunk=512):
    """LSE_i = ln sum_j exp(S_ij) and D_i = dO_i . O_i (float64) of every query row i >= row_lo, for
    the query heads of the KV heads (b, hk) listed in kv_heads (every KV head when None).

    Returns (lse, dvec) of shape [B][Hq][N]; entries not computed are NaN.  Per chunk of query rows
    this is the plain two-pass definition: S = scale Q K^T over the keys j <= i (causal), m = max_j S,
    P = exp(S - m), l = sum_j P, O = (P V) / l, LSE = m + ln l, D = dO . O.
    """
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    lse = np.full((B, Hq, N), np.nan)
    dvec = np.full((B, Hq, N), np.nan)
    pairs = [(b, hk) for b in range(B) for hk in range(Hkv)] if kv_heads is None else list(kv_heads)
    for b, hk in pairs:
        kk, vv = _f64(k[b, hk]), _f64(v[b, hk])
        for h in range(hk * g, (hk + 1) * g):
            for r0 in range(row_lo, N, chunk):
                r1 = min(N, r0 + chunk)
                end = r1 if causal else N                     # keys any row of the chunk can see
                qc, doc = _f64(q[b, h, r0:r1]), _f64(dout[b, h, r0:r1])
                s_ = scale * (qc @ kk[:end].T)                # S: [rows][keys]
                m = np.empty(r1 - r0)
                l_ = np.empty(r1 - r0)

                def softmax(sl, s_=s_, m=m, l_=l_, r0=r0, end=end):
                    x = s_[sl]                                # a view: rows r0 + sl of the chunk
                    if causal:
                        # keys j > i: only among the chunk's own positions [r0, end)
                        i = np.arange(r0 + sl.start, r0 + sl.stop)[:, None]
                        x[:, r0:][np.arange(r0, end)[None, :] > i] = -np.inf
                    m[sl] = x.max(axis=1)
                    x -= m[sl, None]
                    np.exp(x, out=x)                          # P (unnormalised), in place
                    l_[sl] = x.sum(axis=1)

                _rowwise(softmax, r1 - r0)
                o = (s_ @ vv[:end]) / l_[:, None]             # O
                lse[b, h, r0:r1] = m + np.log(l_)
                dvec[b, h, r0:r1] = np.einsum("rd,rd->r", doc, o)
    return lse, dvec


def attn_bwd_kv_rows(q, k, v, dout, lse, dvec, rows, causal=True, scale=None, kv_heads=None, chunk=4096):
    """(dk, dv) [B][Hkv][nrows][d] of key positions `rows`, summed over each KV head's group.

    lse, dvec: [B][Hq][N] LSE_i and D_i = dO_i . O_i (only rows i >= min(rows)
    are read when causal).  kv_heads: the (b, hk) pairs to compute (every KV
    head when None; the others stay zero).  Query rows are taken in chunks
    only to bound memory; each adds its rows' terms of the sums over i.
    """
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    rows = np.asarray(rows, dtype=np.int64)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    lo = int(rows.min()) if (causal and len(rows)) else 0
    dk = np.zeros((B, Hkv, len(rows), d))
    dv = np.zeros((B, Hkv, len(rows), d))
    pairs = [(b, hk) for b in range(B) for hk in range(Hkv)] if kv_heads is None else list(kv_heads)
    for b, hk in pairs:
        kr, vr = _f64(k[b, hk, rows]), _f64(v[b, hk, rows])
        for h in range(hk * g, (hk + 1) * g):
            for i0 in range(lo, N, chunk):                     # query rows that can see the keys
                i1 = min(N, i0 + chunk)
                qq = _f64(q[b, h, i0:i1])
                doo = _f64(dout[b, h, i0:i1])
                st = scale * (kr @ qq.T)                       # S^T: [keys][queries]
                if causal:
                    st[rows[:, None] > np.arange(i0, i1)[None, :]] = -np.inf
                pt = np.exp(st - np.asarray(lse[b, h, i0:i1], dtype=np.float64)[None, :])
                dv[b, hk] += pt @ doo
                dpt = vr @ doo.T
                dst = pt * (dpt - np.asarray(dvec[b, h, i0:i1], dtype=np.float64)[None, :])
                dk[b, hk] += scale * (dst @ qq)
    return dk, dv

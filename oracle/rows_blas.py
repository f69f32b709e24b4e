"""ORACLE -- TEST INFRASTRUCTURE ONLY.

The same float64 definitions as ``attn_oracle.c`` for sampled rows of long
sequences, with numpy matrix products (BLAS) as the only library step:
  S = scale * Q[rows] K^T, masked (causal: j <= i), two-pass softmax,
  O = P V, LSE = ln sum exp(S); gradients from the closed forms
  dP = dO V^T, dS = P (dP - D), dQ = scale dS K, dV = P^T dO, dK = scale dS^T Q.
Rows are processed in chunks only to bound memory; each chunk is the plain
definition.  Pinned against the C oracle and the closed forms in
tests/test_oracle.py.

Inputs: logical [B][H][N][d] arrays of float32 or uint16 bf16 bits.
"""
from __future__ import annotations

import numpy as np

_CHUNK = 64


def _f64(x: np.ndarray) -> np.ndarray:
    if x.dtype == np.uint16:
        return (np.ascontiguousarray(x).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.asarray(x, dtype=np.float64)


def _scores(qr, kk, rows, causal, scale):
    """scale * Q_rows K^T with future keys (j > i) set to -inf."""
    s = scale * (qr @ kk.T)
    if causal:
        s[np.arange(kk.shape[0])[None, :] > rows[:, None]] = -np.inf
    return s


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
                    s = _scores(_f64(q[b, h, r]), kk, r, causal, scale)
                    m = s.max(axis=1)
                    p = np.exp(s - m[:, None])
                    l_ = p.sum(axis=1)
                    o[b, h, c0:c0 + len(r)] = (p @ vv) / l_[:, None]
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
                    s = _scores(_f64(q[b, h, r]), kk, r, causal, scale)
                    m = s.max(axis=1)
                    p = np.exp(s - m[:, None])
                    p /= p.sum(axis=1)[:, None]               # P_ij
                    oi = p @ vv                               # O_i
                    doi = _f64(dout[b, h, r])
                    dvec = np.einsum("rd,rd->r", doi, oi)     # D_i
                    dp = doi @ vv.T                           # dP_ij
                    ds = p * (dp - dvec[:, None])             # dS_ij
                    dq[b, h, c0:c0 + len(r)] = scale * (ds @ kk)
    return dq


def attn_bwd_kv_rows(q, k, v, dout, lse, dvec, rows, causal=True, scale=None):
    """(dk, dv) [B][Hkv][nrows][d] of key positions `rows`, summed over each KV head's group.

    lse, dvec: [B][Hq][N] LSE_i and D_i = dO_i . O_i (only rows i >= min(rows)
    are read when causal).
    """
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    rows = np.asarray(rows, dtype=np.int64)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    lo = int(rows.min()) if (causal and len(rows)) else 0
    dk = np.zeros((B, Hkv, len(rows), d))
    dv = np.zeros((B, Hkv, len(rows), d))
    for b in range(B):
        for hk in range(Hkv):
            kr, vr = _f64(k[b, hk, rows]), _f64(v[b, hk, rows])
            for h in range(hk * g, (hk + 1) * g):
                qq = _f64(q[b, h, lo:])                        # query rows that can see the keys
                doo = _f64(dout[b, h, lo:])
                st = scale * (kr @ qq.T)                       # S^T: [keys][queries]
                if causal:
                    st[rows[:, None] > np.arange(lo, N)[None, :]] = -np.inf
                pt = np.exp(st - np.asarray(lse[b, h, lo:], dtype=np.float64)[None, :])
                dv[b, hk] += pt @ doo
                dpt = vr @ doo.T
                dst = pt * (dpt - np.asarray(dvec[b, h, lo:], dtype=np.float64)[None, :])
                dk[b, hk] += scale * (dst @ qq)
    return dk, dv

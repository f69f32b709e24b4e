"""Shared helpers for the parity tests: seeded inputs, layout views, metrics.

Layout changes here are plain numpy reshape/transpose views of the logical
[B][H][N][d] tensor (the oracle's layout maps are pinned against exactly
these views in test_oracle.py).
"""
from __future__ import annotations

import numpy as np

import synth

# tolerances (floating point; remaps are compared bit for bit)
TOL_F32_MAXABS = 1e-5         # float32 path vs float64
TOL_BF16_O_MAXABS = 2e-2      # bf16 output
TOL_BF16_O_RELFRO = 1e-2
TOL_BF16_GRAD_RELFRO = 2e-2   # bf16 gradients
TOL_LSE_F32 = 1e-4            # LSE, float32 path
TOL_LSE_BF16 = 5e-3           # LSE, bf16 path


def gen(shape, stream, dtype="bf16", seed=0, scale=1.0):
    """Seeded N(0,1) logical tensor: uint16 bf16 bits or float32."""
    return synth.normal(shape, seed=seed, stream=stream, dtype=dtype, scale=scale)


def to_seq(x: np.ndarray, P: int) -> np.ndarray:
    """logical [B][H][N][d] -> sequence-sharded [P][B][N/P][H][d] (copy)."""
    B, H, N, d = x.shape
    return np.ascontiguousarray(x.reshape(B, H, P, N // P, d).transpose(2, 0, 3, 1, 4))


def from_seq(x: np.ndarray) -> np.ndarray:
    """sequence-sharded [P][B][N/P][H][d] -> logical [B][H][N][d] (copy)."""
    P, B, Np, H, d = x.shape
    return np.ascontiguousarray(x.transpose(1, 3, 0, 2, 4).reshape(B, H, P * Np, d))


def to_head(x: np.ndarray, P: int) -> np.ndarray:
    """logical [B][H][N][d] -> head-sharded [P][B][H/P][N][d] (copy)."""
    B, H, N, d = x.shape
    return np.ascontiguousarray(x.reshape(B, P, H // P, N, d).transpose(1, 0, 2, 3, 4))


def from_head(x: np.ndarray) -> np.ndarray:
    """head-sharded [P][B][H/P][N][d] (or [P][B][H/P][N] for LSE) -> logical [B][H][N](...)."""
    P, B, Hl = x.shape[:3]
    rest = x.shape[3:]
    return np.ascontiguousarray(np.swapaxes(x, 0, 1).reshape(B, P * Hl, *rest))


def to_hybrid(x: np.ndarray, P: int, Pu: int) -> np.ndarray:
    """logical [B][H][N][d] -> 2-D layout [P][B][H/Pu][N/Pr][d] (Pr = P/Pu; rank g*Pu + u holds
    heads u*H/Pu .. of token chunk g) (copy)."""
    B, H, N, d = x.shape
    Pr = P // Pu
    y = x.reshape(B, Pu, H // Pu, Pr, N // Pr, d).transpose(3, 1, 0, 2, 4, 5)
    return np.ascontiguousarray(y.reshape(P, B, H // Pu, N // Pr, d))


def from_hybrid(x: np.ndarray, Pu: int) -> np.ndarray:
    """2-D layout [P][B][H/Pu][N/Pr](...) (tensor or LSE) -> logical [B][H][N](...) (copy)."""
    P, B, Hl, Nc = x.shape[:4]
    rest = x.shape[4:]
    Pr = P // Pu
    y = x.reshape(Pr, Pu, B, Hl, Nc, *rest)
    y = np.moveaxis(y, [2, 1, 3, 0, 4], [0, 1, 2, 3, 4])
    return np.ascontiguousarray(y.reshape(B, Pu * Hl, Pr * Nc, *rest))


def lse_from_seq(x: np.ndarray) -> np.ndarray:
    """sequence-sharded LSE [P][B][N/P][Hq] -> logical [B][Hq][N] (copy)."""
    P, B, Np, H = x.shape
    return np.ascontiguousarray(x.transpose(1, 3, 0, 2).reshape(B, H, P * Np))


def f64(x: np.ndarray) -> np.ndarray:
    if x.dtype == np.uint16:
        return synth.bf16_to_f32(x).astype(np.float64)
    return x.astype(np.float64)


def rel_fro(a: np.ndarray, b: np.ndarray) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b.ravel())
    return float(np.linalg.norm((a - b).ravel()) / (den if den > 0 else 1.0))


def bf16_ulp_diff(got: np.ndarray, want: np.ndarray, floor: float = 2.0 ** -16) -> float:
    """Largest |got - want| over the elements, in units of the bf16 spacing (2^(e - 7) for
    2^e <= |x| < 2^(e+1)) at the larger of the two magnitudes, after allowing an absolute
    `floor` * max|want|; bf16 bit arrays in.  Two float32 sums of the same terms in different
    orders, each rounded once to bf16, differ by at most one unit, except where the sum is far
    smaller than its terms (a row of dQ sums terms whose total nearly cancels): there the
    float32 rounding of the terms, about 2^-24 of their size, can exceed a unit of the tiny
    result, and the floor (2^-16 of the largest element, 2^8 times that rounding) covers it."""
    a, b = f64(got), f64(want)
    if not a.size:
        return 0.0
    mag = np.maximum(np.abs(a), np.abs(b))
    tiny = 2.0 ** -126
    ulp = np.exp2(np.floor(np.log2(np.maximum(mag, tiny))) - 7)
    atol = floor * float(np.max(np.abs(b)))
    return float(np.max(np.maximum(np.abs(a - b) - atol, 0.0) / ulp))


def max_abs(a, b) -> float:
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64)))) if np.size(a) else 0.0


def sample_rows(N: int, n: int, P: int, seed: int = 1, extra=()) -> np.ndarray:
    """n positions without replacement, always holding the shard edges (and `extra`)."""
    must = {0, N - 1, *[int(x) for x in extra]}
    Np = N // P
    for p in range(1, P):
        must.update({p * Np - 1, p * Np})
    rng = np.random.default_rng(seed)
    rest = np.setdiff1d(np.arange(N), np.array(sorted(must)))
    pick = rng.choice(rest, size=max(0, min(n, N) - len(must)), replace=False)
    return np.sort(np.concatenate([np.array(sorted(must)), pick])).astype(np.int64)


# ------------------------------------------------------------------ torch glue
def to_dev(x: np.ndarray, dtype: str = "bf16"):
    import torch
    if dtype == "bf16":
        assert x.dtype == np.uint16
        t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.cuda()


def to_host(t) -> np.ndarray:
    import torch
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()

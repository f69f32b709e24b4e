"""GPU parity at the long-context sizes, in the launch configuration the
benchmark times, against the float64 oracle on seeded samples of rows (the
oracle cannot afford every row) and against properties that hold at any size:
  - remapped Q/K/V equal the oracle's all-to-all map bit for bit;
  - forward O and LSE on 1024 seeded query rows per head (shard edges included);
  - dQ on 1024 seeded query rows per head;
  - dK/dV on 1024 seeded key rows per KV head spread over the whole sequence
    (key 0, the shard edges, N/2 and N-1 included), against the oracle's
    gradients built from its own LSE and D of every query row that sees them
    (every KV head at 32K and below; one whole GQA group at 128K, whose
    4 query heads' every row the oracle evaluates) -- key 0 sums over all N
    queries of 4 heads, the longest accumulation the kernels do;
  - sum_j dK_j = 0 (softmax shift invariance) and sum_j dV_j = sum_i dO_i over
    every key row, within the bound the per-element tolerance implies for a sum;
  - the all-to-all fused into the kernels (sequence-sharded operands read and
    written in place) gives the remapped path's O, LSE and gradients bit for bit;
  - ring attention equals one full-sequence pass and the oracle's rows;
  - ring backward gradients equal the one-pass (P = 1) backward's on every
    element within the gradient tolerance, and match the oracle on 1024
    sampled dQ rows per head and on sampled key rows of the last 8192
    positions of two heads (the oracle's LSE and D of every row from there
    on), plus the same sum identities.
"""
import os

import numpy as np
import pytest

from tests.helpers import (TOL_BF16_GRAD_RELFRO, TOL_BF16_O_MAXABS, TOL_BF16_O_RELFRO, TOL_LSE_BF16, bf16_ulp_diff,
                           f64, gen, max_abs, rel_fro, sample_rows, to_dev, to_host)

pytestmark = pytest.mark.gpu

FWD_ROWS = int(os.environ.get("USP_TEST_FWD_ROWS", "1024"))
DQ_ROWS = int(os.environ.get("USP_TEST_DQ_ROWS", "1024"))
KV_ROWS = int(os.environ.get("USP_TEST_KV_ROWS", "1024"))
RING_ROWS = int(os.environ.get("USP_TEST_RING_ROWS", "1024"))
RING_KEY_SPAN = 8192   # the ring's oracle dK/dV rows lie in the last RING_KEY_SPAN positions
VERBOSE = os.environ.get("USP_TEST_VERBOSE", "") == "1"


@pytest.fixture(scope="module")
def usp():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import context_long_attention_ulysses_gb300 as m
    from context_long_attention_ulysses_gb300 import build
    build.build()
    return m


def _seq_on_device(x_logical_dev, P):
    """logical [B][H][N][d] -> sequence-sharded [P][B][N/P][H][d] (test-side layout change)."""
    B, H, N, d = x_logical_dev.shape
    return x_logical_dev.view(B, H, P, N // P, d).permute(2, 0, 3, 1, 4).contiguous()


def _logical_from_seq(x_seq_dev):
    P, B, Np, H, d = x_seq_dev.shape
    return x_seq_dev.permute(1, 3, 0, 2, 4).reshape(B, H, P * Np, d).contiguous()


@pytest.mark.parametrize("B,Hq,Hkv,N,d,P,kv_groups", [
    (1, 32, 8, 32768, 128, 4, None),       # GQA long context, 8192 tokens per shard: every KV head
    (1, 32, 8, 131072, 128, 8, [(0, 5)]),  # 128K-token training step: KV head 5's group of 4 query heads
    (1, 16, 4, 32768, 64, 4, None),        # head dimension 64
    (2, 8, 2, 16384, 128, 2, None),        # two sequences of 16K tokens, GQA group of 4
])
def test_ulysses_long_context(usp, orc, B, Hq, Hkv, N, d, P, kv_groups):
    import torch
    from oracle import rows_blas
    p = usp.Problem(B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, P=P)
    q, k, v, dO = gen((B, Hq, N, d), 0), gen((B, Hkv, N, d), 1), gen((B, Hkv, N, d), 2), gen((B, Hq, N, d), 3)
    qs, ks, vs, dos = (_seq_on_device(to_dev(x), P) for x in (q, k, v, dO))
    o_seq, saved = usp.ulysses_attention_fwd(p, qs, ks, vs)
    dq_s, dk_s, dv_s = usp.ulysses_attention_bwd(p, saved, dos)
    torch.cuda.synchronize()
    assert usp.usp_device_status() == 0

    # the fused path at full size: the same bits (dQ to one bf16 unit: its float32 additions'
    # order varies from run to run), no remap
    o_f, lse_f = usp.fused_attention_fwd(p, qs, ks, vs)
    grads_f = usp.fused_attention_bwd(p, qs, ks, vs, o_f, lse_f, dos)
    torch.cuda.synchronize()
    assert usp.usp_device_status() == 0
    for got, want in zip((o_f, *grads_f[1:]), (o_seq, dk_s, dv_s)):
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    assert bf16_ulp_diff(to_host(grads_f[0]), to_host(dq_s)) <= 1.0
    lse_u = saved["lse"].permute(1, 0, 2, 3).reshape(B, Hq, N)
    assert torch.equal(lse_f.permute(1, 3, 0, 2).reshape(B, Hq, N).view(torch.int32), lse_u.view(torch.int32))
    del o_f, lse_f, grads_f, lse_u
    # the three-pass (deterministic) backward at full size: dK and dV bit for bit, dQ within a tenth
    # of the gradient tolerance (its dQ pass rounds dS its own way)
    grads_3 = usp.ulysses_attention_bwd(p, saved, dos, deterministic=True)
    torch.cuda.synchronize()
    assert usp.usp_device_status() == 0
    for got, want in zip(grads_3[1:], (dk_s, dv_s)):
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    d13 = float((grads_3[0].float() - dq_s.float()).norm() / dq_s.float().norm())
    if VERBOSE:
        print(f"\n[N={N}] one-pass vs three-pass dQ: relative Frobenius {d13:.3e}")
    assert d13 < 0.1 * TOL_BF16_GRAD_RELFRO
    del grads_3

    # all-to-all: the oracle's index map, bit for bit
    assert to_host(saved["k"]).tobytes() == orc.seq2head(to_host(ks)).tobytes()
    if N <= 32768:
        assert to_host(saved["q"]).tobytes() == orc.seq2head(to_host(qs)).tobytes()
    # the head-sharded layout [P][B][Hq/P][N][d] is rank-major; with one sequence it is the logical tensor
    def logical_from_head(x, H):
        return np.ascontiguousarray(x.reshape(P, B, H // P, N, -1).transpose(1, 0, 2, 3, 4).reshape(B, H, N, -1))
    assert logical_from_head(to_host(saved["q"]), Hq).tobytes() == q.tobytes()
    o_head = logical_from_head(to_host(saved["o"]), Hq)
    assert to_host(_logical_from_seq(o_seq)).tobytes() == o_head.tobytes()

    o = o_head
    lse = logical_from_head(to_host(saved["lse"]), Hq).reshape(B, Hq, N)
    dq = to_host(_logical_from_seq(dq_s))
    dk = to_host(_logical_from_seq(dk_s))
    dv = to_host(_logical_from_seq(dv_s))
    del qs, ks, vs, dos, saved, o_seq, dq_s, dk_s, dv_s
    torch.cuda.empty_cache()

    # forward on sampled rows
    rows = sample_rows(N, FWD_ROWS, P, seed=1)
    o_ref, lse_ref = rows_blas.attn_rows(q, k, v, rows, causal=True)
    assert max_abs(f64(o[:, :, rows]), o_ref) < TOL_BF16_O_MAXABS
    assert rel_fro(f64(o[:, :, rows]), o_ref) < TOL_BF16_O_RELFRO
    assert max_abs(lse[:, :, rows], lse_ref) < TOL_LSE_BF16

    _check_sampled_grads(q, k, v, dO, dq, dk, dv, P, kv_groups)


def _check_sampled_grads(q, k, v, dO, dq, dk, dv, P, kv_groups=None, key_lo=0):
    """dQ on seeded query rows; dK/dV on seeded key rows >= key_lo of the KV heads kv_groups
    ((b, hk) pairs, every one when None) against the oracle's own LSE and D of every query row
    >= key_lo; the sum identities over every key row."""
    import time

    from oracle import rows_blas
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    # dQ on sampled rows
    t0 = time.perf_counter()
    rq = sample_rows(N, DQ_ROWS, P, seed=2)
    dq_ref = rows_blas.attn_bwd_q_rows(q, k, v, dO, rq, causal=True)
    err_dq = rel_fro(f64(dq[:, :, rq]), dq_ref)
    assert err_dq < TOL_BF16_GRAD_RELFRO

    # dK/dV on seeded key rows: the oracle's LSE_i and D_i of every query row that sees them
    t1 = time.perf_counter()
    groups = [(b, hk) for b in range(B) for hk in range(Hkv)] if kv_groups is None else list(kv_groups)
    lse_o, dvec_o = rows_blas.attn_lse_dvec(q, k, v, dO, causal=True, kv_heads=groups, row_lo=key_lo)
    if key_lo == 0:
        keys = sample_rows(N, KV_ROWS, P, seed=4, extra=(N // 2,))
    else:
        rng = np.random.default_rng(4)
        span = N - key_lo
        keys = np.union1d([key_lo, N - 1], key_lo + rng.choice(span, size=min(KV_ROWS, span), replace=False))
    t2 = time.perf_counter()
    dk_ref, dv_ref = rows_blas.attn_bwd_kv_rows(q, k, v, dO, lse_o, dvec_o, keys, causal=True, kv_heads=groups)
    t3 = time.perf_counter()
    for b, hk in groups:
        got_k, got_v = f64(dk[b, hk, keys]), f64(dv[b, hk, keys])
        err_k, err_v = rel_fro(got_k, dk_ref[b, hk]), rel_fro(got_v, dv_ref[b, hk])
        if VERBOSE:
            # per key row: relative error of the row and the signed relative bias of dV along its reference
            rk = np.linalg.norm(got_k - dk_ref[b, hk], axis=1) / np.linalg.norm(dk_ref[b, hk], axis=1)
            rv = np.linalg.norm(got_v - dv_ref[b, hk], axis=1) / np.linalg.norm(dv_ref[b, hk], axis=1)
            bias_v = np.einsum("kd,kd->k", got_v - dv_ref[b, hk], dv_ref[b, hk]) / np.einsum(
                "kd,kd->k", dv_ref[b, hk], dv_ref[b, hk])
            first = keys < N // 8
            print(f"\n[N={N} b={b} hk={hk}] dK relfro {err_k:.3e} dV relfro {err_v:.3e}; per-row max dK "
                  f"{rk.max():.3e} dV {rv.max():.3e}; dV bias mean {bias_v.mean():+.3e} "
                  f"(keys < N/8: {bias_v[first].mean() if first.any() else float('nan'):+.3e}, key {keys[0]}: {bias_v[0]:+.3e})")
        assert err_k < TOL_BF16_GRAD_RELFRO, (b, hk, err_k)
        assert err_v < TOL_BF16_GRAD_RELFRO, (b, hk, err_v)
    if VERBOSE:
        print(f"[N={N}] dQ relfro {err_dq:.3e}; oracle seconds: dQ {t1 - t0:.1f}, LSE/D {t2 - t1:.1f}, "
              f"dK/dV {t3 - t2:.1f}")

    # identities over every key row.  If every dK_j, dV_j is within relative
    # error TOL, the triangle inequality bounds the error of their sum by
    # TOL * sum_j |dK_j| (resp. |dV_j|), which is the bound checked here.
    dkf, dvf = f64(dk), f64(dv)
    bound_k = np.linalg.norm(dkf, axis=3).sum(axis=2)   # [B][Hkv]
    bound_v = np.linalg.norm(dvf, axis=3).sum(axis=2)
    sum_dk = dkf.sum(axis=2)                            # exact value: 0
    assert np.all(np.linalg.norm(sum_dk, axis=2) < TOL_BF16_GRAD_RELFRO * bound_k)
    g = Hq // Hkv
    want = f64(dO).reshape(B, Hkv, g, N, d).sum(axis=(2, 3))   # exact value of sum_j dV_j
    assert np.all(np.linalg.norm(dvf.sum(axis=2) - want, axis=2) < TOL_BF16_GRAD_RELFRO * bound_v)


def test_ring_512k(usp, orc):
    """512K tokens, 32 heads, d=128, P=8 shards of 65536: ring forward and backward, zigzag forward."""
    import torch
    from oracle import rows_blas
    B, H, N, d, P = 1, 32, 524288, 128, 8
    p = usp.Problem(B=B, Hq=H, Hkv=H, N=N, d=d, P=P)
    q, k, v, dO = gen((B, H, N, d), 0), gen((B, H, N, d), 1), gen((B, H, N, d), 2), gen((B, H, N, d), 3)
    ql, kl, vl, dol = to_dev(q), to_dev(k), to_dev(v), to_dev(dO)
    # one full-sequence pass, forward and backward: P = 1, the logical tensor is the (single)
    # head-sharded buffer
    p1 = usp.Problem(B=B, Hq=H, Hkv=H, N=N, d=d, P=1)
    o_full = torch.empty_like(ql)
    lse_full = torch.empty((1, B, H, N), dtype=torch.float32, device="cuda")
    usp.usp_attn_fwd(p1, ql, kl, vl, o_full, lse_full)
    g1 = [torch.empty_like(ql), torch.empty_like(kl), torch.empty_like(vl)]
    ws1 = torch.empty(usp.usp_attn_bwd_workspace_size(p1), dtype=torch.uint8, device="cuda")
    usp.usp_attn_bwd(p1, ql, kl, vl, o_full, lse_full, dol, *g1, ws1)
    del ws1
    qs, ks, vs, dos = (_seq_on_device(x, P) for x in (ql, kl, vl, dol))
    del ql, kl, vl, dol
    o_ring, lse_ring = usp.ring_attention_fwd(p, qs, ks, vs)
    torch.cuda.synchronize()
    assert usp.usp_device_status() == 0
    # ring backward with the seeded upstream gradient
    dq_s, dk_s, dv_s = usp.ring_attention_bwd(p, qs, ks, vs, o_ring, lse_ring, dos)
    torch.cuda.synchronize()
    assert usp.usp_device_status() == 0
    # ring gradients == one-pass gradients, every element (per head, relative Frobenius)
    for name, got_s, want in zip(("dq", "dk", "dv"), (dq_s, dk_s, dv_s), g1):
        got = _logical_from_seq(got_s).float()
        err = (got - want.float()).norm(dim=(2, 3)) / want.float().norm(dim=(2, 3))
        assert float(err.max()) < TOL_BF16_GRAD_RELFRO, (name, float(err.max()))
        if VERBOSE:
            print(f"\n[ring 512K vs one pass] {name} per-head relfro max {float(err.max()):.3e}")
        del got, err
    del g1
    dq, dk, dv = (to_host(_logical_from_seq(x)) for x in (dq_s, dk_s, dv_s))
    del dos, dq_s, dk_s, dv_s
    # zigzag (load-balanced) ring forward on the same inputs, back to contiguous shards
    zz = [torch.empty_like(x) for x in (qs, ks, vs)]
    for src, dst in zip((qs, ks, vs), zz):
        usp.usp_zigzag_shard(p, H, src, dst)
    o_zz, _ = usp.zigzag_attention_fwd(p, *zz)
    o_zz_seq = torch.empty_like(o_zz)
    usp.usp_zigzag_unshard(p, H, o_zz, o_zz_seq)
    torch.cuda.synchronize()
    assert usp.usp_device_status() == 0
    dz = _logical_from_seq(o_zz_seq).float() - o_full.float()
    assert float(dz.abs().max()) < TOL_BF16_O_MAXABS
    assert float(dz.norm() / o_full.float().norm()) < TOL_BF16_O_RELFRO
    del qs, ks, vs, zz, o_zz, o_zz_seq, dz
    o_ring_l = _logical_from_seq(o_ring)
    lse_ring_l = lse_ring.permute(1, 3, 0, 2).reshape(B, H, N)
    # ring == one pass (both bf16 outputs of float32 arithmetic)
    diff = (o_ring_l.float() - o_full.float())
    assert float(diff.abs().max()) < TOL_BF16_O_MAXABS
    assert float(diff.norm() / o_full.float().norm()) < TOL_BF16_O_RELFRO
    assert float((lse_ring_l - lse_full.view(B, H, N)).abs().max()) < TOL_LSE_BF16
    o = to_host(o_ring_l)
    lse = lse_ring_l.cpu().numpy()
    del o_full, lse_full, o_ring, lse_ring, o_ring_l, lse_ring_l, diff
    torch.cuda.empty_cache()
    rows = sample_rows(N, RING_ROWS, P, seed=3)
    o_ref, lse_ref = rows_blas.attn_rows(q, k, v, rows, causal=True)
    assert max_abs(f64(o[:, :, rows]), o_ref) < TOL_BF16_O_MAXABS
    assert rel_fro(f64(o[:, :, rows]), o_ref) < TOL_BF16_O_RELFRO
    assert max_abs(lse[:, :, rows], lse_ref) < TOL_LSE_BF16
    # the oracle's every-row LSE and D cost N^2 per head: its key rows lie in the last RING_KEY_SPAN
    # positions of two heads (the one-pass comparison above covers every key)
    _check_sampled_grads(q, k, v, dO, dq, dk, dv, P, kv_groups=[(0, 5), (0, 27)], key_lo=N - RING_KEY_SPAN)

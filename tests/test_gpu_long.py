"""GPU parity at the long-context sizes, in the launch configuration the
benchmark times, against the float64 oracle on seeded samples of rows (the
oracle cannot afford every row) and against properties that hold at any size:
  - remapped Q/K/V equal the oracle's all-to-all map bit for bit;
  - forward O and LSE on 1024 seeded query rows per head (shard edges included);
  - dQ on seeded query rows, dK/dV on the last key rows of every KV head
    (their rows i >= j are few enough for the oracle), plus
    sum_j dK_j = 0 (softmax shift invariance) and sum_j dV_j = sum_i dO_i,
    within the bound the per-element tolerance implies for a sum;
  - the all-to-all fused into the kernels (sequence-sharded operands read and
    written in place) gives the remapped path's O, LSE and gradients bit for bit;
  - ring attention equals one full-sequence pass and the oracle's rows;
  - ring backward gradients against the oracle on sampled dQ rows and tail
    dK/dV rows, plus the same sum identities.
"""
import os

import numpy as np
import pytest

from tests.helpers import (TOL_BF16_GRAD_RELFRO, TOL_BF16_O_MAXABS, TOL_BF16_O_RELFRO, TOL_LSE_BF16, f64, gen,
                           max_abs, rel_fro, sample_rows, to_dev, to_host)

pytestmark = pytest.mark.gpu

FWD_ROWS = int(os.environ.get("USP_TEST_FWD_ROWS", "1024"))
DQ_ROWS = int(os.environ.get("USP_TEST_DQ_ROWS", "256"))
KV_TAIL = int(os.environ.get("USP_TEST_KV_TAIL", "256"))
RING_ROWS = int(os.environ.get("USP_TEST_RING_ROWS", "256"))


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


@pytest.mark.parametrize("B,Hq,Hkv,N,d,P", [
    (1, 32, 8, 32768, 128, 4),     # GQA long context, 8192 tokens per shard
    (1, 32, 8, 131072, 128, 8),    # 128K-token training step
    (1, 16, 4, 32768, 64, 4),      # head dimension 64
    (2, 8, 2, 16384, 128, 2),      # two sequences of 16K tokens, GQA group of 4
])
def test_ulysses_long_context(usp, orc, B, Hq, Hkv, N, d, P):
    import torch
    from oracle import rows_blas
    p = usp.Problem(B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, P=P)
    q, k, v, dO = gen((B, Hq, N, d), 0), gen((B, Hkv, N, d), 1), gen((B, Hkv, N, d), 2), gen((B, Hq, N, d), 3)
    qs, ks, vs, dos = (_seq_on_device(to_dev(x), P) for x in (q, k, v, dO))
    o_seq, saved = usp.ulysses_attention_fwd(p, qs, ks, vs)
    dq_s, dk_s, dv_s = usp.ulysses_attention_bwd(p, saved, dos)
    torch.cuda.synchronize()
    assert usp.usp_device_status() == 0

    # the fused path at full size: the same bits, no remap
    o_f, lse_f = usp.fused_attention_fwd(p, qs, ks, vs)
    grads_f = usp.fused_attention_bwd(p, qs, ks, vs, o_f, lse_f, dos)
    torch.cuda.synchronize()
    assert usp.usp_device_status() == 0
    for got, want in zip((o_f, *grads_f), (o_seq, dq_s, dk_s, dv_s)):
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    lse_u = saved["lse"].permute(1, 0, 2, 3).reshape(B, Hq, N)
    assert torch.equal(lse_f.permute(1, 3, 0, 2).reshape(B, Hq, N).view(torch.int32), lse_u.view(torch.int32))
    del o_f, lse_f, grads_f, lse_u

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

    _check_sampled_grads(q, k, v, dO, dq, dk, dv, P)


def _check_sampled_grads(q, k, v, dO, dq, dk, dv, P):
    """dQ on seeded rows, dK/dV on the last key rows, and the sum identities."""
    from oracle import rows_blas
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    # dQ on sampled rows
    rq = sample_rows(N, DQ_ROWS, P, seed=2)
    dq_ref = rows_blas.attn_bwd_q_rows(q, k, v, dO, rq, causal=True)
    assert rel_fro(f64(dq[:, :, rq]), dq_ref) < TOL_BF16_GRAD_RELFRO

    # dK/dV on the last key rows: they are seen by rows i >= N - KV_TAIL only
    tail = np.arange(N - KV_TAIL, N, dtype=np.int64)
    o_t, lse_t = rows_blas.attn_rows(q, k, v, tail, causal=True)
    lse_full = np.zeros((B, Hq, N))
    dvec_full = np.zeros((B, Hq, N))
    lse_full[:, :, tail] = lse_t
    dvec_full[:, :, tail] = np.einsum("bhnd,bhnd->bhn", f64(dO[:, :, tail]), o_t)
    dk_ref, dv_ref = rows_blas.attn_bwd_kv_rows(q, k, v, dO, lse_full, dvec_full, tail, causal=True)
    assert rel_fro(f64(dk[:, :, tail]), dk_ref) < TOL_BF16_GRAD_RELFRO
    assert rel_fro(f64(dv[:, :, tail]), dv_ref) < TOL_BF16_GRAD_RELFRO

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
    q, k, v = gen((B, H, N, d), 0), gen((B, H, N, d), 1), gen((B, H, N, d), 2)
    ql, kl, vl = to_dev(q), to_dev(k), to_dev(v)
    # one full-sequence pass: P = 1, the logical tensor is the (single) head-sharded buffer
    p1 = usp.Problem(B=B, Hq=H, Hkv=H, N=N, d=d, P=1)
    o_full = torch.empty_like(ql)
    lse_full = torch.empty((1, B, H, N), dtype=torch.float32, device="cuda")
    usp.usp_attn_fwd(p1, ql, kl, vl, o_full, lse_full)
    qs, ks, vs = (_seq_on_device(x, P) for x in (ql, kl, vl))
    del ql, kl, vl
    o_ring, lse_ring = usp.ring_attention_fwd(p, qs, ks, vs)
    torch.cuda.synchronize()
    assert usp.usp_device_status() == 0
    # ring backward with a seeded upstream gradient
    dO = gen((B, H, N, d), 3)
    dos = _seq_on_device(to_dev(dO), P)
    dq_s, dk_s, dv_s = usp.ring_attention_bwd(p, qs, ks, vs, o_ring, lse_ring, dos)
    torch.cuda.synchronize()
    assert usp.usp_device_status() == 0
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
    del o_full, lse_full, o_ring, lse_ring, o_ring_l, lse_ring_l
    torch.cuda.empty_cache()
    rows = sample_rows(N, RING_ROWS, P, seed=3)
    o_ref, lse_ref = rows_blas.attn_rows(q, k, v, rows, causal=True)
    assert max_abs(f64(o[:, :, rows]), o_ref) < TOL_BF16_O_MAXABS
    assert rel_fro(f64(o[:, :, rows]), o_ref) < TOL_BF16_O_RELFRO
    assert max_abs(lse[:, :, rows], lse_ref) < TOL_LSE_BF16
    _check_sampled_grads(q, k, v, dO, dq, dk, dv, P)

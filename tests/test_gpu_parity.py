"""GPU parity of the CUDA path (through the C ABI) against the float64 oracle,
at sizes the oracle finishes in seconds: every element compared."""
import numpy as np
import pytest

from tests.helpers import (TOL_BF16_GRAD_RELFRO, TOL_BF16_O_MAXABS, TOL_BF16_O_RELFRO, TOL_F32_MAXABS, TOL_LSE_BF16,
                           TOL_LSE_F32, bf16_ulp_diff, f64, from_head, from_hybrid, from_seq, gen, lse_from_seq,
                           max_abs, rel_fro, to_dev, to_head, to_host, to_hybrid, to_seq)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def usp():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import context_long_attention_ulysses_gb300 as m
    from context_long_attention_ulysses_gb300 import build
    build.build()
    return m


def _sync():
    import torch
    torch.cuda.synchronize()


def _status_ok(usp):
    assert usp.usp_device_status() == 0


# ---------------------------------------------------------------- remaps
@pytest.mark.parametrize("dtype,B,H,N,d,P", [
    ("f32", 1, 4, 256, 64, 2), ("bf16", 1, 4, 4096, 64, 2), ("bf16", 2, 8, 1000, 128, 4),
    ("bf16", 1, 32, 2048, 128, 8), ("f32", 3, 6, 96, 128, 3), ("bf16", 1, 8, 64, 32, 8)])
def test_remap_bit_exact(usp, orc, dtype, B, H, N, d, P):
    import torch
    p = usp.Problem(B=B, Hq=H, Hkv=H, N=N, d=d, P=P, dtype=dtype)
    x = gen((B, H, N, d), 0, dtype)
    seq = to_seq(x, P)
    src = to_dev(seq, dtype)
    head = torch.empty(p.head_shape(H), dtype=p.torch_dtype, device="cuda")
    back = torch.empty_like(src)
    usp.usp_a2a_seq2head(p, H, src, head)
    usp.usp_a2a_head2seq(p, H, head, back)
    _sync()
    want = orc.seq2head(seq)
    got = to_host(head)
    assert got.tobytes() == want.tobytes()
    assert to_host(back).tobytes() == seq.tobytes()
    _status_ok(usp)


# ---------------------------------------------------------------- tiny fp32 case
def test_tiny_exactness_case_fp32(usp, orc):
    """B=1, H=4, N=256, d=64, fp32, causal, P=2: remap -> attention -> remap, in full."""
    B, H, N, d, P = 1, 4, 256, 64, 2
    p = usp.Problem(B=B, Hq=H, Hkv=H, N=N, d=d, P=P, dtype="f32")
    q, k, v = (gen((B, H, N, d), s, "f32") for s in (0, 1, 2))
    o_seq, saved = usp.ulysses_attention_fwd(p, to_dev(to_seq(q, P), "f32"), to_dev(to_seq(k, P), "f32"),
                                             to_dev(to_seq(v, P), "f32"))
    _sync()
    # the all-to-all results are the oracle's, bit for bit
    assert to_host(saved["q"]).tobytes() == orc.seq2head(to_seq(q, P)).tobytes()
    o_ref, lse_ref = orc.attn_rows(q, k, v, causal=True)
    o = from_seq(to_host(o_seq))
    assert max_abs(o, o_ref) < TOL_F32_MAXABS
    assert max_abs(from_head(to_host(saved["lse"])), lse_ref) < TOL_LSE_F32
    _status_ok(usp)


# ---------------------------------------------------------------- bf16 fwd + bwd
def _ulysses_fwd_bwd(usp, B, Hq, Hkv, N, d, P, causal, dO=None):
    import torch
    p = usp.Problem(B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, P=P, causal=causal)
    q, k, v = gen((B, Hq, N, d), 0), gen((B, Hkv, N, d), 1), gen((B, Hkv, N, d), 2)
    o_seq, saved = usp.ulysses_attention_fwd(p, to_dev(to_seq(q, P)), to_dev(to_seq(k, P)), to_dev(to_seq(v, P)))
    if dO is None:  # loss = mean(out.float()^2): dO = 2 O / numel, formed in float32 and rounded to bf16
        do_seq = (2.0 * o_seq.float() / o_seq.numel()).to(torch.bfloat16)
    else:
        do_seq = to_dev(to_seq(dO, P))
    dq, dk, dv = usp.ulysses_attention_bwd(p, saved, do_seq)
    _sync()
    out = dict(o=from_seq(to_host(o_seq)), lse=from_head(to_host(saved["lse"])), dq=from_seq(to_host(dq)),
               dk=from_seq(to_host(dk)), dv=from_seq(to_host(dv)))
    return (q, k, v), out


def _check_fwd(o, lse, o_ref, lse_ref):
    assert max_abs(f64(o), o_ref) < TOL_BF16_O_MAXABS
    assert rel_fro(f64(o), o_ref) < TOL_BF16_O_RELFRO
    assert max_abs(lse, lse_ref) < TOL_LSE_BF16


def _check_grads(out, dq, dk, dv):
    for name, ref in (("dq", dq), ("dk", dk), ("dv", dv)):
        err = rel_fro(f64(out[name]), ref)
        assert err < TOL_BF16_GRAD_RELFRO, (name, err)


def test_example_shape_fwd_bwd_mean_square_loss(usp, orc):
    """The glossary page's example: B=1, H=4, N=4096, d=64, bf16, causal, P=2, loss mean(out^2)."""
    B, H, N, d, P = 1, 4, 4096, 64, 2
    (q, k, v), out = _ulysses_fwd_bwd(usp, B, H, H, N, d, P, True)
    o_ref, lse_ref = orc.attn_rows(q, k, v, causal=True)
    _check_fwd(out["o"], out["lse"], o_ref, lse_ref)
    # the oracle's own loss gradient, from its own output
    dO_ref = (2.0 * o_ref / o_ref.size).astype(np.float32)
    dq, dk, dv, _, _ = orc.attn_bwd_full(q, k, v, dO_ref, causal=True)
    _check_grads(out, dq, dk, dv)
    _status_ok(usp)


@pytest.mark.parametrize("B,Hq,Hkv,N,d,P,causal", [
    (1, 8, 2, 1000, 128, 2, True),     # GQA, ragged tail (N not a multiple of 128)
    (2, 4, 4, 520, 64, 2, True),       # two sequences, ragged
    (1, 4, 2, 384, 128, 2, False),     # full (non-causal) attention
    (1, 2, 1, 200, 64, 1, True),       # one rank: no exchange at all
    (1, 8, 8, 130, 128, 2, True),      # one full tile plus a 2-row tail per head
])
def test_fwd_bwd_edge_cases(usp, orc, B, Hq, Hkv, N, d, P, causal):
    dO = gen((B, Hq, N, d), 3)
    (q, k, v), out = _ulysses_fwd_bwd(usp, B, Hq, Hkv, N, d, P, causal, dO)
    o_ref, lse_ref = orc.attn_rows(q, k, v, causal=causal)
    _check_fwd(out["o"], out["lse"], o_ref, lse_ref)
    dq, dk, dv, _, _ = orc.attn_bwd_full(q, k, v, dO, causal=causal)
    _check_grads(out, dq, dk, dv)
    _status_ok(usp)


def test_sharded_equals_unsharded_bitwise(usp):
    """Sharded attention is the same per-head work as one unsharded pass: bit-identical."""
    import torch
    B, Hq, Hkv, N, d = 1, 8, 4, 768, 128
    q, k, v = gen((B, Hq, N, d), 0), gen((B, Hkv, N, d), 1), gen((B, Hkv, N, d), 2)
    outs = []
    for P in (1, 4):
        p = usp.Problem(B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, P=P)
        o_seq, saved = usp.ulysses_attention_fwd(p, to_dev(to_seq(q, P)), to_dev(to_seq(k, P)), to_dev(to_seq(v, P)))
        torch.cuda.synchronize()
        outs.append((from_seq(to_host(o_seq)), from_head(to_host(saved["lse"]))))
    assert outs[0][0].tobytes() == outs[1][0].tobytes()
    assert outs[0][1].tobytes() == outs[1][1].tobytes()


def test_rank_reads_only_its_own_buffers(usp):
    """Poison one rank's query heads with NaN: every other rank's output is unchanged."""
    import torch
    B, Hq, Hkv, N, d, P = 1, 8, 4, 512, 64, 4
    p = usp.Problem(B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, P=P)
    q, k, v = gen((B, Hq, N, d), 0), gen((B, Hkv, N, d), 1), gen((B, Hkv, N, d), 2)
    qh, kh, vh = to_dev(to_head(q, P)), to_dev(to_head(k, P)), to_dev(to_head(v, P))
    o1 = torch.empty_like(qh)
    l1 = torch.empty(p.lse_head_shape(), dtype=torch.float32, device="cuda")
    usp.usp_attn_fwd(p, qh, kh, vh, o1, l1)
    qh2 = qh.clone()
    qh2[2] = float("nan")
    kh2 = kh.clone()
    kh2[1] = float("nan")
    o2, l2 = torch.empty_like(o1), torch.empty_like(l1)
    usp.usp_attn_fwd(p, qh2, kh2, vh, o2, l2)
    torch.cuda.synchronize()
    for r in range(P):
        if r in (1, 2):
            assert torch.isnan(o2[r].float()).all()
        else:
            assert torch.equal(o1[r], o2[r]) and torch.equal(l1[r], l2[r])


# ---------------------------------------------------------------- ring mode
def test_lse_merge_kernel(usp, orc):
    import torch
    rows, d = 3000, 128
    rng = np.random.default_rng(5)
    oa, ob = rng.standard_normal((2, rows, d)).astype(np.float32)
    la, lb = (rng.standard_normal((2, rows)) * 4).astype(np.float32)
    la[::7] = -np.inf
    lb[::11] = -np.inf
    lb[::77] = -np.inf  # both empty on rows divisible by 77
    la[::77] = -np.inf
    oa[::7] = np.nan    # an empty partial's output must not leak
    ref_o, ref_l = orc.lse_merge(np.nan_to_num(oa), la, ob, lb)
    t = [torch.from_numpy(x).cuda() for x in (oa, la, ob, lb)]
    o = torch.empty_like(t[0])
    lse = torch.empty_like(t[1])
    usp.usp_ring_merge(rows, d, t[0], t[1], t[2], t[3], o, lse)
    # in place into the first operand
    usp.usp_ring_merge(rows, d, t[0], t[1], t[2], t[3], t[0], t[1])
    torch.cuda.synchronize()
    for oo, ll in ((o, lse), (t[0], t[1])):
        assert max_abs(oo.cpu().numpy(), ref_o) < 1e-5
        lh = ll.cpu().numpy()
        assert np.array_equal(np.isinf(lh), np.isinf(ref_l))
        fin = np.isfinite(ref_l)
        assert max_abs(lh[fin], ref_l[fin]) < 1e-5


@pytest.mark.parametrize("B,H,Hkv,N,d,P,causal", [
    (1, 4, 4, 2048, 128, 4, True), (1, 4, 2, 1536, 64, 3, True), (2, 2, 2, 1000, 128, 2, True),
    (1, 4, 4, 1024, 128, 4, False)])
def test_ring_attention_small(usp, orc, B, H, Hkv, N, d, P, causal):
    import torch
    p = usp.Problem(B=B, Hq=H, Hkv=Hkv, N=N, d=d, P=P, causal=causal)
    q, k, v = gen((B, H, N, d), 0), gen((B, Hkv, N, d), 1), gen((B, Hkv, N, d), 2)
    o, lse = usp.ring_attention_fwd(p, to_dev(to_seq(q, P)), to_dev(to_seq(k, P)), to_dev(to_seq(v, P)))
    torch.cuda.synchronize()
    o_ref, lse_ref = orc.attn_rows(q, k, v, causal=causal)
    o_log = from_seq(to_host(o))
    lse_log = np.ascontiguousarray(to_host(lse).transpose(1, 3, 0, 2).reshape(B, H, N))
    _check_fwd(o_log, lse_log, o_ref, lse_ref)
    _status_ok(usp)


@pytest.mark.parametrize("B,H,Hkv,N,d,P,causal", [
    (1, 4, 4, 2048, 128, 4, True),     # four ranks of 512 tokens
    (1, 4, 2, 1536, 64, 3, True),      # GQA, three ranks
    (2, 2, 2, 1000, 128, 2, True),     # two sequences, ragged shards of 500 tokens
    (1, 4, 4, 1024, 128, 4, False),    # full attention: every block pair, no mask
    (1, 8, 2, 600, 128, 2, True)])     # shards of 300 tokens, GQA group of 4
def test_ring_attention_backward_small(usp, orc, B, H, Hkv, N, d, P, causal):
    """Ring backward (fp32 accumulation of per-step partials) against the oracle's full backward."""
    import torch
    p = usp.Problem(B=B, Hq=H, Hkv=Hkv, N=N, d=d, P=P, causal=causal)
    q, k, v, dO = gen((B, H, N, d), 0), gen((B, Hkv, N, d), 1), gen((B, Hkv, N, d), 2), gen((B, H, N, d), 3)
    qs, ks, vs, dos = (to_dev(to_seq(x, P)) for x in (q, k, v, dO))
    o, lse = usp.ring_attention_fwd(p, qs, ks, vs)
    dq, dk, dv = usp.ring_attention_bwd(p, qs, ks, vs, o, lse, dos)
    torch.cuda.synchronize()
    out = dict(dq=from_seq(to_host(dq)), dk=from_seq(to_host(dk)), dv=from_seq(to_host(dv)))
    ref_dq, ref_dk, ref_dv, _, _ = orc.attn_bwd_full(q, k, v, dO, causal=causal)
    _check_grads(out, ref_dq, ref_dk, ref_dv)
    _status_ok(usp)


@pytest.mark.parametrize("B,H,Hkv,N,d,P,causal", [
    (1, 4, 4, 1024, 128, 4, True),     # four ranks of 256 tokens
    (2, 4, 2, 1000, 64, 2, True),      # two sequences, GQA, ragged shards of 500 tokens
    (1, 8, 2, 600, 128, 2, True),      # shards of 300 tokens: tiles straddle the rank boundary
    (1, 4, 4, 768, 128, 3, False)])    # full attention
def test_allgather_kv_fwd_bwd(usp, orc, B, H, Hkv, N, d, P, causal):
    """All-gather-KV context parallelism: every rank attends its query shard against all keys."""
    import torch
    p = usp.Problem(B=B, Hq=H, Hkv=Hkv, N=N, d=d, P=P, causal=causal)
    q, k, v, dO = gen((B, H, N, d), 0), gen((B, Hkv, N, d), 1), gen((B, Hkv, N, d), 2), gen((B, H, N, d), 3)
    qs, ks, vs, dos = (to_dev(to_seq(x, P)) for x in (q, k, v, dO))
    o, lse = usp.allgather_attention_fwd(p, qs, ks, vs)
    dq, dk, dv = usp.allgather_attention_bwd(p, qs, ks, vs, o, lse, dos)
    torch.cuda.synchronize()
    o_ref, lse_ref = orc.attn_rows(q, k, v, causal=causal)
    lse_log = np.ascontiguousarray(to_host(lse).transpose(1, 3, 0, 2).reshape(B, H, N))
    _check_fwd(from_seq(to_host(o)), lse_log, o_ref, lse_ref)
    out = dict(dq=from_seq(to_host(dq)), dk=from_seq(to_host(dk)), dv=from_seq(to_host(dv)))
    ref_dq, ref_dk, ref_dv, _, _ = orc.attn_bwd_full(q, k, v, dO, causal=causal)
    _check_grads(out, ref_dq, ref_dk, ref_dv)
    _status_ok(usp)


def _zigzag_host(x_seq, P):
    """contiguous shards [P][B][2c][H][d] -> zigzag shards (rank r: chunks r, 2P-1-r), host-side index map."""
    Pn, B, Np, H, d = x_seq.shape
    c = Np // 2
    chunks = x_seq.reshape(P, B, 2, c, H, d).transpose(1, 0, 2, 3, 4, 5).reshape(B, 2 * P, c, H, d)  # [B][g]
    out = np.empty((P, B, 2, c, H, d), dtype=x_seq.dtype)
    for r in range(P):
        out[r, :, 0] = chunks[:, r]
        out[r, :, 1] = chunks[:, 2 * P - 1 - r]
    return out.reshape(P, B, Np, H, d)


@pytest.mark.parametrize("dtype,B,H,N,d,P", [("bf16", 1, 4, 2048, 128, 4), ("f32", 2, 3, 600, 64, 3)])
def test_zigzag_shard_bit_exact(usp, dtype, B, H, N, d, P):
    import torch
    p = usp.Problem(B=B, Hq=H, Hkv=H, N=N, d=d, P=P, dtype=dtype)
    x = gen((B, H, N, d), 5, dtype=dtype)
    seq = to_seq(x, P)
    src = to_dev(seq, dtype)
    zz = torch.empty_like(src)
    back = torch.empty_like(src)
    usp.usp_zigzag_shard(p, H, src, zz)
    usp.usp_zigzag_unshard(p, H, zz, back)
    torch.cuda.synchronize()
    assert to_host(zz).tobytes() == _zigzag_host(to_host(src), P).tobytes()
    assert to_host(back).tobytes() == to_host(src).tobytes()


@pytest.mark.parametrize("B,H,Hkv,N,d,P,causal", [
    (1, 4, 4, 2048, 128, 4, True),     # chunks of 256 tokens
    (2, 4, 2, 1200, 64, 2, True),      # two sequences, GQA, chunks of 300 tokens
    (1, 8, 2, 1536, 128, 3, True),     # three ranks, GQA group of 4
    (1, 4, 4, 1024, 128, 2, False)])   # full attention
def test_zigzag_ring_fwd_bwd(usp, orc, B, H, Hkv, N, d, P, causal):
    """Zigzag ring attention (forward and backward) against the oracle, through the shard/unshard maps."""
    import torch
    p = usp.Problem(B=B, Hq=H, Hkv=Hkv, N=N, d=d, P=P, causal=causal)
    q, k, v, dO = gen((B, H, N, d), 0), gen((B, Hkv, N, d), 1), gen((B, Hkv, N, d), 2), gen((B, H, N, d), 3)

    def zz(x, h):
        s = to_dev(to_seq(x, P))
        out = torch.empty_like(s)
        usp.usp_zigzag_shard(p, h, s, out)
        return out

    def unzz(x, h):
        out = torch.empty_like(x)
        usp.usp_zigzag_unshard(p, h, x, out)
        return out

    qz, kz, vz, doz = zz(q, H), zz(k, Hkv), zz(v, Hkv), zz(dO, H)
    o, lse = usp.zigzag_attention_fwd(p, qz, kz, vz)
    dq, dk, dv = usp.zigzag_attention_bwd(p, qz, kz, vz, o, lse, doz)
    # lse through the same chunk permutation (one "head" of d = 1 is not a valid problem: permute on the host)
    torch.cuda.synchronize()
    o_log = from_seq(to_host(unzz(o, H)))
    lz = to_host(lse).reshape(P, B, 2, N // (2 * P), H)
    lse_seq = np.empty_like(lz)
    for r in range(P):
        for h2 in range(2):
            g = r if h2 == 0 else 2 * P - 1 - r
            lse_seq[g // 2, :, g % 2] = lz[r, :, h2]
    lse_log = np.ascontiguousarray(lse_seq.reshape(P, B, N // P, H).transpose(1, 3, 0, 2).reshape(B, H, N))
    o_ref, lse_ref = orc.attn_rows(q, k, v, causal=causal)
    _check_fwd(o_log, lse_log, o_ref, lse_ref)
    out = dict(dq=from_seq(to_host(unzz(dq, H))), dk=from_seq(to_host(unzz(dk, Hkv))),
               dv=from_seq(to_host(unzz(dv, Hkv))))
    ref_dq, ref_dk, ref_dv, _, _ = orc.attn_bwd_full(q, k, v, dO, causal=causal)
    _check_grads(out, ref_dq, ref_dk, ref_dv)
    _status_ok(usp)


# ---------------------------------------------------------------- all-to-all fused into attention
@pytest.mark.parametrize("B,Hq,Hkv,N,d,P,causal", [
    (1, 8, 4, 1024, 128, 4, True),     # GQA, four shards of 256 tokens
    (1, 16, 4, 512, 128, 4, True),     # GQA group of 4, shards of one tile
    (2, 4, 4, 512, 64, 2, True),       # two sequences
    (1, 4, 2, 768, 128, 2, False),     # full attention, shards of 384 tokens
    (1, 2, 2, 256, 64, 1, True),       # one rank
    (1, 8, 8, 1024, 128, 8, True),     # eight shards of one 128-row tile each
    (1, 6, 3, 384, 64, 3, True)])      # three shards: the last 256-row block's second tile is past N
def test_fused_equals_remapped(usp, B, Hq, Hkv, N, d, P, causal):
    """Attention reading and writing the sequence-sharded layout in place gives the remapped
    path's O, LSE, dK and dV bit for bit (the same per-head work, tile for tile), and its dQ to
    one bf16 unit (both add the same float32 dQ partials, in orders that vary from run to run)."""
    import torch
    p = usp.Problem(B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, P=P, causal=causal)
    q, k, v, dO = gen((B, Hq, N, d), 0), gen((B, Hkv, N, d), 1), gen((B, Hkv, N, d), 2), gen((B, Hq, N, d), 3)
    qs, ks, vs, dos = (to_dev(to_seq(x, P)) for x in (q, k, v, dO))
    o_r, saved = usp.ulysses_attention_fwd(p, qs, ks, vs)
    dq_r, dk_r, dv_r = usp.ulysses_attention_bwd(p, saved, dos)
    o, lse = usp.fused_attention_fwd(p, qs, ks, vs)
    dq, dk, dv = usp.fused_attention_bwd(p, qs, ks, vs, o, lse, dos)
    torch.cuda.synchronize()
    for got, want in ((o, o_r), (dk, dk_r), (dv, dv_r)):
        assert to_host(got).tobytes() == to_host(want).tobytes()
    assert bf16_ulp_diff(to_host(dq), to_host(dq_r)) <= 1.0
    assert lse_from_seq(to_host(lse)).tobytes() == from_head(to_host(saved["lse"])).tobytes()
    _status_ok(usp)


# ---------------------------------------------------------------- one-pass backward vs the three-pass one
@pytest.mark.parametrize("B,Hq,Hkv,N,d,P,causal", [
    (1, 8, 2, 1000, 128, 2, True),     # GQA group of 4, ragged last tile
    (2, 4, 4, 640, 64, 2, True),       # two sequences, d = 64
    (1, 4, 2, 768, 128, 2, False),     # full attention
    (1, 2, 2, 130, 128, 1, True),      # one rank, two tiles, the second almost empty
    (1, 16, 4, 2048, 64, 4, True)])    # GQA at d = 64, 16 query tiles
def test_one_pass_backward_matches_three_pass(usp, orc, B, Hq, Hkv, N, d, P, causal):
    """usp_attn_bwd (S and dP once per block pair, dQ partials added into a float32 accumulator)
    against usp_attn_bwd_deterministic (dK/dV pass, then a dQ pass): dK and dV bit for bit; dQ
    within a tenth of the gradient tolerance (relative Frobenius), and each against the oracle on
    every element.  The dQ pass of the three-pass backward recomputes dS with its own rounding
    (lse and D subtracted in registers instead of inside the product), so its bf16 dS can differ
    from the one dK uses in the last bit: on entries of dQ whose terms nearly cancel, the two dQ
    then differ by more than a unit of the (small) result."""
    import torch
    p = usp.Problem(B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, P=P, causal=causal)
    q, k, v, dO = gen((B, Hq, N, d), 0), gen((B, Hkv, N, d), 1), gen((B, Hkv, N, d), 2), gen((B, Hq, N, d), 3)
    qh, kh, vh, doh = (to_dev(to_head(x, P)) for x in (q, k, v, dO))
    oh = torch.empty_like(qh)
    lse = torch.empty(p.lse_head_shape(), dtype=torch.float32, device="cuda")
    usp.usp_attn_fwd(p, qh, kh, vh, oh, lse)
    one = [torch.empty_like(qh), torch.empty_like(kh), torch.empty_like(vh)]
    three = [torch.empty_like(qh), torch.empty_like(kh), torch.empty_like(vh)]
    ws1 = torch.empty(usp.usp_attn_bwd_workspace_size(p), dtype=torch.uint8, device="cuda")
    ws3 = torch.empty(usp.usp_attn_bwd_deterministic_workspace_size(p), dtype=torch.uint8, device="cuda")
    usp.usp_attn_bwd(p, qh, kh, vh, oh, lse, doh, *one, ws1)
    usp.usp_attn_bwd_deterministic(p, qh, kh, vh, oh, lse, doh, *three, ws3)
    torch.cuda.synchronize()
    _status_ok(usp)
    assert to_host(one[1]).tobytes() == to_host(three[1]).tobytes()
    assert to_host(one[2]).tobytes() == to_host(three[2]).tobytes()
    dq1, dq3 = f64(from_head(to_host(one[0]))), f64(from_head(to_host(three[0])))
    assert rel_fro(dq1, dq3) < 0.1 * TOL_BF16_GRAD_RELFRO
    # each dQ against the oracle, every element
    ref_dq, _, _, _, _ = orc.attn_bwd_full(q, k, v, dO, causal=causal)
    assert rel_fro(dq1, ref_dq) < TOL_BF16_GRAD_RELFRO
    assert rel_fro(dq3, ref_dq) < TOL_BF16_GRAD_RELFRO


def test_fused_against_oracle_mean_square_loss(usp, orc):
    """The fused path against the float64 oracle on its own: loss mean(out^2), GQA, four shards."""
    import torch
    B, Hq, Hkv, N, d, P = 1, 8, 4, 2048, 128, 4
    p = usp.Problem(B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, P=P)
    q, k, v = gen((B, Hq, N, d), 0), gen((B, Hkv, N, d), 1), gen((B, Hkv, N, d), 2)
    qs, ks, vs = (to_dev(to_seq(x, P)) for x in (q, k, v))
    o, lse = usp.fused_attention_fwd(p, qs, ks, vs)
    do_seq = (2.0 * o.float() / o.numel()).to(torch.bfloat16)
    dq, dk, dv = usp.fused_attention_bwd(p, qs, ks, vs, o, lse, do_seq)
    torch.cuda.synchronize()
    o_ref, lse_ref = orc.attn_rows(q, k, v, causal=True)
    _check_fwd(from_seq(to_host(o)), lse_from_seq(to_host(lse)), o_ref, lse_ref)
    dO_ref = (2.0 * o_ref / o_ref.size).astype(np.float32)
    ref_dq, ref_dk, ref_dv, _, _ = orc.attn_bwd_full(q, k, v, dO_ref, causal=True)
    out = dict(dq=from_seq(to_host(dq)), dk=from_seq(to_host(dk)), dv=from_seq(to_host(dv)))
    _check_grads(out, ref_dq, ref_dk, ref_dv)
    _status_ok(usp)


# ---------------------------------------------------------------- 2-D (hybrid) Ulysses x ring
@pytest.mark.parametrize("dtype,B,H,N,d,P,Pu", [
    ("bf16", 2, 8, 1200, 128, 4, 2), ("f32", 1, 6, 768, 64, 6, 3), ("bf16", 1, 4, 512, 64, 4, 1),
    ("bf16", 1, 8, 512, 128, 4, 4)])
def test_hybrid_remap_bit_exact(usp, orc, dtype, B, H, N, d, P, Pu):
    """The all-to-all inside each ring group: the oracle's Ulysses map on the group's shards."""
    import torch
    p = usp.Problem(B=B, Hq=H, Hkv=H, N=N, d=d, P=P, dtype=dtype)
    x = gen((B, H, N, d), 4, dtype)
    seq = to_seq(x, P)
    src = to_dev(seq, dtype)
    hyb = torch.empty(p.hybrid_shape(H, Pu), dtype=p.torch_dtype, device="cuda")
    back = torch.empty_like(src)
    usp.usp_hybrid_seq2head(p, Pu, H, src, hyb)
    usp.usp_hybrid_head2seq(p, Pu, H, hyb, back)
    _sync()
    want = np.concatenate([orc.seq2head(seq[g * Pu:(g + 1) * Pu]) for g in range(P // Pu)])
    assert to_host(hyb).tobytes() == want.tobytes()
    assert to_host(hyb).tobytes() == to_hybrid(x, P, Pu).tobytes()
    assert to_host(back).tobytes() == seq.tobytes()
    _status_ok(usp)


@pytest.mark.parametrize("B,Hq,Hkv,N,d,P,Pu,causal", [
    (1, 8, 4, 2048, 128, 4, 2, True),     # two ring groups of two Ulysses ranks
    (2, 4, 2, 1200, 64, 4, 2, True),      # two sequences, GQA, chunks of 600 tokens (ragged tiles)
    (1, 8, 8, 1536, 128, 6, 2, True),     # three ring groups
    (1, 8, 2, 1024, 128, 4, 2, False)])   # full attention, GQA group of 4
def test_hybrid_fwd_bwd(usp, orc, B, Hq, Hkv, N, d, P, Pu, causal):
    """2-D sequence parallelism (forward and backward) against the oracle."""
    import torch
    p = usp.Problem(B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, P=P, causal=causal)
    q, k, v, dO = gen((B, Hq, N, d), 0), gen((B, Hkv, N, d), 1), gen((B, Hkv, N, d), 2), gen((B, Hq, N, d), 3)
    qs, ks, vs, dos = (to_dev(to_seq(x, P)) for x in (q, k, v, dO))
    o, saved = usp.hybrid_attention_fwd(p, Pu, qs, ks, vs)
    dq, dk, dv = usp.hybrid_attention_bwd(p, Pu, saved, dos)
    torch.cuda.synchronize()
    o_ref, lse_ref = orc.attn_rows(q, k, v, causal=causal)
    _check_fwd(from_seq(to_host(o)), from_hybrid(to_host(saved["lse"]), Pu), o_ref, lse_ref)
    ref_dq, ref_dk, ref_dv, _, _ = orc.attn_bwd_full(q, k, v, dO, causal=causal)
    out = dict(dq=from_seq(to_host(dq)), dk=from_seq(to_host(dk)), dv=from_seq(to_host(dv)))
    _check_grads(out, ref_dq, ref_dk, ref_dv)
    _status_ok(usp)


def test_hybrid_reduces_to_ulysses_and_ring_bitwise(usp):
    """Pu = P is one ring group: the Ulysses path; Pu = 1 is the ring.  Both bit for bit, except dQ
    to one bf16 unit (every path adds its float32 dQ partials in an order that varies)."""
    import torch
    B, Hq, Hkv, N, d, P = 1, 8, 4, 1024, 128, 4
    p = usp.Problem(B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, P=P)
    q, k, v, dO = gen((B, Hq, N, d), 0), gen((B, Hkv, N, d), 1), gen((B, Hkv, N, d), 2), gen((B, Hq, N, d), 3)
    qs, ks, vs, dos = (to_dev(to_seq(x, P)) for x in (q, k, v, dO))
    o_u, saved_u = usp.ulysses_attention_fwd(p, qs, ks, vs)
    g_u = usp.ulysses_attention_bwd(p, saved_u, dos)
    o_h, saved_h = usp.hybrid_attention_fwd(p, P, qs, ks, vs)
    g_h = usp.hybrid_attention_bwd(p, P, saved_h, dos)
    o_r, lse_r = usp.ring_attention_fwd(p, qs, ks, vs)
    g_r = usp.ring_attention_bwd(p, qs, ks, vs, o_r, lse_r, dos)
    o_1, saved_1 = usp.hybrid_attention_fwd(p, 1, qs, ks, vs)
    g_1 = usp.hybrid_attention_bwd(p, 1, saved_1, dos)
    torch.cuda.synchronize()
    for got, want in zip((o_h, *g_h[1:]), (o_u, *g_u[1:])):
        assert to_host(got).tobytes() == to_host(want).tobytes()
    assert bf16_ulp_diff(to_host(g_h[0]), to_host(g_u[0])) <= 1.0
    assert to_host(saved_h["lse"]).tobytes() == to_host(saved_u["lse"]).tobytes()
    for got, want in zip((o_1, *g_1[1:]), (o_r, *g_r[1:])):
        assert to_host(got).tobytes() == to_host(want).tobytes()
    assert bf16_ulp_diff(to_host(g_1[0]), to_host(g_r[0])) <= 1.0
    assert from_hybrid(to_host(saved_1["lse"]), 1).tobytes() == lse_from_seq(to_host(lse_r)).tobytes()
    _status_ok(usp)


# ---------------------------------------------------------------- failure detection
def test_step_captured_in_a_cuda_graph(usp):
    """The whole Ulysses step (remaps, forward, backward, remaps back) captured once into a CUDA
    graph and replayed gives the eagerly launched step's results: O, dK, dV bit for bit, dQ to one
    bf16 unit (its float32 partial sums are added in an order that varies). Every call only
    enqueues work on the stream it is given, so a caller can capture it."""
    import torch
    B, Hq, Hkv, N, d, P = 1, 8, 2, 1280, 128, 2
    p = usp.Problem(B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, P=P)
    q, k, v, dO = gen((B, Hq, N, d), 40), gen((B, Hkv, N, d), 41), gen((B, Hkv, N, d), 42), gen((B, Hq, N, d), 43)
    qs, ks, vs, dos = (to_dev(to_seq(x, P)) for x in (q, k, v, dO))
    bf = torch.bfloat16
    qh, oh, doh, dqh = (torch.empty(p.head_shape(Hq), dtype=bf, device="cuda") for _ in range(4))
    kh, vh, dkh, dvh = (torch.empty(p.head_shape(Hkv), dtype=bf, device="cuda") for _ in range(4))
    lse = torch.empty(p.lse_head_shape(), dtype=torch.float32, device="cuda")
    outs = [torch.empty_like(qs), torch.empty_like(qs), torch.empty_like(ks), torch.empty_like(vs)]
    ws = torch.empty(usp.usp_attn_bwd_workspace_size(p), dtype=torch.uint8, device="cuda")

    def step(sh):
        usp.usp_a2a_seq2head(p, Hq, qs, qh, sh)
        usp.usp_a2a_seq2head(p, Hkv, ks, kh, sh)
        usp.usp_a2a_seq2head(p, Hkv, vs, vh, sh)
        usp.usp_attn_fwd(p, qh, kh, vh, oh, lse, sh)
        usp.usp_a2a_head2seq(p, Hq, oh, outs[0], sh)
        usp.usp_a2a_seq2head(p, Hq, dos, doh, sh)
        usp.usp_attn_bwd(p, qh, kh, vh, oh, lse, doh, dqh, dkh, dvh, ws, None, sh)
        usp.usp_a2a_head2seq(p, Hq, dqh, outs[1], sh)
        usp.usp_a2a_head2seq(p, Hkv, dkh, outs[2], sh)
        usp.usp_a2a_head2seq(p, Hkv, dvh, outs[3], sh)

    step(torch.cuda.current_stream().cuda_stream)
    _sync()
    eager = [t.clone() for t in outs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(torch.cuda.current_stream().cuda_stream)
    for t in outs:
        t.zero_()
    g.replay()
    _sync()
    _status_ok(usp)
    for i in (0, 2, 3):
        assert torch.equal(outs[i].view(torch.int16), eager[i].view(torch.int16))
    assert bf16_ulp_diff(to_host(outs[1]), to_host(eager[1])) <= 1.0
    # a replay after new inputs are written into the captured buffers follows them
    qs.copy_(to_dev(to_seq(gen((B, Hq, N, d), 44), P)))
    g.replay()
    _sync()
    replayed = [t.clone() for t in outs]
    step(torch.cuda.current_stream().cuda_stream)
    _sync()
    _status_ok(usp)
    assert not torch.equal(replayed[0], eager[0])
    for i in (0, 2, 3):
        assert torch.equal(replayed[i].view(torch.int16), outs[i].view(torch.int16))


def test_bounded_wait_times_out_and_the_context_survives(usp):
    """A wait that nothing completes gives up after the 2 s limit: the host reads USP_ERR_TIMEOUT,
    the word is cleared, and the next work on the same context runs and is correct."""
    import time

    import torch
    from context_long_attention_ulysses_gb300 import _lib
    assert usp.usp_device_status() == _lib.USP_OK
    t0 = time.perf_counter()
    usp.usp_diag_wait_timeout()
    assert usp.usp_device_status() == _lib.USP_ERR_TIMEOUT   # synchronises, reads and clears the word
    assert time.perf_counter() - t0 > 1.9                    # the wait ran to its limit
    assert usp.usp_device_status() == _lib.USP_OK
    p = usp.Problem(B=1, Hq=4, Hkv=4, N=512, d=128, P=2)
    x = gen((1, 4, 512, 128), 6)
    src = to_dev(to_seq(x, 2))
    head = torch.empty(p.head_shape(4), dtype=torch.bfloat16, device="cuda")
    usp.usp_a2a_seq2head(p, 4, src, head)
    _sync()
    assert to_host(head).tobytes() == to_head(x, 2).tobytes()
    _status_ok(usp)


def test_aborted_attention_kernels_drain_and_the_context_survives(usp):
    """The status word is set before real attention launches, so every CTA of the forward, the
    one-pass backward and the three-pass backward's dK/dV and dQ kernels gives up at its first wait
    that is not yet satisfied, with its TMA loads and MMAs in flight. Each CTA waits for those
    before it frees TMEM and exits. The launches end fast (no drain ran to its 2 s limit), the host
    reads USP_ERR_TIMEOUT once, and the same context then gives the clean run's results: bit for
    bit, except the one-pass dQ, to one bf16 unit (its float32 additions' order varies)."""
    import time

    import torch
    from context_long_attention_ulysses_gb300 import _lib
    B, Hq, Hkv, N, d, P = 1, 8, 2, 4096, 128, 2
    p = usp.Problem(B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, P=P)
    q, k, v, dO = gen((B, Hq, N, d), 0), gen((B, Hkv, N, d), 1), gen((B, Hkv, N, d), 2), gen((B, Hq, N, d), 3)
    qh, kh, vh, doh = (to_dev(to_head(x, P)) for x in (q, k, v, dO))
    ws = torch.empty(usp.usp_attn_bwd_workspace_size(p), dtype=torch.uint8, device="cuda")

    def run():
        o = torch.empty_like(qh)
        lse = torch.empty(p.lse_head_shape(), dtype=torch.float32, device="cuda")
        grads = [torch.empty_like(qh), torch.empty_like(kh), torch.empty_like(vh)]
        grads3 = [torch.empty_like(qh), torch.empty_like(kh), torch.empty_like(vh)]
        usp.usp_attn_fwd(p, qh, kh, vh, o, lse)
        usp.usp_attn_bwd(p, qh, kh, vh, o, lse, doh, *grads, ws)
        usp.usp_attn_bwd_deterministic(p, qh, kh, vh, o, lse, doh, *grads3, ws)
        return [o, lse, *grads, *grads3]

    assert usp.usp_device_status() == _lib.USP_OK
    clean = [to_host(t) for t in run()]
    _sync()
    t0 = time.perf_counter()
    usp.usp_diag_raise_status()
    run()
    assert usp.usp_device_status() == _lib.USP_ERR_TIMEOUT   # synchronises, reads and clears the word
    assert time.perf_counter() - t0 < 1.5                     # every CTA gave up fast and drained at once
    assert usp.usp_device_status() == _lib.USP_OK
    again = [to_host(t) for t in run()]
    _status_ok(usp)
    for i, (got, want) in enumerate(zip(again, clean)):
        if i == 2:  # the one-pass dQ
            assert bf16_ulp_diff(got, want) <= 1.0
        else:
            assert got.tobytes() == want.tobytes()


# ---------------------------------------------------------------- writes stay inside their buffers
def test_no_write_outside_any_buffer(usp):
    """Every output and workspace of every path sits between 4 KiB guard regions (a fixed byte
    pattern); after the remapped, fused, ring, zigzag, all-gather and 2-D paths ran forward and
    backward, every guard is unchanged.  Ragged 300- and 600-token shards, two sequences, GQA."""
    import torch
    from tests.guarded import Guarded
    dev = "cuda"
    damaged = {}

    def inputs(p):
        q = to_dev(to_seq(gen((p.B, p.Hq, p.N, p.d), 0), p.P))
        k = to_dev(to_seq(gen((p.B, p.Hkv, p.N, p.d), 1), p.P))
        v = to_dev(to_seq(gen((p.B, p.Hkv, p.N, p.d), 2), p.P))
        do = to_dev(to_seq(gen((p.B, p.Hq, p.N, p.d), 3), p.P))
        return q, k, v, do

    # remapped Ulysses and the fused path (shards of whole 128-row tiles)
    p = usp.Problem(B=2, Hq=4, Hkv=2, N=512, d=128, P=2)
    q, k, v, do = inputs(p)
    g = Guarded()
    qh, oh, doh, dqh = (g.empty(p.head_shape(p.Hq), torch.bfloat16, dev) for _ in range(4))
    kh, vh, dkh, dvh = (g.empty(p.head_shape(p.Hkv), torch.bfloat16, dev) for _ in range(4))
    lse = g.empty(p.lse_head_shape(), torch.float32, dev)
    o, dq = g.empty_like(q), g.empty_like(q)
    dk, dv = g.empty_like(k), g.empty_like(v)
    ws = g.bytes(usp.usp_attn_bwd_workspace_size(p), dev)
    usp.usp_a2a_seq2head(p, p.Hq, q, qh)
    usp.usp_a2a_seq2head(p, p.Hkv, k, kh)
    usp.usp_a2a_seq2head(p, p.Hkv, v, vh)
    usp.usp_attn_fwd(p, qh, kh, vh, oh, lse)
    usp.usp_a2a_head2seq(p, p.Hq, oh, o)
    usp.usp_a2a_seq2head(p, p.Hq, do, doh)
    usp.usp_attn_bwd(p, qh, kh, vh, oh, lse, doh, dqh, dkh, dvh, ws)
    for src, dst, h in ((dqh, dq, p.Hq), (dkh, dk, p.Hkv), (dvh, dv, p.Hkv)):
        usp.usp_a2a_head2seq(p, h, src, dst)
    _sync()
    damaged["remapped"] = g.damaged()
    g = Guarded()
    o, dq = g.empty_like(q), g.empty_like(q)
    dk, dv = g.empty_like(k), g.empty_like(v)
    lse = g.empty(p.lse_seq_shape(), torch.float32, dev)
    ws = g.bytes(usp.usp_fused_attn_bwd_workspace_size(p), dev)
    usp.usp_fused_attn_fwd(p, q, k, v, o, lse)
    usp.usp_fused_attn_bwd(p, q, k, v, o, lse, do, dq, dk, dv, ws)
    _sync()
    damaged["fused"] = g.damaged()

    # sequence-sharded paths on ragged shards of 300 tokens (2-D: chunks of 600)
    p = usp.Problem(B=2, Hq=4, Hkv=2, N=1200, d=64, P=4)
    q, k, v, do = inputs(p)
    for name, fwd, bwd, ws_f, ws_b in (
            ("ring", usp.usp_ring_attn_fwd, usp.usp_ring_attn_bwd, usp.usp_ring_workspace_size,
             usp.usp_ring_bwd_workspace_size),
            ("zigzag", usp.usp_zigzag_attn_fwd, usp.usp_zigzag_attn_bwd, usp.usp_zigzag_workspace_size,
             usp.usp_zigzag_bwd_workspace_size),
            ("allgather", usp.usp_allgather_attn_fwd, usp.usp_allgather_attn_bwd,
             usp.usp_allgather_workspace_size, usp.usp_allgather_bwd_workspace_size)):
        g = Guarded()
        o, dq = g.empty_like(q), g.empty_like(q)
        dk, dv = g.empty_like(k), g.empty_like(v)
        lse = g.empty(p.lse_seq_shape(), torch.float32, dev)
        ws, bws = g.bytes(ws_f(p), dev), g.bytes(ws_b(p), dev)
        fwd(p, q, k, v, o, lse, ws)
        bwd(p, q, k, v, o, lse, do, dq, dk, dv, bws)
        _sync()
        damaged[name] = g.damaged()
    Pu = 2
    g = Guarded()
    hq, ho, hdo, hdq = (g.empty(p.hybrid_shape(p.Hq, Pu), torch.bfloat16, dev) for _ in range(4))
    hk, hv, hdk, hdv = (g.empty(p.hybrid_shape(p.Hkv, Pu), torch.bfloat16, dev) for _ in range(4))
    hlse = g.empty(p.lse_hybrid_shape(Pu), torch.float32, dev)
    ws, bws = g.bytes(usp.usp_hybrid_workspace_size(p, Pu), dev), g.bytes(usp.usp_hybrid_bwd_workspace_size(p, Pu), dev)
    o, dq = g.empty_like(q), g.empty_like(q)
    usp.usp_hybrid_seq2head(p, Pu, p.Hq, q, hq)
    usp.usp_hybrid_seq2head(p, Pu, p.Hkv, k, hk)
    usp.usp_hybrid_seq2head(p, Pu, p.Hkv, v, hv)
    usp.usp_hybrid_seq2head(p, Pu, p.Hq, do, hdo)
    usp.usp_hybrid_attn_fwd(p, Pu, hq, hk, hv, ho, hlse, ws)
    usp.usp_hybrid_attn_bwd(p, Pu, hq, hk, hv, ho, hlse, hdo, hdq, hdk, hdv, bws)
    usp.usp_hybrid_head2seq(p, Pu, p.Hq, ho, o)
    usp.usp_hybrid_head2seq(p, Pu, p.Hq, hdq, dq)
    _sync()
    damaged["2-D"] = g.damaged()
    assert all(not v_ for v_ in damaged.values()), damaged
    _status_ok(usp)


"""Pins of the float64 oracle against things other than itself.

Each test checks the oracle against what the pages or the mathematics fix:
worked examples printed on the pages (tests/golden/), library special cases
(numpy reshape/transpose, scipy logsumexp + matmul), closed forms,
invariants, brute force on tiny inputs and finite differences.  CPU only.
"""
import os

import numpy as np
import pytest
from scipy.special import logsumexp

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([float(x) if "." in x else int(x) for x in line.split()])
    return rows


def _coded(shape, dtype=np.float32):
    """Array whose every element is distinct (its flat index)."""
    n = int(np.prod(shape))
    if dtype == np.uint16:
        assert n < 65536
        return np.arange(n, dtype=np.uint16).reshape(shape)
    return np.arange(n, dtype=np.float32).reshape(shape)


def _brute(q, k, v, causal, scale):
    """Full softmax(scale*QK^T + mask) V with scipy/numpy (GQA by repeat)."""
    B, Hq, N, d = q.shape
    g = Hq // k.shape[1]
    kk = np.repeat(k, g, axis=1)
    vv = np.repeat(v, g, axis=1)
    s = scale * np.einsum("bhid,bhjd->bhij", q, kk)
    if causal:
        s = np.where(np.tril(np.ones((N, N), dtype=bool)), s, -np.inf)
    lse = logsumexp(s, axis=-1)
    p = np.exp(s - lse[..., None])
    return p @ vv, lse


def _rand(shape, stream, dtype="f32", seed=7):
    x = synth.normal(shape, seed=seed, stream=stream, dtype=dtype)
    return x


# ------------------------------------------------------------------ generator
def test_philox_known_answers():
    # Known-answer vectors of Philox4x32-10 published with the Random123
    # reference implementation (Salmon et al., SC'11).
    assert list(synth.philox4x32_10([0, 0, 0, 0], [0, 0])) == [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]
    assert list(synth.philox4x32_10([0xFFFFFFFF] * 4, [0xFFFFFFFF] * 2)) == [
        0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD]
    assert list(synth.philox4x32_10([0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344],
                                    [0xA4093822, 0x299F31D0])) == [0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1]


def test_generator_distribution_and_bf16_rounding():
    x = synth.normal((1 << 20,), seed=0, stream=0)
    assert abs(float(x.mean())) < 5e-3 and abs(float(x.std()) - 1.0) < 5e-3
    xb = synth.normal((1 << 20,), seed=0, stream=0, dtype="bf16")
    assert np.array_equal(xb, synth.f32_to_bf16(x))
    # round-to-nearest-even on exact ties
    ties = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8)], dtype=np.float32)
    assert list(synth.bf16_to_f32(synth.f32_to_bf16(ties))) == [1.0, 1.0 + 2.0 ** -6, -1.0]
    # offset selects a later part of the same sequence
    assert np.array_equal(synth.normal((100,), seed=0, stream=0, offset=37), x[37:137])


# ---------------------------------------------------------------- layout maps
def test_shard_golden_worked_example(orc):
    N, P, per, *firsts = _golden("shard_split.txt")[0]
    x = _coded((1, 1, N, 1))
    s = orc.shard_seq(x, P)
    assert s.shape == (P, 1, per, 1, 1)
    for p in range(P):
        assert s[p, 0, 0, 0, 0] == firsts[p]
        assert np.array_equal(s[p, 0, :, 0, 0], np.arange(firsts[p], firsts[p] + per, dtype=np.float32))


@pytest.mark.parametrize("B,H,N,d,P", [(1, 4, 16, 3, 2), (2, 8, 12, 2, 4), (3, 2, 6, 5, 1), (2, 6, 18, 4, 3)])
def test_shard_seq_is_reshape_transpose(orc, B, H, N, d, P):
    x = _coded((B, H, N, d))
    ref = x.reshape(B, H, P, N // P, d).transpose(2, 0, 3, 1, 4)
    s = orc.shard_seq(x, P)
    assert np.array_equal(s, ref)
    assert np.array_equal(orc.unshard_seq(s), x)


@pytest.mark.parametrize("B,H,N,d,P", [(1, 4, 16, 3, 2), (2, 8, 12, 2, 4), (2, 6, 18, 4, 3), (1, 8, 8, 1, 8)])
@pytest.mark.parametrize("dtype", [np.float32, np.uint16])
def test_seq2head_matches_head_split(orc, B, H, N, d, P, dtype):
    x = _coded((B, H, N, d), dtype)
    seq = orc.shard_seq(x, P)
    head = orc.seq2head(seq)
    # head-sharded rank r holds heads [r*H/P, (r+1)*H/P) with every token
    ref = x.reshape(B, P, H // P, N, d).transpose(1, 0, 2, 3, 4)
    assert head.shape == (P, B, H // P, N, d)
    assert np.array_equal(head, ref)
    if B == 1:
        # with one sequence the head-sharded buffers concatenated are the logical tensor
        assert head.tobytes() == x.tobytes()
    # the reverse all-to-all is the inverse permutation, both ways round
    assert np.array_equal(orc.head2seq(head), seq)
    y = _coded((P, B, H // P, N, d), dtype)[::-1].copy()
    assert np.array_equal(orc.seq2head(orc.head2seq(y)), y)


@pytest.mark.parametrize("B,H,N,d,P,Pu", [(2, 8, 24, 3, 4, 2), (1, 6, 36, 2, 6, 3), (1, 4, 16, 1, 4, 1),
                                          (2, 4, 16, 2, 4, 4)])
def test_group_seq2head_gives_the_2d_layout(orc, B, H, N, d, P, Pu):
    """2-D sequence parallelism: the all-to-all inside each ring group of Pu consecutive ranks
    (the oracle's Ulysses map on that group's shards) leaves rank g*Pu + u with heads
    u*H/Pu .. of token chunk g -- element by element."""
    from tests.helpers import from_hybrid, to_hybrid
    x = _coded((B, H, N, d), np.float32)
    seq = orc.shard_seq(x, P)
    Pr, Nc, Hl = P // Pu, N // (P // Pu), H // Pu
    hyb = np.concatenate([orc.seq2head(seq[g * Pu:(g + 1) * Pu]) for g in range(Pr)])
    assert hyb.shape == (P, B, Hl, Nc, d)
    for g in range(Pr):
        for u in range(Pu):
            for b in range(B):
                for hl in range(Hl):
                    assert np.array_equal(hyb[g * Pu + u, b, hl], x[b, u * Hl + hl, g * Nc:(g + 1) * Nc])
    assert np.array_equal(hyb, to_hybrid(x, P, Pu))
    assert np.array_equal(from_hybrid(hyb, Pu), x)


def test_seq2head_is_a_permutation(orc):
    B, H, N, d, P = 2, 8, 16, 3, 4
    x = _coded((P, B, N // P, H, d))
    y = orc.seq2head(x)
    assert np.array_equal(np.sort(y.ravel()), np.sort(x.ravel()))
    assert np.unique(y).size == y.size


def test_layout_rejects_bad_sizes(orc):
    with pytest.raises(ValueError):
        orc.seq2head(np.zeros((3, 1, 2, 4, 1), np.float32))  # H=4 not divisible by P=3


# ---------------------------------------------------------------- attention
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("B,Hq,Hkv,N,d", [(1, 2, 2, 9, 4), (2, 4, 2, 16, 8), (1, 6, 2, 13, 5), (1, 1, 1, 1, 3)])
def test_attention_brute_force(orc, causal, B, Hq, Hkv, N, d):
    q = _rand((B, Hq, N, d), 0)
    k = _rand((B, Hkv, N, d), 1)
    v = _rand((B, Hkv, N, d), 2)
    scale = 1.0 / np.sqrt(d)
    o, lse = orc.attn_rows(q, k, v, causal=causal)
    ob, lseb = _brute(*(t.astype(np.float64) for t in (q, k, v)), causal, scale)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lseb, rtol=0, atol=1e-12)
    # a subset of rows, in any order, gives the same rows
    rows = np.array([N - 1, 0, N // 2], dtype=np.int64)
    o2, l2 = orc.attn_rows(q, k, v, rows=rows, causal=causal)
    assert np.array_equal(o2, o[:, :, rows]) and np.array_equal(l2, lse[:, :, rows])


def test_attention_bf16_inputs_are_exact_values(orc):
    qb, kb, vb = (_rand((1, 2, 11, 8), s, "bf16") for s in (0, 1, 2))
    o, lse = orc.attn_rows(qb, kb, vb)
    q, k, v = (synth.bf16_to_f32(t) for t in (qb, kb, vb))
    o2, lse2 = orc.attn_rows(q, k, v)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def test_softmax_rows_sum_to_one_and_mask_future(orc):
    N = 16
    q = _rand((1, 1, N, N), 0)
    k = _rand((1, 1, N, N), 1)
    v = np.eye(N, dtype=np.float32)[None, None]
    p, _ = orc.attn_rows(q, k, v, causal=True)  # with V = I the output rows are softmax rows
    p = p[0, 0]
    assert np.all(np.abs(p.sum(axis=1) - 1.0) < 1e-12)
    assert np.all(p[np.triu_indices(N, 1)] == 0.0)
    assert np.all(p[np.tril_indices(N)] > 0.0)


def test_causal_future_values_do_not_matter(orc):
    B, H, N, d = 1, 2, 12, 4
    q, k, v = _rand((B, H, N, d), 0), _rand((B, H, N, d), 1), _rand((B, H, N, d), 2)
    o, lse = orc.attn_rows(q, k, v, causal=True)
    for i in (0, 5, 10):
        v2, k2 = v.copy(), k.copy()
        v2[:, :, i + 1:] += 100.0
        k2[:, :, i + 1:] -= 3.0
        o2, l2 = orc.attn_rows(q, k2, v2, rows=[i], causal=True)
        assert np.array_equal(o2[:, :, 0], o[:, :, i]) and np.array_equal(l2[:, :, 0], lse[:, :, i])


def test_constant_values_give_constant_output(orc):
    B, Hq, Hkv, N, d = 1, 4, 2, 20, 6
    q, k = _rand((B, Hq, N, d), 0), _rand((B, Hkv, N, d), 1)
    v = np.full((B, Hkv, N, d), 0.75, dtype=np.float32)
    for causal in (True, False):
        o, _ = orc.attn_rows(q, k, v, causal=causal)
        np.testing.assert_allclose(o, 0.75, rtol=0, atol=1e-14)


def test_zero_keys_closed_form(orc):
    # K = 0: every score is 0, so O_i is the mean of the visible V_j and LSE_i = ln(#visible)
    B, Hq, Hkv, N, d = 2, 4, 2, 17, 5
    q, v = _rand((B, Hq, N, d), 0), _rand((B, Hkv, N, d), 2)
    k = np.zeros((B, Hkv, N, d), np.float32)
    o, lse = orc.attn_rows(q, k, v, causal=True)
    vf = np.repeat(v.astype(np.float64), Hq // Hkv, axis=1)
    mean = np.cumsum(vf, axis=2) / np.arange(1, N + 1)[None, None, :, None]
    np.testing.assert_allclose(o, mean, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, np.log(np.arange(1, N + 1))[None, None, :].repeat(Hq, 1).repeat(B, 0),
                               rtol=0, atol=1e-14)
    o, lse = orc.attn_rows(q, k, v, causal=False)
    np.testing.assert_allclose(o, vf.mean(axis=2, keepdims=True).repeat(N, axis=2), rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, np.log(N), rtol=0, atol=1e-14)


def test_default_scale_is_inverse_sqrt_d(orc):
    q, k, v = (_rand((1, 1, 8, 64), s) for s in (0, 1, 2))
    o1, l1 = orc.attn_rows(q, k, v)
    o2, l2 = orc.attn_rows(q, k, v, scale=0.125)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    o3, _ = orc.attn_rows(q, k, v, scale=0.5)
    assert not np.allclose(o1, o3)


def test_library_special_case_tiny_exactness_size(orc):
    # shape of the tiny exactness case: B=1, H=4, N=256, d=64, fp32, causal
    q, k, v = (_rand((1, 4, 256, 64), s, seed=0) for s in (0, 1, 2))
    o, lse = orc.attn_rows(q, k, v, causal=True)
    ob, lseb = _brute(*(t.astype(np.float64) for t in (q, k, v)), True, 0.125)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lseb, rtol=0, atol=1e-12)


@pytest.mark.parametrize("P", [2, 4])
def test_partial_attention_merge_equals_full_sequence(orc, P):
    # ring attention: partials over KV blocks merged by LSE equal full attention
    B, Hq, Hkv, N, d = 1, 4, 2, 24, 8
    q, k, v = _rand((B, Hq, N, d), 0), _rand((B, Hkv, N, d), 1), _rand((B, Hkv, N, d), 2)
    o_full, lse_full = orc.attn_rows(q, k, v, causal=True)
    blk = N // P
    o_acc = np.zeros_like(o_full)
    lse_acc = np.full_like(lse_full, -np.inf)
    for j in range(P):
        o_j, lse_j = orc.attn_rows(q, k, v, causal=True, key_lo=j * blk, key_hi=(j + 1) * blk)
        # rows before the block see none of it
        assert np.all(lse_j[:, :, : j * blk] == -np.inf) and np.all(o_j[:, :, : j * blk] == 0)
        o_acc, lse_acc = orc.lse_merge(o_acc, lse_acc, o_j, lse_j)
    np.testing.assert_allclose(o_acc, o_full, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse_acc, lse_full, rtol=0, atol=1e-13)


def test_lse_merge_identities(orc):
    rng = np.random.default_rng(3)
    o_a, o_b = rng.standard_normal((2, 10, 4))
    l_a, l_b = rng.standard_normal((2, 10)) * 3
    o, l = orc.lse_merge(o_a, l_a, o_b, l_b)
    o2, l2 = orc.lse_merge(o_b, l_b, o_a, l_a)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-15)
    np.testing.assert_allclose(l, l2, rtol=0, atol=1e-15)
    np.testing.assert_allclose(l, np.logaddexp(l_a, l_b), rtol=0, atol=1e-14)
    # merging a partial with itself keeps O and adds ln 2
    o3, l3 = orc.lse_merge(o_a, l_a, o_a, l_a)
    np.testing.assert_allclose(o3, o_a, rtol=0, atol=1e-15)
    np.testing.assert_allclose(l3, l_a + np.log(2.0), rtol=0, atol=1e-14)
    # an empty partial (-inf) is the identity
    o4, l4 = orc.lse_merge(o_a, l_a, np.zeros_like(o_b), np.full_like(l_b, -np.inf))
    assert np.array_equal(o4, o_a) and np.array_equal(l4, l_a)
    o5, l5 = orc.lse_merge(np.zeros_like(o_b), np.full_like(l_b, -np.inf), np.zeros_like(o_b),
                           np.full_like(l_b, -np.inf))
    assert np.all(l5 == -np.inf) and np.all(o5 == 0)


# ---------------------------------------------------------------- backward
def _grid(shape, stream, seed=11):
    """Values on a 2^-8 grid in [-2, 2): exact in float32 and after +-2^-12 steps."""
    x = synth.normal(shape, seed=seed, stream=stream)
    return np.clip(np.round(x * 256.0) / 256.0, -2.0, 2.0 - 2 ** -8).astype(np.float32)


def _fd_grad(f, x, h):
    """Richardson-extrapolated central differences of scalar f at float32 x."""
    g = np.zeros(x.shape, dtype=np.float64)
    for idx in np.ndindex(x.shape):
        def cd(hh):
            xp, xm = x.copy(), x.copy()
            xp[idx] += hh
            xm[idx] -= hh
            return (f(xp) - f(xm)) / (2 * hh)
        g[idx] = (4 * cd(h / 2) - cd(h)) / 3
    return g


@pytest.mark.parametrize("causal", [True, False])
def test_backward_finite_differences(orc, causal):
    B, Hq, Hkv, N, d = 1, 4, 2, 7, 3
    q, k, v = _grid((B, Hq, N, d), 0), _grid((B, Hkv, N, d), 1), _grid((B, Hkv, N, d), 2)
    G = _grid((B, Hq, N, d), 3)  # upstream gradient: loss = sum(O * G)
    h = 2.0 ** -11

    def loss(qq, kk, vv):
        o, _ = orc.attn_rows(qq, kk, vv, causal=causal)
        return float(np.sum(o * G.astype(np.float64)))

    dq, dk, dv, _, _ = orc.attn_bwd_full(q, k, v, G, causal=causal)
    fq = _fd_grad(lambda x: loss(x, k, v), q, h)
    fk = _fd_grad(lambda x: loss(q, x, v), k, h)
    fv = _fd_grad(lambda x: loss(q, k, x), v, h)
    for a, b in ((dq, fq), (dk, fk), (dv, fv)):
        rel = np.abs(a - b).max() / np.abs(b).max()
        assert rel < 1e-6, rel


def test_backward_of_mean_square_loss(orc):
    # loss of the glossary page's example: mean(out.float()^2); dO = 2 O / numel
    B, Hq, Hkv, N, d = 1, 2, 2, 6, 4
    q, k, v = _grid((B, Hq, N, d), 0), _grid((B, Hkv, N, d), 1), _grid((B, Hkv, N, d), 2)
    o, _ = orc.attn_rows(q, k, v, causal=True)
    dO = (2.0 * o / o.size).astype(np.float32)

    def loss(qq, kk, vv):
        oo, _ = orc.attn_rows(qq, kk, vv, causal=True)
        return float(np.mean(oo * oo))

    dq, dk, dv, _, _ = orc.attn_bwd_full(q, k, v, dO, causal=True)
    h = 2.0 ** -11
    for a, b in ((dq, _fd_grad(lambda x: loss(x, k, v), q, h)),
                 (dk, _fd_grad(lambda x: loss(q, x, v), k, h)),
                 (dv, _fd_grad(lambda x: loss(q, k, x), v, h))):
        rel = np.abs(a - b).max() / np.abs(b).max()
        assert rel < 1e-5, rel  # dO rounded to float32


@pytest.mark.parametrize("causal", [True, False])
def test_gradient_sum_identities(orc, causal):
    # softmax is shift invariant: sum_j dK_j = 0; rows of P sum to 1: sum_j dV_j = sum_{group,i} dO_i
    B, Hq, Hkv, N, d = 2, 4, 2, 19, 6
    q, k, v, dO = (_rand(s_, st) for s_, st in (((B, Hq, N, d), 0), ((B, Hkv, N, d), 1),
                                                 ((B, Hkv, N, d), 2), ((B, Hq, N, d), 3)))
    dq, dk, dv, _, _ = orc.attn_bwd_full(q, k, v, dO, causal=causal)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, rtol=0, atol=1e-12)
    g = Hq // Hkv
    want = dO.astype(np.float64).reshape(B, Hkv, g, N, d).sum(axis=(2, 3))
    np.testing.assert_allclose(dv.sum(axis=2), want, rtol=0, atol=1e-11)


def test_backward_row_subsets(orc):
    B, Hq, Hkv, N, d = 1, 4, 1, 21, 5
    q, k, v, dO = (_rand(s_, st, "bf16") for s_, st in (((B, Hq, N, d), 0), ((B, Hkv, N, d), 1),
                                                         ((B, Hkv, N, d), 2), ((B, Hq, N, d), 3)))
    dq, dk, dv, o, lse = orc.attn_bwd_full(q, k, v, dO)
    rows = np.array([20, 3, 0, 11], dtype=np.int64)
    dq2 = orc.attn_bwd_q_rows(q, k, v, dO, rows=rows)
    assert np.array_equal(dq2, dq[:, :, rows])
    dvec = np.einsum("bhnd,bhnd->bhn", orc.as_f64(dO), o)
    # rows below the smallest selected key are never read: poison them
    lse_p, dvec_p = lse.copy(), dvec.copy()
    lse_p[:, :, :3] = np.nan
    dvec_p[:, :, :3] = np.nan
    dk2, dv2 = orc.attn_bwd_kv_rows(q, k, v, dO, lse_p, dvec_p, rows=np.array([3, 20, 11]))
    assert np.array_equal(dk2, dk[:, :, [3, 20, 11]]) and np.array_equal(dv2, dv[:, :, [3, 20, 11]])


# ------------------------------------------------ BLAS-backed row oracle (large sampled checks)
@pytest.mark.parametrize("causal", [True, False])
def test_blas_rows_match_c_oracle(orc, causal):
    from oracle import rows_blas
    B, Hq, Hkv, N, d = 2, 4, 2, 150, 16
    q, k, v, dO = (_rand(s_, st, "bf16") for s_, st in (((B, Hq, N, d), 0), ((B, Hkv, N, d), 1),
                                                         ((B, Hkv, N, d), 2), ((B, Hq, N, d), 3)))
    rows = np.array([0, 1, 63, 64, 65, 100, 149], dtype=np.int64)
    o, lse = orc.attn_rows(q, k, v, rows=rows, causal=causal)
    o2, lse2 = rows_blas.attn_rows(q, k, v, rows, causal=causal)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-12)
    dq = orc.attn_bwd_q_rows(q, k, v, dO, rows=rows, causal=causal)
    np.testing.assert_allclose(rows_blas.attn_bwd_q_rows(q, k, v, dO, rows, causal=causal), dq, rtol=0, atol=1e-11)
    _, _, _, oa, lsea = orc.attn_bwd_full(q, k, v, dO, causal=causal)
    dvec = np.einsum("bhnd,bhnd->bhn", orc.as_f64(dO), oa)
    dk, dv = orc.attn_bwd_kv_rows(q, k, v, dO, lsea, dvec, rows=rows, causal=causal)
    dk2, dv2 = rows_blas.attn_bwd_kv_rows(q, k, v, dO, lsea, dvec, rows, causal=causal)
    np.testing.assert_allclose(dk2, dk, rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv2, dv, rtol=0, atol=1e-11)


def test_blas_rows_closed_forms():
    from oracle import rows_blas
    B, Hq, Hkv, N, d = 1, 4, 2, 40, 8
    q, v = _rand((B, Hq, N, d), 0), _rand((B, Hkv, N, d), 2)
    k = np.zeros((B, Hkv, N, d), np.float32)
    rows = np.arange(N)
    o, lse = rows_blas.attn_rows(q, k, v, rows, causal=True)
    vf = np.repeat(v.astype(np.float64), 2, axis=1)
    np.testing.assert_allclose(o, np.cumsum(vf, axis=2) / np.arange(1, N + 1)[None, None, :, None], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], np.log(np.arange(1, N + 1)), rtol=0, atol=1e-14)
    vc = np.full_like(v, -1.25)
    o, _ = rows_blas.attn_rows(q, _rand((B, Hkv, N, d), 1), vc, rows, causal=False)
    np.testing.assert_allclose(o, -1.25, rtol=0, atol=1e-14)


@pytest.mark.parametrize("causal", [True, False])
def test_blas_full_rows_lse_dvec_and_chunked_kv_match_c_oracle(orc, causal):
    """Every row's LSE and D_i = dO_i . O_i (chunks of 64 rows, the element-wise steps split over
    threads) and dK/dV with query chunks of 37 rows, on a subset of KV heads, equal the C oracle."""
    from oracle import rows_blas
    B, Hq, Hkv, N, d = 2, 4, 2, 150, 16
    q, k, v, dO = (_rand(s_, st, "bf16") for s_, st in (((B, Hq, N, d), 0), ((B, Hkv, N, d), 1),
                                                         ((B, Hkv, N, d), 2), ((B, Hq, N, d), 3)))
    dq, dk, dv, o, lse = orc.attn_bwd_full(q, k, v, dO, causal=causal)
    dvec = np.einsum("bhnd,bhnd->bhn", orc.as_f64(dO), o)
    lse2, dvec2 = rows_blas.attn_lse_dvec(q, k, v, dO, causal=causal, chunk=64)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dvec2, dvec, rtol=0, atol=1e-12)
    # one KV head of one batch, rows from 70 on: the group's two query heads there, NaN elsewhere
    lse3, dvec3 = rows_blas.attn_lse_dvec(q, k, v, dO, causal=causal, kv_heads=[(1, 0)], row_lo=70, chunk=64)
    np.testing.assert_allclose(lse3[1, 0:2, 70:], lse[1, 0:2, 70:], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dvec3[1, 0:2, 70:], dvec[1, 0:2, 70:], rtol=0, atol=1e-12)
    assert np.isnan(lse3[1, 0:2, :70]).all() and np.isnan(lse3[0]).all() and np.isnan(lse3[1, 2:]).all()
    rows = np.array([0, 1, 36, 37, 74, 100, 149], dtype=np.int64)
    dk2, dv2 = rows_blas.attn_bwd_kv_rows(q, k, v, dO, lse2, dvec2, rows, causal=causal, chunk=37)
    np.testing.assert_allclose(dk2, dk[:, :, rows], rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv2, dv[:, :, rows], rtol=0, atol=1e-11)
    dk3, dv3 = rows_blas.attn_bwd_kv_rows(q, k, v, dO, lse2, dvec2, rows, causal=causal, chunk=37,
                                          kv_heads=[(0, 1)])
    np.testing.assert_allclose(dk3[0, 1], dk[0, 1][rows], rtol=0, atol=1e-11)
    assert not dk3[0, 0].any() and not dv3[1].any()


def test_blas_full_rows_closed_form():
    """K = 0: every visible score is 0, so LSE_i = ln(i + 1) and O_i is the mean of V_0..V_i,
    whence D_i = dO_i . mean_{j <= i} V_j."""
    from oracle import rows_blas
    B, Hq, Hkv, N, d = 1, 4, 2, 300, 8
    q, v, dO = _rand((B, Hq, N, d), 0), _rand((B, Hkv, N, d), 2), _rand((B, Hq, N, d), 3)
    k = np.zeros((B, Hkv, N, d), np.float32)
    lse, dvec = rows_blas.attn_lse_dvec(q, k, v, dO, causal=True, chunk=128)
    np.testing.assert_allclose(lse, np.broadcast_to(np.log(np.arange(1, N + 1)), lse.shape), rtol=0, atol=1e-13)
    mean_v = np.repeat(np.cumsum(v.astype(np.float64), axis=2) / np.arange(1, N + 1)[None, None, :, None], 2, axis=1)
    np.testing.assert_allclose(dvec, np.einsum("bhnd,bhnd->bhn", dO.astype(np.float64), mean_v), rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [True, False])
def test_blas_rows_many_rows_match_c_oracle(orc, causal):
    """Every row of 300 (three chunks, each split over several threads' row slices) equals the C
    oracle: forward O, LSE and dQ."""
    from oracle import rows_blas
    B, Hq, Hkv, N, d = 1, 2, 1, 300, 16
    q, k, v, dO = (_rand(s_, st, "bf16") for s_, st in (((B, Hq, N, d), 0), ((B, Hkv, N, d), 1),
                                                         ((B, Hkv, N, d), 2), ((B, Hq, N, d), 3)))
    rows = np.arange(N, dtype=np.int64)
    o, lse = orc.attn_rows(q, k, v, rows=rows, causal=causal)
    o2, lse2 = rows_blas.attn_rows(q, k, v, rows, causal=causal)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-12)
    dq = orc.attn_bwd_q_rows(q, k, v, dO, rows=rows, causal=causal)
    np.testing.assert_allclose(rows_blas.attn_bwd_q_rows(q, k, v, dO, rows, causal=causal), dq, rtol=0, atol=1e-11)

"""The benchmark's work accounting (CPU only): the algorithmic FLOPs and bytes
that every reported rate and roofline fraction divides by.

Closed forms: causal attention over N tokens has N(N+1)/2 visible
(query, key) pairs per head; the forward costs 4*d FLOPs per pair (Q K^T and
P V) and the backward 10*d (dV, dP, dK, dQ), so one training step is 3.5x the
forward. The Ulysses remaps move every byte of Q, K, V, dO in and O, dQ, dK,
dV out, each read once and written once."""
import bench


def _w(B=1, Hq=32, Hkv=8, N=131072, d=128, P=8):
    return dict(B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, P=P)


def test_causal_pair_count_by_enumeration():
    for N in (1, 2, 3, 7, 64, 129):
        assert bench.causal_pairs(N) == sum(1 for i in range(N) for j in range(N) if j <= i)


def test_forward_flops_of_the_workloads():
    # 4 * B * Hq * d * N(N+1)/2, written out per workload
    cases = [
        (_w(B=1, Hq=4, Hkv=4, N=4096, d=64, P=2), 8.59e9),     # the glossary page's 4096-token example
        (_w(Hq=32, Hkv=8, N=32768, d=128, P=4), 8.80e12),      # 32K tokens on four ranks
        (_w(), 140.7e12),                                      # the 128K-token step
        (_w(Hq=32, Hkv=32, N=524288, d=128, P=8), 2252e12),    # the 512K ring workload
    ]
    for w, want in cases:
        got = bench.fwd_flops(w)
        assert got == 4 * w["B"] * w["Hq"] * w["d"] * w["N"] * (w["N"] + 1) // 2
        assert abs(got - want) / want < 5e-3, (w, got)


def test_step_and_kernel_work_at_128k():
    w = _w()
    f = bench.fwd_flops(w)
    assert abs(3.5 * f - 492.6e12) / 492.6e12 < 1e-3          # forward 4d + backward 10d per pair
    bound, fw = bench.kernel_work("attn_fwd", w, 1)
    assert (bound, fw) == ("tensor", f)
    _, dkdv = bench.kernel_work("attn_bwd_dkdv", w, 1)
    _, dq = bench.kernel_work("attn_bwd_dq", w, 1)
    assert dkdv == 2 * f                                       # S^T, dP^T, dV, dK: 8d per pair
    assert dq == 1.5 * f                                       # S, dP (recomputed), dQ: 6d per pair
    # together: the algorithmic backward (10d per pair: S, dV, dP, dK, dQ) plus the dQ pass's
    # recomputed S and dP (4d per pair, one forward's worth)
    assert dkdv + dq == 2.5 * f + f


def test_remap_bytes_per_step_at_128k():
    w = _w()
    q_bytes = 1 * 32 * 131072 * 128 * 2
    kv_bytes = 1 * 8 * 131072 * 128 * 2
    per_launch = {n: bench.kernel_work(n, w, 4)[1] for n in ("a2a_seq2head", "a2a_head2seq")}
    # four launches of each direction per step; each byte read once and written once
    total = 4 * (per_launch["a2a_seq2head"] + per_launch["a2a_head2seq"])
    assert total == 2 * (4 * q_bytes + 4 * kv_bytes) == 10 * 2**30
    assert bench.kernel_work("a2a_seq2head", w, 4)[0] == "hbm"


def test_traffic_is_only_reported_for_its_workload():
    assert bench.measured_traffic("attn_fwd", _w(N=32768, P=4)) is None
    assert bench.measured_traffic("attn_fwd", _w(d=64)) is None
    assert bench.measured_traffic("no_such_kernel", _w()) is None

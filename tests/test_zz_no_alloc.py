"""The backward entry point for callers that cannot allocate device memory.

usp_attn_bwd_noalloc serves code that is not allowed to call cudaMalloc (for
example inside a framework that owns all device memory): it runs the same
backward as usp_attn_bwd but keeps its workspace in a fixed array built into
the library.  These tests call it through the C ABI and compare it with the
workspace-taking entry point on the same inputs, on two calls in a row (the
second call finds the first call's data in the shared array).  This file is
collected last on purpose.
"""
import pytest

from tests.helpers import TOL_BF16_GRAD_RELFRO, f64, gen, rel_fro, to_dev, to_head, to_host


@pytest.fixture(scope="module")
def usp():
    import context_long_attention_ulysses_gb300 as m
    from context_long_attention_ulysses_gb300 import build
    build.build()
    return m


def test_rejects_problems_larger_than_the_scratch(usp):
    # needs 40 bytes * 32 heads * 524288 rows = 640 MiB > the built-in 64 MiB; refused before any CUDA call
    p = usp.Problem(B=1, Hq=32, Hkv=8, N=524288, d=128, P=8)
    assert usp.usp_attn_bwd_workspace_size(p) > usp.NOALLOC_SCRATCH_BYTES
    fake = 1 << 20
    with pytest.raises(usp.UspError) as e:
        usp.usp_attn_bwd_noalloc(p, *([fake] * 9))
    assert e.value.status == 4  # USP_ERR_WORKSPACE


@pytest.mark.gpu
def test_noalloc_backward_matches_workspace_backward(usp):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B, Hq, Hkv, N, d, P = 1, 8, 2, 1000, 128, 2
    p = usp.Problem(B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, P=P)
    q, k, v, dO = gen((B, Hq, N, d), 0), gen((B, Hkv, N, d), 1), gen((B, Hkv, N, d), 2), gen((B, Hq, N, d), 3)
    qh, kh, vh, doh = (to_dev(to_head(x, P)) for x in (q, k, v, dO))
    oh = torch.empty_like(qh)
    lse = torch.empty(p.lse_head_shape(), dtype=torch.float32, device="cuda")
    usp.usp_attn_fwd(p, qh, kh, vh, oh, lse)

    # reference: the entry point that takes a caller-allocated workspace
    ws = torch.empty(usp.usp_attn_bwd_workspace_size(p), dtype=torch.uint8, device="cuda")
    ref = [torch.empty_like(qh), torch.empty_like(kh), torch.empty_like(vh)]
    usp.usp_attn_bwd(p, qh, kh, vh, oh, lse, doh, *ref, ws)
    torch.cuda.synchronize()
    ref_h = [f64(to_host(t)) for t in ref]

    for call in range(2):
        out = [torch.full_like(t, float("nan")) for t in ref]
        usp.usp_attn_bwd_noalloc(p, qh, kh, vh, oh, lse, doh, *out)
        torch.cuda.synchronize()
        assert usp.usp_device_status() == 0
        for name, got, want in zip(("dq", "dk", "dv"), out, ref_h):
            err = rel_fro(f64(to_host(got)), want)
            assert err < TOL_BF16_GRAD_RELFRO, (call, name, err)

"""The backward entry point for callers that cannot allocate device memory.

usp_attn_bwd_noalloc serves code that is not allowed to call cudaMalloc (for
example inside a framework that owns all device memory): it runs the same
deterministic backward as usp_attn_bwd_deterministic but keeps its workspace
in a fixed array built into the library.  These tests call it through the C
ABI and compare it with the workspace-taking entry point on the same inputs,
bit for bit, on two calls in a row, after a call on a larger, different
problem has left its own rows (padding rows included) in the shared array.
This file is collected last on purpose.
"""
import pytest

from tests.helpers import gen, to_dev, to_head, to_host


@pytest.fixture(scope="module")
def usp():
    import context_long_attention_ulysses_gb300 as m
    from context_long_attention_ulysses_gb300 import build
    build.build()
    return m


def test_rejects_problems_larger_than_the_scratch(usp):
    # needs 40 bytes * 32 heads * 524288 rows = 640 MiB > the built-in 64 MiB; refused before any CUDA call
    p = usp.Problem(B=1, Hq=32, Hkv=8, N=524288, d=128, P=8)
    assert usp.usp_attn_bwd_deterministic_workspace_size(p) > usp.NOALLOC_SCRATCH_BYTES
    fake = 1 << 20
    with pytest.raises(usp.UspError) as e:
        usp.usp_attn_bwd_noalloc(p, *([fake] * 9))
    assert e.value.status == 4  # USP_ERR_WORKSPACE


@pytest.mark.parametrize("d,dtype,status", [(96, "bf16", 2), (128, "f32", 2)])
def test_unsupported_problems_are_refused_before_any_cuda_call(usp, d, dtype, status):
    # a head dimension or dtype the backward does not implement: USP_ERR_UNSUPPORTED, as from
    # usp_attn_bwd, with no scratch lookup (fake pointers; runs without a GPU)
    p = usp.Problem(B=1, Hq=4, Hkv=4, N=256, d=d, P=2, dtype=dtype)
    fake = 1 << 20
    with pytest.raises(usp.UspError) as e:
        usp.usp_attn_bwd_noalloc(p, *([fake] * 9))
    assert e.value.status == status


def test_misaligned_pointers_are_refused_before_any_cuda_call(usp):
    p = usp.Problem(B=1, Hq=4, Hkv=4, N=256, d=128, P=2)
    ptrs = [1 << 20] * 9
    ptrs[3] += 8  # o not 16-byte aligned
    with pytest.raises(usp.UspError) as e:
        usp.usp_attn_bwd_noalloc(p, *ptrs)
    assert e.value.status == 3  # USP_ERR_MISALIGNED


def _problem_inputs(usp, B, Hq, Hkv, N, d, P, seed):
    import torch
    p = usp.Problem(B=B, Hq=Hq, Hkv=Hkv, N=N, d=d, P=P)
    q, k, v, dO = (gen(s, st, seed=seed) for s, st in (((B, Hq, N, d), 0), ((B, Hkv, N, d), 1),
                                                           ((B, Hkv, N, d), 2), ((B, Hq, N, d), 3)))
    qh, kh, vh, doh = (to_dev(to_head(x, P)) for x in (q, k, v, dO))
    oh = torch.empty_like(qh)
    lse = torch.empty(p.lse_head_shape(), dtype=torch.float32, device="cuda")
    usp.usp_attn_fwd(p, qh, kh, vh, oh, lse)
    return p, (qh, kh, vh, oh, lse, doh)


@pytest.mark.gpu
def test_noalloc_backward_matches_workspace_backward(usp):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    # a larger, different problem first, so the shared array holds rows (and padding rows) that do
    # not belong to the checked problem when it runs
    p_big, big = _problem_inputs(usp, 1, 16, 4, 3000, 128, 4, seed=7)
    out_big = [torch.empty_like(big[0]), torch.empty_like(big[1]), torch.empty_like(big[2])]
    usp.usp_attn_bwd_noalloc(p_big, *big, *out_big)
    torch.cuda.synchronize()
    assert usp.usp_device_status() == 0

    p, ins = _problem_inputs(usp, 1, 8, 2, 1000, 128, 2, seed=0)
    qh, kh, vh = ins[:3]
    # reference: the entry point that takes a caller-allocated workspace
    ws = torch.empty(usp.usp_attn_bwd_deterministic_workspace_size(p), dtype=torch.uint8, device="cuda")
    ref = [torch.empty_like(qh), torch.empty_like(kh), torch.empty_like(vh)]
    usp.usp_attn_bwd_deterministic(p, *ins, *ref, ws)
    torch.cuda.synchronize()
    want = [to_host(t).tobytes() for t in ref]

    for call in range(2):
        out = [torch.full_like(t, float("nan")) for t in ref]
        usp.usp_attn_bwd_noalloc(p, *ins, *out)
        torch.cuda.synchronize()
        assert usp.usp_device_status() == 0
        for name, got, w in zip(("dq", "dk", "dv"), out, want):
            assert to_host(got).tobytes() == w, (call, name)

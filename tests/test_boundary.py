"""C-ABI boundary checks that need no GPU: the library loads, exports every
symbol include/usp.h declares, and rejects bad arguments on the host before
any CUDA call (no compute call is made here)."""
import ctypes
import os
import re

import pytest

import context_long_attention_ulysses_gb300 as usp
from context_long_attention_ulysses_gb300 import _lib, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "usp.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(usp_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_symbols():
    assert _declared() == sorted(_lib.SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    assert usp.usp_status_string(0) == "USP_OK"
    assert usp.usp_status_string(6) == "USP_ERR_TIMEOUT"
    assert usp.usp_status_string(99) == "USP_ERR_UNKNOWN"
    assert "sm_103a" in usp.usp_build_info()


def _p(**kw):
    base = dict(B=1, Hq=4, Hkv=4, N=256, d=64, P=2, causal=True, scale=0.0, dtype="bf16")
    base.update(kw)
    return usp.Problem(**base)


FAKE = 1 << 20  # 16-byte aligned fake device address; never dereferenced here


@pytest.mark.parametrize("kw,code", [
    (dict(N=255), _lib.USP_ERR_INVALID_ARG),          # N % P
    (dict(Hq=6, Hkv=4), _lib.USP_ERR_INVALID_ARG),    # Hq % Hkv
    (dict(Hq=3, Hkv=3), _lib.USP_ERR_INVALID_ARG),    # Hq % P
    (dict(Hq=4, Hkv=1), _lib.USP_ERR_INVALID_ARG),    # Hkv % P
    (dict(P=0), _lib.USP_ERR_INVALID_ARG),
    (dict(B=-1), _lib.USP_ERR_INVALID_ARG),
    (dict(scale=-1.0), _lib.USP_ERR_INVALID_ARG),
    (dict(d=96), _lib.USP_ERR_UNSUPPORTED),           # attention only for d in {64, 128}
])
def test_attention_argument_errors(lib, kw, code):
    with pytest.raises(usp.UspError) as e:
        usp.usp_attn_fwd(_p(**kw), FAKE, FAKE, FAKE, FAKE, FAKE)
    assert e.value.status == code


def test_null_problem_and_pointers(lib):
    assert lib.usp_attn_fwd(None, FAKE, FAKE, FAKE, FAKE, FAKE, None) == _lib.USP_ERR_INVALID_ARG
    with pytest.raises(usp.UspError) as e:
        usp.usp_attn_fwd(_p(), FAKE, 0, FAKE, FAKE, FAKE)
    assert e.value.status == _lib.USP_ERR_MISALIGNED
    with pytest.raises(usp.UspError) as e:
        usp.usp_a2a_seq2head(_p(), 4, FAKE + 8, FAKE * 2)
    assert e.value.status == _lib.USP_ERR_MISALIGNED


def test_remap_argument_errors(lib):
    with pytest.raises(usp.UspError) as e:
        usp.usp_a2a_seq2head(_p(), 3, FAKE, FAKE * 2)       # Hx is neither Hq nor Hkv
    assert e.value.status == _lib.USP_ERR_INVALID_ARG
    with pytest.raises(usp.UspError) as e:
        usp.usp_a2a_seq2head(_p(d=48), 4, FAKE, FAKE * 2)   # 96-byte rows
    assert e.value.status == _lib.USP_ERR_UNSUPPORTED
    with pytest.raises(usp.UspError) as e:
        usp.usp_a2a_head2seq(_p(), 4, FAKE, FAKE + 4096)    # overlapping buffers
    assert e.value.status == _lib.USP_ERR_INVALID_ARG


def test_backward_and_ring_argument_errors(lib):
    p = _p()
    ws = usp.usp_attn_bwd_workspace_size(p)
    with pytest.raises(usp.UspError) as e:
        usp.usp_attn_bwd(p, *([FAKE] * 9), FAKE, ws - 256)
    assert e.value.status == _lib.USP_ERR_WORKSPACE
    with pytest.raises(usp.UspError) as e:
        usp.usp_attn_bwd(p, *([FAKE] * 9), FAKE + 16, ws)   # workspace must be 256-byte aligned
    assert e.value.status == _lib.USP_ERR_MISALIGNED
    with pytest.raises(usp.UspError) as e:
        usp.usp_attn_bwd(_p(dtype="f32"), *([FAKE] * 9), FAKE, ws)
    assert e.value.status == _lib.USP_ERR_UNSUPPORTED
    rws = usp.usp_ring_workspace_size(p)
    with pytest.raises(usp.UspError) as e:
        usp.usp_ring_attn_fwd(p, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, rws - 1)
    assert e.value.status == _lib.USP_ERR_WORKSPACE
    with pytest.raises(usp.UspError) as e:
        usp.usp_ring_merge(10, 6, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE)   # d % 4
    assert e.value.status == _lib.USP_ERR_INVALID_ARG
    bws = usp.usp_ring_bwd_workspace_size(p)
    with pytest.raises(usp.UspError) as e:
        usp.usp_ring_attn_bwd(p, *([FAKE] * 9), FAKE, bws - 256)
    assert e.value.status == _lib.USP_ERR_WORKSPACE
    with pytest.raises(usp.UspError) as e:
        usp.usp_ring_attn_bwd(p, *([FAKE] * 9), FAKE + 128, bws)   # workspace must be 256-byte aligned
    assert e.value.status == _lib.USP_ERR_MISALIGNED
    with pytest.raises(usp.UspError) as e:
        usp.usp_ring_attn_bwd(p, FAKE + 8, *([FAKE] * 8), FAKE, bws)   # q not 16-byte aligned
    assert e.value.status == _lib.USP_ERR_MISALIGNED
    with pytest.raises(usp.UspError) as e:
        usp.usp_ring_attn_bwd(_p(d=96), *([FAKE] * 9), FAKE, bws)
    assert e.value.status == _lib.USP_ERR_UNSUPPORTED
    with pytest.raises(usp.UspError) as e:
        usp.usp_ring_attn_bwd(_p(dtype="f32"), *([FAKE] * 9), FAKE, bws)
    assert e.value.status == _lib.USP_ERR_UNSUPPORTED


def test_empty_problems_enqueue_nothing(lib):
    # B == 0 or N == 0 is valid and returns before any CUDA call
    for kw in (dict(N=0), dict(B=0)):
        p = _p(**kw)
        usp.usp_a2a_seq2head(p, 4, 0, 0)
        usp.usp_attn_fwd(p, 0, 0, 0, 0, 0)
        usp.usp_attn_bwd(p, *([0] * 9), 0, 0)
        usp.usp_ring_attn_fwd(p, 0, 0, 0, 0, 0, 0, 0)
        usp.usp_ring_attn_bwd(p, *([0] * 9), 0, 0)
        usp.usp_allgather_attn_fwd(p, 0, 0, 0, 0, 0, 0, 0)
        usp.usp_allgather_attn_bwd(p, *([0] * 9), 0, 0)
        usp.usp_zigzag_attn_fwd(p, 0, 0, 0, 0, 0, 0, 0)
        usp.usp_zigzag_attn_bwd(p, *([0] * 9), 0, 0)
        usp.usp_zigzag_shard(p, 4, 0, 0)
        usp.usp_fused_attn_fwd(p, 0, 0, 0, 0, 0)
        usp.usp_fused_attn_bwd(p, *([0] * 9), 0, 0)
        usp.usp_hybrid_seq2head(p, 2, 4, 0, 0)
        usp.usp_hybrid_attn_fwd(p, 2, 0, 0, 0, 0, 0, 0, 0)
        usp.usp_hybrid_attn_bwd(p, 2, *([0] * 9), 0, 0)
    usp.usp_ring_merge(0, 64, 0, 0, 0, 0, 0, 0)


def test_workspaces_are_linear_in_sequence_length(lib):
    for N in (1024, 4096, 131072):
        a = usp.usp_attn_bwd_deterministic_workspace_size(_p(N=N, Hq=32, Hkv=8, d=128, P=8))
        b = usp.usp_attn_bwd_deterministic_workspace_size(_p(N=2 * N, Hq=32, Hkv=8, d=128, P=8))
        assert b == 2 * a
        assert a == 40 * 32 * N  # per query row: D_i, lse_i*log2(e) (float32) and two 16-byte bf16 split rows
        # the one-pass backward adds a float32 dQ accumulator row of d values per query row
        a1 = usp.usp_attn_bwd_workspace_size(_p(N=N, Hq=32, Hkv=8, d=128, P=8))
        assert a1 == (40 + 4 * 128) * 32 * N
        assert usp.usp_attn_bwd_workspace_size(_p(N=2 * N, Hq=32, Hkv=8, d=128, P=8)) == 2 * a1
        assert usp.usp_fused_attn_bwd_workspace_size(_p(N=N, Hq=32, Hkv=8, d=128, P=8)) == a1
        r1 = usp.usp_ring_workspace_size(_p(N=N, Hq=32, Hkv=32, d=128, P=8))
        r2 = usp.usp_ring_workspace_size(_p(N=2 * N, Hq=32, Hkv=32, d=128, P=8))
        assert r2 == 2 * r1
        b1 = usp.usp_ring_bwd_workspace_size(_p(N=N, Hq=32, Hkv=8, d=128, P=8))
        b2 = usp.usp_ring_bwd_workspace_size(_p(N=2 * N, Hq=32, Hkv=8, d=128, P=8))
        assert b2 == 2 * b1
        # 40 bytes per padded query row, float32 dQ (Hq) and dK, dV (Hkv) accumulators
        assert b1 == 40 * 32 * N + 4 * N * 128 * (32 + 2 * 8)
    assert usp.usp_attn_bwd_workspace_size(_p(N=255)) == 0  # invalid problem


def test_trace_report_without_launches(lib):
    usp.usp_trace_reset()
    usp.usp_trace_enable(True)
    assert usp.usp_trace_report() == {}
    usp.usp_trace_enable(False)
    usp.usp_trace_reset()


def test_allgather_argument_errors(lib):
    p = _p()
    ws = usp.usp_allgather_workspace_size(p)
    bws = usp.usp_allgather_bwd_workspace_size(p)
    assert ws == 2 * p.B * p.N * p.Hkv * p.d * 2   # gathered K and V, bf16
    assert bws > ws
    with pytest.raises(usp.UspError) as e:
        usp.usp_allgather_attn_fwd(p, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws - 256)
    assert e.value.status == _lib.USP_ERR_WORKSPACE
    with pytest.raises(usp.UspError) as e:
        usp.usp_allgather_attn_fwd(p, FAKE, FAKE + 4, FAKE, FAKE, FAKE, FAKE, ws)   # k not 16-byte aligned
    assert e.value.status == _lib.USP_ERR_MISALIGNED
    with pytest.raises(usp.UspError) as e:
        usp.usp_allgather_attn_bwd(p, *([FAKE] * 9), FAKE, bws - 256)
    assert e.value.status == _lib.USP_ERR_WORKSPACE
    with pytest.raises(usp.UspError) as e:
        usp.usp_allgather_attn_bwd(_p(dtype="f32"), *([FAKE] * 9), FAKE, bws)
    assert e.value.status == _lib.USP_ERR_UNSUPPORTED
    with pytest.raises(usp.UspError) as e:
        usp.usp_allgather_attn_fwd(_p(N=255), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws)   # N % P
    assert e.value.status == _lib.USP_ERR_INVALID_ARG


def test_zigzag_argument_errors(lib):
    p = _p()
    ws = usp.usp_zigzag_workspace_size(p)
    bws = usp.usp_zigzag_bwd_workspace_size(p)
    assert ws == usp.usp_ring_workspace_size(p) and bws > 0
    odd = _p(N=p.N + p.P)                       # N % P == 0 but N % (2P) != 0
    assert usp.usp_zigzag_workspace_size(odd) == 0
    with pytest.raises(usp.UspError) as e:
        usp.usp_zigzag_attn_fwd(odd, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40)
    assert e.value.status == _lib.USP_ERR_INVALID_ARG
    with pytest.raises(usp.UspError) as e:
        usp.usp_zigzag_shard(odd, 4, FAKE, FAKE * 2)
    assert e.value.status == _lib.USP_ERR_INVALID_ARG
    with pytest.raises(usp.UspError) as e:
        usp.usp_zigzag_shard(p, 4, FAKE, FAKE + 64)   # overlapping buffers
    assert e.value.status == _lib.USP_ERR_INVALID_ARG
    with pytest.raises(usp.UspError) as e:
        usp.usp_zigzag_attn_fwd(p, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws - 256)
    assert e.value.status == _lib.USP_ERR_WORKSPACE
    with pytest.raises(usp.UspError) as e:
        usp.usp_zigzag_attn_bwd(p, *([FAKE] * 9), FAKE + 64, bws)   # workspace must be 256-byte aligned
    assert e.value.status == _lib.USP_ERR_MISALIGNED


def test_fused_argument_errors(lib):
    p = _p()                                                   # N/P = 128: one tile per shard
    bws = usp.usp_fused_attn_bwd_workspace_size(p)
    assert bws == usp.usp_attn_bwd_workspace_size(p) == (40 + 4 * p.d) * p.B * p.Hq * p.N  # rows + dQ accumulator
    for kw, code in ((dict(N=200), _lib.USP_ERR_UNSUPPORTED),  # shards of 100 tokens: tiles would straddle
                     (dict(N=384), _lib.USP_ERR_UNSUPPORTED),  # shards of 192 tokens
                     (dict(Hq=3, Hkv=3), _lib.USP_ERR_INVALID_ARG),   # heads are split over the ranks
                     (dict(dtype="f32"), _lib.USP_ERR_UNSUPPORTED),
                     (dict(d=32), _lib.USP_ERR_UNSUPPORTED)):
        with pytest.raises(usp.UspError) as e:
            usp.usp_fused_attn_fwd(_p(**kw), FAKE, FAKE, FAKE, FAKE, FAKE)
        assert e.value.status == code, kw
        with pytest.raises(usp.UspError) as e:
            usp.usp_fused_attn_bwd(_p(**kw), *([FAKE] * 9), FAKE, 1 << 40)
        assert e.value.status == code, kw
    with pytest.raises(usp.UspError) as e:
        usp.usp_fused_attn_fwd(p, FAKE, FAKE, FAKE + 8, FAKE, FAKE)   # v not 16-byte aligned
    assert e.value.status == _lib.USP_ERR_MISALIGNED
    with pytest.raises(usp.UspError) as e:
        usp.usp_fused_attn_bwd(p, *([FAKE] * 9), FAKE, bws - 256)
    assert e.value.status == _lib.USP_ERR_WORKSPACE
    with pytest.raises(usp.UspError) as e:
        usp.usp_fused_attn_bwd(p, *([FAKE] * 9), FAKE + 16, bws)       # workspace must be 256-byte aligned
    assert e.value.status == _lib.USP_ERR_MISALIGNED


def test_hybrid_argument_errors(lib):
    p = _p(P=4, N=1024, Hq=8, Hkv=4, d=128)
    for Pu in (0, -2, 3, 8):                                   # Pu >= 1 dividing P
        assert usp.usp_hybrid_workspace_size(p, Pu) == 0
        assert usp.usp_hybrid_bwd_workspace_size(p, Pu) == 0
        with pytest.raises(usp.UspError) as e:
            usp.usp_hybrid_seq2head(p, Pu, 8, FAKE, FAKE * 64)
        assert e.value.status == _lib.USP_ERR_INVALID_ARG
        with pytest.raises(usp.UspError) as e:
            usp.usp_hybrid_attn_fwd(p, Pu, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40)
        assert e.value.status == _lib.USP_ERR_INVALID_ARG
    with pytest.raises(usp.UspError) as e:                     # Hkv % Pu
        usp.usp_hybrid_attn_fwd(_p(P=4, N=1024, Hq=8, Hkv=2, d=128), 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40)
    assert e.value.status == _lib.USP_ERR_INVALID_ARG
    # heads split over Pu only: Hq = 8 on P = 6 ranks is a valid 2 x 3 problem
    assert usp.usp_hybrid_workspace_size(_p(P=6, N=1536, Hq=8, Hkv=4, d=128), 2) > 0
    for Pu in (1, 2, 4):
        Pr, Nc = 4 // Pu, 1024 // (4 // Pu)
        ws = usp.usp_hybrid_workspace_size(p, Pu)
        assert ws == usp.usp_ring_workspace_size(p)            # float32 running and partial O, partial LSE
        bws = usp.usp_hybrid_bwd_workspace_size(p, Pu)
        # 40 bytes per padded query row of every (rank, local head), float32 dQ, dK, dV accumulators
        assert bws == 40 * 4 * (8 // Pu) * ((Nc + 127) // 128 * 128) + 4 * 1024 * 128 * (8 + 2 * 4)
        with pytest.raises(usp.UspError) as e:
            usp.usp_hybrid_attn_fwd(p, Pu, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws - 256)
        assert e.value.status == _lib.USP_ERR_WORKSPACE
        with pytest.raises(usp.UspError) as e:
            usp.usp_hybrid_attn_bwd(p, Pu, *([FAKE] * 9), FAKE, bws - 256)
        assert e.value.status == _lib.USP_ERR_WORKSPACE
    with pytest.raises(usp.UspError) as e:
        usp.usp_hybrid_seq2head(p, 2, 8, FAKE, FAKE + 256)       # overlapping buffers
    assert e.value.status == _lib.USP_ERR_INVALID_ARG
    with pytest.raises(usp.UspError) as e:
        usp.usp_hybrid_seq2head(_p(P=4, N=1024, Hq=8, Hkv=4, d=24), 2, 8, FAKE, FAKE * 64)   # 48-byte rows
    assert e.value.status == _lib.USP_ERR_UNSUPPORTED
    with pytest.raises(usp.UspError) as e:
        usp.usp_hybrid_attn_fwd(_p(P=4, N=1024, Hq=8, Hkv=4, d=128, dtype="f32"), 2, *([FAKE] * 6), 1 << 40)
    assert e.value.status == _lib.USP_ERR_UNSUPPORTED
    with pytest.raises(usp.UspError) as e:
        usp.usp_hybrid_attn_bwd(p, 2, *([FAKE] * 9), FAKE + 64, 1 << 40)   # workspace must be 256-byte aligned
    assert e.value.status == _lib.USP_ERR_MISALIGNED


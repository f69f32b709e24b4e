// Internal host-side interface between the C-ABI layer (api.cu) and the
// kernel translation units.  Every launcher enqueues on `stream`, returns the
// launch's cudaError_t and assumes its arguments were validated by api.cu.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/usp.h"

namespace usp {

// ---- all-to-all layout remap (remap.cu)
// One side is sequence-sharded [P][B][N/P][Hx][d], the other head-sharded
// [P][B][Hx/P][N][d].  dir 0: seq -> head; dir 1: head -> seq.
cudaError_t launch_remap(int dir, const void* src, void* dst, int B, int Hx, int N, int P, int row_bytes,
                         cudaStream_t stream);

// ---- float32 attention forward on CUDA cores (attn_f32.cu)
// q, o: [Zq][N][d]; k, v: [Zq/g][N][d]; lse: [Zq][N].  Query slot z uses KV slot z/g.
cudaError_t launch_attn_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse, int Zq,
                                int g, int N, int d, int causal, float scale, cudaStream_t stream);

// ---- bf16 tensor-core attention (attn_fwd.cu / attn_bwd.cu)
// Addressing of one operand family: element (x = column, head, token, outer)
// sits at x + head*s_head + token*s_tok + outer*s_outer (elements).
struct Tensor4 {
    void* ptr;
    int64_t s_head, s_tok, s_outer;  // strides in elements
    int n_head, n_tok, n_outer;      // extents
};

// Work decomposition shared by the Ulysses (head-sharded) and ring
// (sequence-sharded) forward.  A work item is (q tile, query head, o) with
// o in [0, n_outer): query rank i = ring_i0 + o/bsz, batch b = o%bsz, KV rank
// j = (i - ring_t) mod ring_p.  Outer index of q/o/lse: i*bsz + b; of k/v:
// j*bsz + b.  Token positions: q i*np + token, k/v j*np + token.
// Head-sharded layout: ring_i0 = ring_t = 0, ring_p = bsz = 1, np = 0, n_outer = 1.
// kv_gathered = 1 (all-gather-KV): k/v hold the whole sequence per batch, outer
// index b and token positions 0..kv_len-1, for every query rank.
// zigzag = 1 (zigzag ring): every rank's shard is two chunks of np tokens, rank i
// holding chunks i and 2P-1-i (outer index (i*bsz + b)*2 + half); o decodes to
// (i, b, query half), the launch's KV half is zz_kh, positions are chunk * np.
// split_np > 0 (Ulysses attention read and written in place in the sequence-
// sharded layout [P][B][split_np][H][d]): the launch decodes like the head-
// sharded path with one outer index per batch (ring_p = 1, bsz = n_outer = B)
// over global positions, and every token coordinate passes through split_pos
// (ptx.cuh): position pos of batch b is token pos % split_np of outer index
// (pos / split_np) * split_b + b.  split_np must be a multiple of 128, so that
// no 128-row tile straddles two shards.
struct FwdParams {
    Tensor4 q, k, v;
    int d;
    int g;            // query heads per KV head
    int n_heads;      // query heads per outer index
    int n_outer;      // outer indices processed by this launch
    int q_len, kv_len;
    int ring_i0, ring_t, ring_p, bsz, np;
    int kv_gathered;
    int zigzag, zz_kh;
    int split_np, split_b;
    int causal;
    float scale;
    // epilogue: o_bf16 (bf16, strides as q) or o_f32 (float32); one is null
    void* o_bf16;
    float* o_f32;
    int64_t o_s_head, o_s_tok, o_s_outer;   // elements
    float* lse;
    int64_t l_s_head, l_s_tok, l_s_outer;   // elements
    int* status;
};
cudaError_t launch_attn_fwd_bf16(const FwdParams& p, cudaStream_t stream);

// Backward.  Tensors are addressed as (d, head, token, outer) like the
// forward: the Ulysses path passes head-sharded buffers as B*Hq "heads" of N
// tokens with one outer index; ring mode passes sequence-sharded buffers
// ([P][B][N/P][H][d], outer = rank * B + b) and one launch per ring step, the
// launch's outer indices decoded as in FwdParams (query outer i*bsz + b, KV
// outer j*bsz + b with j = (i - ring_t) mod ring_p).
struct BwdParams {
    Tensor4 q, k, v, o, dout;  // o and dout shaped and strided as q
    const float* lse;          // strides l_s_*: element of (head, token, outer)
    int64_t l_s_head, l_s_tok, l_s_outer;
    float* ws;  // workspace base: per query row z*Npad + n (z = outer * heads + head), padded to 128:
                // D_i = dO_i . O_i and lse_i*log2(e) (float32), then -lse_i/scale and -D_i as
                // 16-byte rows of three bf16
    int n_z;    // query (outer, head) pairs covered by the workspace
    // results: bf16 (dq strided as q, dk and dv as k), or float32 arrays with the
    // same strides, overwritten or (accumulate != 0) added to
    void *dq, *dk, *dv;
    float *dq_f32, *dk_f32, *dv_f32;
    int accumulate;
    int d, g, causal;
    int ring_i0, ring_t, ring_p, bsz, n_outer;  // Ulysses: 0, 0, 1, 1, 1
    int kv_gathered;  // all-gather-KV: k/v (and dk/dv) hold the whole sequence, outer index b
    // zigzag ring (as FwdParams): zz_kh is the launch's KV half; zz_qh >= 0 fixes the query half
    // (the outer index is then (rank, batch) only), -1 takes it from the outer index
    int zigzag, zz_kh, zz_qh;
    // in place in the sequence-sharded layout (as FwdParams): q, k, v, o, dout, lse and the results;
    // the workspace rows are indexed by (batch, head, global position)
    int split_np, split_b;
    float scale;
    int* status;
    // one-pass backward only: float32 dQ accumulator, n_z * Npad rows of d values in 128-row tiles,
    // each tile stored as [d/4 column groups][128 rows][4] (so that a warp's 32 rows of one group
    // are 512 contiguous bytes); null for the three-pass backward
    float* dq_acc;
};
// The three passes, in this order: the workspace rows (launch_bwd_pre covers
// all n_z rows), then dK/dV, then dQ (these two cover the launch's outer indices).
cudaError_t launch_bwd_pre(const BwdParams& p, cudaStream_t stream);
cudaError_t launch_bwd_dkdv(const BwdParams& p, cudaStream_t stream);
cudaError_t launch_bwd_dq(const BwdParams& p, cudaStream_t stream);
// The one-pass backward (bf16 results only), in this order: the workspace rows with the dQ
// accumulator zeroed (launch_bwd_pre, when p.dq_acc is set), dK, dV and the dQ partials of every
// block pair (launch_bwd_dkdvq), then dQ = scale * accumulator rounded to bf16
// (launch_bwd_dq_store).
cudaError_t launch_bwd_dkdvq(const BwdParams& p, cudaStream_t stream);
cudaError_t launch_bwd_dq_store(const BwdParams& p, cudaStream_t stream);

// ---- ring attention merge (ring.cu)
cudaError_t launch_lse_merge(int64_t rows, int d, const float* o_a, const float* lse_a, const float* o_b,
                             const float* lse_b, float* o, float* lse, cudaStream_t stream);
// fp32 partial -> bf16 output (final ring step)
cudaError_t launch_f32_to_bf16(const float* src, void* dst, int64_t n, cudaStream_t stream);
// fill float32 buffer with a constant (running LSE starts at -inf)
cudaError_t launch_fill_f32(float* dst, float value, int64_t n, cudaStream_t stream);

// ---- failure-detection probe (diag.cu): one CTA whose bounded wait gives up and records a
// timeout in *status, then returns
cudaError_t launch_wait_timeout_probe(int* status, cudaStream_t stream);
// sets *status as a timed-out wait would (if it is clear)
cudaError_t launch_raise_status(int* status, cudaStream_t stream);

// ---- argument checks of usp_attn_bwd that need no workspace (api.cu): the status usp_attn_bwd
// returns for these arguments before it looks at its workspace (USP_OK for a valid or empty problem)
usp_status attn_bwd_check(const usp_problem* p, const void* q, const void* k, const void* v, const void* o,
                          const float* lse, const void* dout, const void* dq, const void* dk, const void* dv);

// ---- tensor maps (api.cu)
// 4-D bf16 tensor map over Tensor4 with box {64, 1, 128, 1} and 128-byte swizzle.
bool make_tmap_bf16(CUtensorMap* map, const Tensor4& t, int d, int box_rows);

}  // namespace usp

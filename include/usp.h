/*
 * usp.h -- C ABI of libusp: Ulysses sequence-parallel attention on one GB300.
 *
 * What the library computes (sources are the web pages on Ulysses sequence
 * parallelism and context parallelism):
 *  - "Million-Token-Kontexte im Training" (bytewire.ai), section "Ulysses: Die
 *    Sequenz als Verteilungseinheit": the sequence is split along tokens over
 *    P devices; for attention, Q, K and V are exchanged by an all-to-all.
 *  - "Ulysses Sequence Parallelism" (topot.news), section "Как работает
 *    Ulysses": equal parts per device; after the all-to-all each device has
 *    the full context for its share of the attention.
 *  - "Context Parallelism" (ultralytics.com glossary), sections "So
 *    funktioniert Kontextparallelitaet" (ring attention: partial attention
 *    per KV block, exact equality with full-sequence attention; token-local
 *    layers on the local shard) and "Praktische Anwendung und Kompromisse"
 *    (B x H x N x d tensors with the sequence at dimension 2, causal scaled
 *    dot product attention, loss mean(out^2) and its backward).
 *
 * The P "ranks" are P slices of device buffers on ONE GPU; the all-to-all is
 * an on-device layout remap.
 *
 * Layouts (row-major, innermost last; every tensor is one contiguous device
 * buffer):
 *   logical          [B][H][N][d]
 *   sequence-sharded [P][B][N/P][H][d]   rank p holds tokens [p*N/P, (p+1)*N/P)
 *   head-sharded     [P][B][H/P][N][d]   rank r holds heads  [r*H/P, (r+1)*H/P)
 *   hybrid (2-D)     [P][B][H/Pu][N/Pr][d] rank g*Pu + u holds heads
 *                    [u*H/Pu, (u+1)*H/Pu) of token chunk g (P = Pu * Pr)
 *   LSE (head-sharded attention)    float32 [P][B][Hq/P][N]
 *   LSE (sequence-sharded ring, all-gather, fused) float32 [P][B][N/P][Hq]
 *   LSE (hybrid)                    float32 [P][B][Hq/Pu][N/Pr]
 * H is Hq for Q, O, dO, dQ and Hkv for K, V, dK, dV.  Query head h attends
 * with KV head h / (Hq/Hkv) (contiguous groups); each rank's query heads then
 * use only that rank's KV heads.
 *
 * Conventions for every entry point:
 *  - Ownership: the caller allocates and owns every buffer.  The library
 *    never allocates, frees or synchronises (except usp_device_status, which
 *    synchronises the given stream to read the status word).
 *  - Streams: all work is enqueued on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream) in call order.  Inputs must stay valid until the
 *    work completes.
 *  - Errors: arguments are validated on the host before anything is
 *    enqueued; a non-OK status means nothing was enqueued.  A launch failure
 *    returns USP_ERR_CUDA.  Device-side waits are bounded; a wait that gives
 *    up records USP_ERR_TIMEOUT in a device status word that
 *    usp_device_status() reads.  No C++ exception crosses this ABI.
 *  - Pointers: device pointers, 16-byte aligned, non-overlapping unless a
 *    function says otherwise.  Empty problems (B == 0 or N == 0) are valid
 *    and enqueue nothing.
 *  - Precision: USP_BF16 tensors are bf16 with float32 accumulation; the
 *    softmax probabilities are rounded to bf16 before the P.V product.
 *    USP_F32 attention runs in true float32 (CUDA cores, forward only).
 */
#ifndef USP_H
#define USP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    USP_OK = 0,
    USP_ERR_INVALID_ARG = 1, /* null problem, bad sizes or divisibility */
    USP_ERR_UNSUPPORTED = 2, /* valid request the library does not implement (e.g. d not 64/128) */
    USP_ERR_MISALIGNED = 3,  /* a pointer is NULL or not 16-byte aligned */
    USP_ERR_WORKSPACE = 4,   /* workspace too small */
    USP_ERR_CUDA = 5,        /* a CUDA runtime/driver call or launch failed */
    USP_ERR_TIMEOUT = 6      /* a bounded device-side wait gave up */
} usp_status;

typedef enum { USP_F32 = 0, USP_BF16 = 1 } usp_dtype;

/* The problem of the glossary page's example: Q of shape B x Hq x N x d,
 * K and V of shape B x Hkv x N x d, sequence-parallel degree P, causal flag
 * (is_causal), softmax scale (0 selects the default 1/sqrt(d)).
 * Requirements: B, N >= 0; Hq, Hkv, P >= 1; N % P == 0; Hq % Hkv == 0;
 * B * Hq <= 65535; d in {64, 128} for attention.  Every entry point except
 * the ring ones also needs Hq % P == 0 and Hkv % P == 0 (each rank gets whole
 * heads after the all-to-all). */
typedef struct {
    int B;
    int Hq;
    int Hkv;
    int N;
    int d;
    int P;
    int causal;
    float scale;
    int dtype; /* usp_dtype */
} usp_problem;

typedef void* usp_stream; /* cudaStream_t */

/* All-to-all before attention (bytewire.ai "Ulysses: Die Sequenz als
 * Verteilungseinheit"; topot.news "Как работает Ulysses"):
 *   dst[r][b][h'][n][:] = src[n/(N/P)][b][n%(N/P)][r*Hx/P + h'][:]
 * src: sequence-sharded [P][B][N/P][Hx][d]; dst: head-sharded
 * [P][B][Hx/P][N][d]; element type p->dtype.  Hx is the head count of the
 * tensor moved (p->Hq or p->Hkv); Hx % P == 0.  A bit-exact copy.
 * d * element size must be a multiple of 16 bytes.  src and dst must not
 * overlap. */
usp_status usp_a2a_seq2head(const usp_problem* p, int Hx, const void* src, void* dst, usp_stream stream);

/* All-to-all after attention, the inverse of usp_a2a_seq2head (token-local
 * layers then run on the local shard: ultralytics.com "So funktioniert"):
 *   dst[p][b][n'][h][:] = src[h/(Hx/P)][b][h%(Hx/P)][p*N/P + n'][:]
 * src head-sharded, dst sequence-sharded.  Same rules as above. */
usp_status usp_a2a_head2seq(const usp_problem* p, int Hx, const void* src, void* dst, usp_stream stream);

/* Attention forward on head-sharded buffers (every rank, one call):
 *   S_ij = scale * Q_i . K_j ;  causal: keys j > i are masked
 *   O_i  = softmax_j(S_i) V ;   lse_i = ln sum_j exp(S_ij)   (float32)
 * q, o: [P][B][Hq/P][N][d]; k, v: [P][B][Hkv/P][N][d]; lse: [P][B][Hq/P][N].
 * dtype BF16: tensor cores (d = 64 or 128).  dtype F32: float32 CUDA cores.
 * ("Context Parallelism", ultralytics.com: scaled_dot_product_attention with
 * is_causal=True in "Praktische Anwendung und Kompromisse".) */
usp_status usp_attn_fwd(const usp_problem* p, const void* q, const void* k, const void* v, void* o,
                        float* lse, usp_stream stream);

/* Bytes of workspace usp_attn_bwd needs: linear in N, never quadratic: per
 * query row, rows padded to 128-row tiles, 40 bytes (D_i and lse_i*log2(e)
 * as float32, and -lse_i/scale and -D_i each as three bf16 numbers in a
 * 16-byte row) plus the float32 dQ accumulator (4*d bytes).  Returns 0 for an
 * invalid problem. */
size_t usp_attn_bwd_workspace_size(const usp_problem* p);

/* Attention backward on head-sharded buffers (the backward of the glossary
 * page's example, any upstream gradient dO):
 *   P_ij = exp(S_ij - lse_i);  D_i = dO_i . O_i
 *   dV_j = sum_{h in group} sum_i P_ij dO_i
 *   dS_ij = P_ij (dO_i . V_j - D_i)
 *   dQ_i = scale sum_j dS_ij K_j ;  dK_j = scale sum_{h in group} sum_i dS_ij Q_i
 * q, o, dout, dq as q above; k, v, dk, dv as k above; lse from usp_attn_fwd.
 * ws: device workspace of at least usp_attn_bwd_workspace_size(p) bytes,
 * 256-byte aligned; its contents on entry do not matter.  dtype BF16 only
 * (USP_ERR_UNSUPPORTED for F32).
 * One pass over the visible block pairs computes S and dP once per pair: dK
 * and dV accumulate in fixed order (bit-reproducible); each pair's part of
 * dQ is added into a float32 accumulator in the workspace by atomic
 * reductions, whose order varies from run to run, so dQ can differ between
 * runs in its last bf16 bit.  usp_attn_bwd_deterministic gives bit-
 * reproducible results. */
usp_status usp_attn_bwd(const usp_problem* p, const void* q, const void* k, const void* v, const void* o,
                        const float* lse, const void* dout, void* dq, void* dk, void* dv, void* ws,
                        size_t ws_bytes, usp_stream stream);

/* Bytes of workspace usp_attn_bwd_deterministic needs: 40 bytes per query
 * row, rows padded to 128-row tiles (the rows of usp_attn_bwd's workspace,
 * without the dQ accumulator).  Returns 0 for an invalid problem. */
size_t usp_attn_bwd_deterministic_workspace_size(const usp_problem* p);

/* usp_attn_bwd with bit-reproducible results: the same operation, layouts and
 * checks, computed in three passes without atomics (the softmax statistics,
 * then dK and dV per key tile, then dQ per query tile, which computes S and
 * dP a second time).  dK and dV equal usp_attn_bwd's bit for bit; dQ agrees
 * within the rounding of dS to bf16 (the dQ pass forms dS its own way).
 * ws: at least usp_attn_bwd_deterministic_workspace_size(p) bytes, 256-byte
 * aligned. */
usp_status usp_attn_bwd_deterministic(const usp_problem* p, const void* q, const void* k, const void* v,
                                      const void* o, const float* lse, const void* dout, void* dq, void* dk,
                                      void* dv, void* ws, size_t ws_bytes, usp_stream stream);

/* Size of the scratch array built into the library for
 * usp_attn_bwd_noalloc: 64 MiB, enough for B*Hq*roundup(N,128) <= 1.6 Mi
 * query rows at 40 bytes each (e.g. 32 heads of 49 152 tokens): the workspace
 * of usp_attn_bwd_deterministic. */
#define USP_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/* usp_attn_bwd for callers that cannot allocate device memory -- code inside
 * a framework that owns every device allocation, plugins handed no
 * allocator, or code that must not call the allocator once running.  The
 * pages have no counterpart to this entry point; it exists for such callers.
 * Same arguments, layouts and results as usp_attn_bwd_deterministic (whose
 * small workspace suits a fixed array), minus the workspace:
 * the workspace is a file-scope device array of USP_NOALLOC_SCRATCH_BYTES
 * inside the library, held on every GPU that loads it until the process
 * exits.  Nothing is allocated or freed by the call.
 *  - Set-up: the first call on each device looks up the array's device
 *    address (cudaGetSymbolAddress) with that device current; make that first
 *    call before any stream capture.  The address is kept for the life of the
 *    process: after cudaDeviceReset on a device this entry point must not be
 *    called there again (the array may have moved; the same holds for every
 *    entry point, whose device status word is looked up the same way).
 *  - Checks: every argument check of usp_attn_bwd (sizes, d, dtype,
 *    pointers), then the size limit, come before any CUDA call.  Problems
 *    needing more than USP_NOALLOC_SCRATCH_BYTES
 *    (usp_attn_bwd_deterministic_workspace_size) return USP_ERR_WORKSPACE
 *    with nothing enqueued.
 *  - Sharing: every call on a device uses the same array, and the array keeps
 *    the last call's contents (each call rewrites every entry it reads before
 *    reading it).  Calls that can overlap on the GPU -- on different streams,
 *    or from different host threads -- race on the array and must be
 *    serialised by the caller. */
usp_status usp_attn_bwd_noalloc(const usp_problem* p, const void* q, const void* k, const void* v, const void* o,
                                const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                usp_stream stream);

/* Bytes of workspace usp_ring_attn_fwd needs: a float32 running output and a
 * float32 partial output (d values per query row) plus a float32 partial LSE
 * per query row -- linear in N.  The running LSE lives in the caller's lse. */
size_t usp_ring_workspace_size(const usp_problem* p);

/* Ring attention forward on sequence-sharded buffers ("Context
 * Parallelism", ultralytics.com, "So funktioniert Kontextparallelitaet"):
 * for step t = 0..P-1 rank i attends KV block j = (i - t) mod P -- skipped
 * when j > i under the causal mask, masked only when j == i -- and merges the
 * partial into its running result by log-sum-exp (usp_ring_merge).  Passing
 * a KV block to the next rank is an index rotation on one GPU.
 * q, o: [P][B][N/P][Hq][d] bf16; k, v: [P][B][N/P][Hkv][d] bf16;
 * lse: float32 [P][B][N/P][Hq].  ws: at least usp_ring_workspace_size(p)
 * bytes, 256-byte aligned.  dtype BF16, d in {64, 128}. */
usp_status usp_ring_attn_fwd(const usp_problem* p, const void* q, const void* k, const void* v, void* o,
                             float* lse, void* ws, size_t ws_bytes, usp_stream stream);

/* Bytes of workspace usp_ring_attn_bwd needs: 40 bytes per query row of
 * every rank and head (rows padded to 128 per rank: D_i and lse_i*log2(e) as
 * float32, -lse_i/scale and -D_i as three bf16 each), plus float32
 * accumulators for dQ, dK and dV (d values per row) -- linear in N. */
size_t usp_ring_bwd_workspace_size(const usp_problem* p);

/* Ring attention backward on sequence-sharded buffers: the gradients of the
 * causal attention of the whole sequence, computed with the ring schedule of
 * usp_ring_attn_fwd ("Context Parallelism", ultralytics.com, "So funktioniert
 * Kontextparallelitaet": at step t = 0..P-1 rank i holds KV block
 * j = (i - t) mod P, skipped when j > i under the causal mask, masked only
 * when j == i).  Each step adds rank i's partial gradients for the block
 * pair (i, j), taken with the merged LSE of the forward and D_i = dO_i . O_i:
 *   dQ_i += scale sum_j dS_ij K_j   (stays on rank i)
 *   dK_j += scale sum_{h in group} sum_i dS_ij Q_i,  dV_j += sum P_ij dO_i
 *                                   (travel with the KV block)
 * in float32, then rounds once to bf16.  The pages name no ring backward;
 * this is the plain reading that the forward's schedule and the backward of
 * the glossary page's example leave.
 * q, o, dout, dq: [P][B][N/P][Hq][d] bf16; k, v, dk, dv: [P][B][N/P][Hkv][d]
 * bf16; lse: float32 [P][B][N/P][Hq] from usp_ring_attn_fwd.  ws: at least
 * usp_ring_bwd_workspace_size(p) bytes, 256-byte aligned, contents on entry
 * irrelevant.  dtype BF16, d in {64, 128}; Hq % Hkv == 0; N % P == 0. */
usp_status usp_ring_attn_bwd(const usp_problem* p, const void* q, const void* k, const void* v, const void* o,
                             const float* lse, const void* dout, void* dq, void* dk, void* dv, void* ws,
                             size_t ws_bytes, usp_stream stream);

/* ---- all-gather-KV context parallelism ("Context Parallelism",
 * ultralytics.com, "So funktioniert Kontextparallelitaet": the variant in
 * which every rank gathers the whole K and V and attends its own query
 * shard).  On one GPU the gather is one device copy per (rank, batch) chunk
 * into the workspace; the attention of rank i uses global token positions
 * (its queries are tokens i*N/P ..), so causal masking spans shards. */

/* Bytes of workspace usp_allgather_attn_fwd needs: the gathered K and V
 * (bf16, B*N*Hkv*d each) -- linear in N. */
size_t usp_allgather_workspace_size(const usp_problem* p);

/* Forward: o, lse of every rank's query shard against all keys.
 * q, o: [P][B][N/P][Hq][d] bf16; k, v: [P][B][N/P][Hkv][d] bf16; lse: float32
 * [P][B][N/P][Hq].  ws: at least usp_allgather_workspace_size(p) bytes,
 * 256-byte aligned.  dtype BF16, d in {64, 128}; Hq % Hkv == 0; N % P == 0. */
usp_status usp_allgather_attn_fwd(const usp_problem* p, const void* q, const void* k, const void* v, void* o,
                                  float* lse, void* ws, size_t ws_bytes, usp_stream stream);

/* Bytes of workspace usp_allgather_attn_bwd needs: the gathered K and V,
 * 40 bytes per padded query row of every rank and head, and float32 dK, dV
 * accumulators for the whole sequence -- linear in N. */
size_t usp_allgather_bwd_workspace_size(const usp_problem* p);

/* Backward of usp_allgather_attn_fwd: dQ_i from one pass of rank i over the
 * gathered keys; dK and dV as the sum over ranks of each rank's partial over
 * all keys (float32, summed in rank order: the reduce of a reduce-scatter),
 * after which rank j keeps its shard's rows, rounded to bf16 (the scatter).
 * Layouts as in the forward; dout, dq like q; dk, dv like k.  ws: at least
 * usp_allgather_bwd_workspace_size(p) bytes, 256-byte aligned. */
usp_status usp_allgather_attn_bwd(const usp_problem* p, const void* q, const void* k, const void* v, const void* o,
                                  const float* lse, const void* dout, void* dq, void* dk, void* dv, void* ws,
                                  size_t ws_bytes, usp_stream stream);

/* ---- zigzag (load-balanced) ring attention.  Causal ring attention over
 * contiguous shards gives rank i i+1 of the P block pairs; the zigzag layout
 * cuts the sequence into 2P chunks of c = N/(2P) tokens and gives rank r
 * chunks r and 2P-1-r, so that every rank does the same work at every ring
 * step.  The pages describe the ring without a balance; this layout is the
 * plain balanced reading of it.
 * Zigzag-sharded buffers: [P][B][2][c][H][d] -- rank r's shard holds chunk r
 * then chunk 2P-1-r.  Requires N % (2P) == 0 (USP_ERR_INVALID_ARG otherwise). */

/* Contiguous sequence shards ([P][B][N/P][Hx][d], as usp_a2a_seq2head reads)
 * to zigzag shards and back: a permutation of c-token chunks, one device copy
 * each.  dtype gives the element size; src and dst must not overlap. */
usp_status usp_zigzag_shard(const usp_problem* p, int Hx, const void* src, void* dst, usp_stream stream);
usp_status usp_zigzag_unshard(const usp_problem* p, int Hx, const void* src, void* dst, usp_stream stream);

/* Workspace of usp_zigzag_attn_fwd (equal to usp_ring_workspace_size) and of
 * usp_zigzag_attn_bwd (40 bytes per padded query row of every chunk and head,
 * float32 dQ, dK, dV accumulators) -- linear in N; 0 for an invalid problem. */
size_t usp_zigzag_workspace_size(const usp_problem* p);
size_t usp_zigzag_bwd_workspace_size(const usp_problem* p);

/* Zigzag ring forward: at step t = 0..P-1 rank i holds the KV chunks of rank
 * j = (i - t) mod P and attends both of its query chunks to each of them at
 * global positions (pairs wholly in the future are empty), merging every
 * partial by log-sum-exp as usp_ring_attn_fwd does.  q, o, lse, k, v in the
 * zigzag layout (lse: float32 [P][B][2][c][Hq]).  dtype BF16, d in {64, 128}. */
usp_status usp_zigzag_attn_fwd(const usp_problem* p, const void* q, const void* k, const void* v, void* o,
                               float* lse, void* ws, size_t ws_bytes, usp_stream stream);

/* Zigzag ring backward: usp_ring_attn_bwd's accumulation over the same chunk
 * pairs (dK, dV travel with the KV chunks, dQ stays), float32, rounded once
 * to bf16.  Layouts as in the forward. */
usp_status usp_zigzag_attn_bwd(const usp_problem* p, const void* q, const void* k, const void* v, const void* o,
                               const float* lse, const void* dout, void* dq, void* dk, void* dv, void* ws,
                               size_t ws_bytes, usp_stream stream);

/* ---- Ulysses attention with the all-to-all fused into the kernels ("Million-
 * Token-Kontexte im Training", bytewire.ai, "Ulysses: Die Sequenz als
 * Verteilungseinheit": the exchange that gives each rank the whole sequence
 * for its heads).  The attention kernels read Q, K, V and dO and write O, LSE,
 * dQ, dK and dV in place in the sequence-sharded layout: every tile load and
 * every result row addresses token n of a head as row n mod (N/P) of shard
 * n div (N/P), so no remap runs and no head-sharded copy exists.  Results are
 * those of usp_a2a_seq2head -> usp_attn_fwd / usp_attn_bwd -> usp_a2a_head2seq,
 * bit for bit (the same per-head work, tile for tile), except dQ, whose
 * float32 accumulation order varies from run to run in both (see
 * usp_attn_bwd); only the LSE layout differs: float32 [P][B][N/P][Hq], as in
 * ring mode.
 * Preconditions as usp_attn_fwd (Hq % P = Hkv % P = 0, dtype BF16, d in
 * {64, 128}) plus (N/P) % 128 == 0: a 128-row tile never straddles two shards
 * (USP_ERR_UNSUPPORTED otherwise). */
usp_status usp_fused_attn_fwd(const usp_problem* p, const void* q, const void* k, const void* v, void* o,
                              float* lse, usp_stream stream);

/* Bytes of workspace usp_fused_attn_bwd needs (equal to
 * usp_attn_bwd_workspace_size); 0 for an invalid problem. */
size_t usp_fused_attn_bwd_workspace_size(const usp_problem* p);

/* Backward of usp_fused_attn_fwd (the one-pass backward of usp_attn_bwd):
 * q, k, v, o, dout, dq, dk, dv sequence-sharded, lse as the forward wrote it.
 * ws: at least usp_fused_attn_bwd_workspace_size(p) bytes, 256-byte
 * aligned. */
usp_status usp_fused_attn_bwd(const usp_problem* p, const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dout, void* dq, void* dk, void* dv, void* ws,
                              size_t ws_bytes, usp_stream stream);

/* ---- 2-D (hybrid) sequence parallelism: Ulysses inside groups of Pu ranks,
 * ring attention across the Pr = P/Pu groups (the pages name hybrid
 * strategies -- bytewire.ai, "Praktische Implikationen fuer den Einsatz" --
 * and both exchanges: the all-to-all, and the ring of "Context Parallelism",
 * ultralytics.com, "So funktioniert Kontextparallelitaet").
 * Group g holds the contiguous token chunk g of Nc = N/Pr tokens (its ranks
 * g*Pu .. g*Pu + Pu - 1 hold the chunk's Pu shards of N/P tokens).  The
 * all-to-all inside the group gives rank g*Pu + u the heads u*H/Pu ..
 * (u+1)*H/Pu - 1 of the chunk: the hybrid layout [P][B][H/Pu][Nc][d], LSE
 * float32 [P][B][Hq/Pu][Nc].  Pu = P is the Ulysses layout (Pr = 1), Pu = 1
 * per-rank head-major shards of the ring.
 * Every hybrid call: Pu >= 1, P % Pu == 0, Hq % Pu == 0, Hkv % Pu == 0 (else
 * USP_ERR_INVALID_ARG), plus the usp_problem checks without the head split. */

/* Sequence-sharded [P][B][N/P][Hx][d] -> hybrid layout (one Ulysses remap of
 * Nc tokens over Pu ranks per group), and back.  Bit copies, any dtype,
 * d * element size in {64, 128, 256, 512} bytes; src and dst must not
 * overlap. */
usp_status usp_hybrid_seq2head(const usp_problem* p, int Pu, int Hx, const void* src, void* dst, usp_stream stream);
usp_status usp_hybrid_head2seq(const usp_problem* p, int Pu, int Hx, const void* src, void* dst, usp_stream stream);

/* Bytes of workspace usp_hybrid_attn_fwd needs (float32 running and partial
 * outputs and partial LSE, as usp_ring_workspace_size) and usp_hybrid_attn_bwd
 * needs (40 bytes per padded query row of every rank and local head, float32
 * dQ, dK, dV accumulators); 0 for an invalid problem. */
size_t usp_hybrid_workspace_size(const usp_problem* p, int Pu);
size_t usp_hybrid_bwd_workspace_size(const usp_problem* p, int Pu);

/* Hybrid forward on hybrid-layout q, k, v: at ring step t = 0..Pr-1 the ranks
 * of group i attend their heads of chunk i to the same heads' KV of chunk
 * j = (i - t) mod Pr (skipped when j > i under the causal mask), each partial
 * merged by log-sum-exp as usp_ring_attn_fwd does; o (bf16) and lse in the
 * hybrid layout.  dtype BF16, d in {64, 128}; ws 256-byte aligned. */
usp_status usp_hybrid_attn_fwd(const usp_problem* p, int Pu, const void* q, const void* k, const void* v, void* o,
                               float* lse, void* ws, size_t ws_bytes, usp_stream stream);

/* Hybrid backward: usp_ring_attn_bwd's schedule over the groups (dK, dV
 * travel with the KV chunk, dQ stays), float32, rounded once to bf16; every
 * tensor in the hybrid layout, lse as the forward wrote it. */
usp_status usp_hybrid_attn_bwd(const usp_problem* p, int Pu, const void* q, const void* k, const void* v,
                               const void* o, const float* lse, const void* dout, void* dq, void* dk, void* dv,
                               void* ws, size_t ws_bytes, usp_stream stream);

/* Exact merge of two partial attentions over disjoint key sets, float32
 * (the merge step of ring attention):
 *   lse = ln(exp(lse_a) + exp(lse_b))
 *   o   = exp(lse_a - lse) o_a + exp(lse_b - lse) o_b
 * A row with lse = -inf is an empty partial and contributes nothing; two
 * empty rows give lse = -inf and o = 0.
 * o_*: [rows][d]; lse_*: [rows].  o may alias o_a or o_b and lse may alias
 * lse_a or lse_b (element-wise, in place).  d >= 1 and d % 4 == 0. */
usp_status usp_ring_merge(int64_t rows, int d, const float* o_a, const float* lse_a, const float* o_b,
                          const float* lse_b, float* o, float* lse, usp_stream stream);

/* ---- kernel tracing ----
 * When enabled, every kernel the library launches is bracketed by two CUDA
 * events recorded on the launch's stream (a few microseconds per launch).
 * usp_trace_report() waits for the pending events and accumulates, per
 * kernel name, the launch count and the summed event-to-event milliseconds.
 * Tracing state is process-wide and not meant for concurrent threads. */
typedef struct {
    char name[32];    /* kernel name, e.g. "attn_fwd", "attn_bwd_dkdv", "a2a_seq2head" */
    int64_t launches; /* launches since the last reset */
    double total_ms;  /* summed durations */
} usp_trace_entry;

/* Turn tracing on (on != 0) or off.  Always USP_OK. */
usp_status usp_trace_enable(int on);

/* Drop pending events and accumulated totals.  Always USP_OK. */
usp_status usp_trace_reset(void);

/* Resolve pending events (this synchronises on them) and write up to
 * max_entries totals into out (out may be NULL to query the count).
 * Returns the number of distinct kernel names, or -1 if an event failed. */
int usp_trace_report(usp_trace_entry* out, int max_entries);

/* Synchronises `stream` and reads the device status word that bounded
 * device-side waits write: USP_OK, or USP_ERR_TIMEOUT (the word is then
 * cleared).  USP_ERR_CUDA if the synchronisation itself fails. */
usp_status usp_device_status(usp_stream stream);

/* Failure-detection check, without a fault: enqueues one CTA that waits on a
 * barrier phase nothing completes.  Its bounded wait gives up after the wait
 * limit (2 s), records a timeout in the device status word exactly as a
 * stalled kernel would, and returns.  usp_device_status() then reports
 * USP_ERR_TIMEOUT and clears the word; the context stays usable.  USP_OK once
 * enqueued, USP_ERR_CUDA if the launch fails. */
usp_status usp_diag_wait_timeout(usp_stream stream);

/* Failure-detection check of the attention kernels' abort path, without a
 * fault: enqueues a write of a timeout record into the device status word
 * (if it is clear), as a wait that gave up would.  Every CTA of the kernels
 * enqueued after it then gives up at its first wait that is not already
 * satisfied, waits (bounded) for its own TMA loads and MMAs in flight, frees
 * its TMEM and returns; their outputs are then undefined.
 * usp_device_status() reports USP_ERR_TIMEOUT and clears the word, after
 * which the context runs every path normally.  USP_OK once enqueued,
 * USP_ERR_CUDA if the launch fails. */
usp_status usp_diag_raise_status(usp_stream stream);

/* Static, human-readable name of a status code. */
const char* usp_status_string(usp_status s);

/* Static build description (architecture, version). */
const char* usp_build_info(void);

#ifdef __cplusplus
}
#endif

#endif /* USP_H */

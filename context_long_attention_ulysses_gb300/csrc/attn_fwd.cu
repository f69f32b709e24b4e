// Causal, GQA-aware flash-attention forward on sm_103a tensor cores.
//
// Computes, per query row i of a head, S_ij = scale * Q_i . K_j (keys j <= i
// under the causal mask), O_i = softmax_j(S_ij) V and lse_i = ln sum_j
// exp(S_ij): the scaled dot product attention of the code example on the
// "Context Parallelism" glossary page (ultralytics.com, "Praktische
// Anwendung und Kompromisse"), evaluated per rank after the Ulysses
// all-to-all, or per KV block as the partial attention of ring attention
// ("So funktioniert Kontextparallelitaet" on the same page).
//
// One CTA owns a 128-row query tile and walks the visible 128-key tiles:
//   warp 4      TMA producer: K_j and V_j into 3-4 stage rings
//   warp 5      TMEM owner + single-thread tcgen05.mma issuer:
//                 S_j = Q K_j^T  (Q from TMEM as bf16, K_j K-major in shared memory)
//                 O  += P_j V_j  (P_j from TMEM as bf16, V_j MN-major)
//   warps 0-3   softmax: thread = query row = TMEM lane; online softmax in
//               the log2 domain with lazy rescaling of O (only when the
//               running max grows by more than 2^8), P written back to TMEM
//               as bf16, final normalisation, O and LSE stores.
// TMEM columns: S0 [0,128), S1 [128,256), O [256,256+D), P (64), Q (D/2).
// S is double-buffered so QK^T of tile j+2 and PV of tile j run on the tensor
// core while the softmax works on tile j+1.  Q sits in TMEM (staged once by
// the softmax threads from global memory) so that the tensor core reads only
// K and V from shared memory: per tile 32 KB K + 32 KB V of MMA reads plus
// 64 KB of TMA writes, which shared-memory bandwidth (128 B/clk) serves in
// the 1024 cycles the two 128x128x128 products take.  P is single-buffered:
// the softmax of tile j writes it only after PV of tile j-1 has completed.
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"

namespace usp {

namespace {

constexpr int kBM = 128;           // query rows per CTA
constexpr int kBN = 128;           // keys per tile
constexpr int kSoftmaxWarps = 4;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreads = 6 * 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8

template <int D>
struct FwdCfg {
    static constexpr int kChunks = D / 64;                 // 64-column (128-byte) swizzle atoms per row
    static constexpr int kTileBytes = kChunks * 128 * 128; // one 128-row bf16 tile
    // 3-4 tiles in flight per ring hide the L2->SMEM latency (Q lives in TMEM, not here)
    static constexpr int kKStages = 4;
    static constexpr int kVStages = D == 64 ? 4 : 3;
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + kKStages * kTileBytes;
    static constexpr int kOffBar = kOffV + kVStages * kTileBytes;
    static constexpr int kNumBars = 1 + 2 * kKStages + 2 * kVStages + 2 + 2 + 2;
    static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;  // + TMEM slot, + alignment slack
    // TMEM: S double-buffered, O, P (bf16, single), Q (bf16, the A operand of Q K^T)
    static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256, kColP = 256 + D, kColQ = 256 + D + 64;
    static constexpr uint32_t kTmemCols = 512;
};

struct DevFwd {
    const uint16_t* q;                       // bf16 Q, addressed like Tensor4
    int64_t q_s_head, q_s_tok, q_s_outer;    // elements
    int d, g, n_heads, n_outer, q_len, kv_len;
    int ring_i0, ring_t, ring_p, bsz, np;
    int causal;
    float scale_log2;
    void* o_bf16;
    float* o_f32;
    int64_t o_s_head, o_s_tok, o_s_outer;
    float* lse;
    int64_t l_s_head, l_s_tok, l_s_outer;
    int* status;
};

// Where a work item sits: query tile, heads, outer indices and token offsets.
struct WorkItem {
    int r0;          // first query row (local token) of the tile
    int head, kv_head;
    int q_outer, kv_outer;
    long q_pos0, kv_pos0;  // global positions of local token 0
    int n_tiles;     // visible key tiles (0: nothing visible)
};

__device__ __forceinline__ WorkItem decode_item(const DevFwd& p) {
    const int n_qt = (p.q_len + kBM - 1) / kBM;
    const int per_tile = p.n_heads * p.n_outer;
    const int item = blockIdx.x;
    WorkItem w;
    // heaviest (last) query tiles first: causal work grows with the tile index
    const int qt = n_qt - 1 - item / per_tile;
    const int rest = item % per_tile;
    w.head = rest % p.n_heads;
    const int o = rest / p.n_heads;
    w.kv_head = w.head / p.g;
    const int i = p.ring_i0 + o / p.bsz;
    const int b = o % p.bsz;
    const int j = ((i - p.ring_t) % p.ring_p + p.ring_p) % p.ring_p;
    w.q_outer = i * p.bsz + b;
    w.kv_outer = j * p.bsz + b;
    w.q_pos0 = (long)i * p.np;
    w.kv_pos0 = (long)j * p.np;
    w.r0 = qt * kBM;
    int kv_end = p.kv_len;
    if (p.causal) {
        const long last_q = w.q_pos0 + min(w.r0 + kBM, p.q_len) - 1;  // position of the tile's last row
        const long vis = last_q - w.kv_pos0 + 1;                      // keys with position <= last_q
        kv_end = (int)max(0L, min((long)p.kv_len, vis));
    }
    w.n_tiles = (kv_end + kBN - 1) / kBN;
    return w;
}

template <int D, bool OUT_F32>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v, const DevFwd p) {
    using C = FwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + C::kNumBars * 8);
    __shared__ int abort_flag;

    // barrier indices
    const uint32_t bar0 = smem_u32(bars);
    auto BAR = [&](int idx) { return bar0 + 8u * (uint32_t)idx; };
    const int kQFull = 0;
    const int kKFull = 1, kKEmpty = kKFull + C::kKStages;
    const int kVFull = kKEmpty + C::kKStages, kVEmpty = kVFull + C::kVStages;
    const int kSFull = kVEmpty + C::kVStages;  // 2
    const int kPReady = kSFull + 2;            // 2
    const int kPvDone = kPReady + 2;
    const int kOReady = kPvDone + 1;

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const WorkItem w = decode_item(p);

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(BAR(kQFull), kSoftmaxWarps * 32);  // the softmax threads stage Q into TMEM
        for (int s = 0; s < C::kKStages; ++s) { mbar_init(BAR(kKFull + s), 1); mbar_init(BAR(kKEmpty + s), 1); }
        for (int s = 0; s < C::kVStages; ++s) { mbar_init(BAR(kVFull + s), 1); mbar_init(BAR(kVEmpty + s), 1); }
        for (int s = 0; s < 2; ++s) {
            mbar_init(BAR(kSFull + s), 1);
            mbar_init(BAR(kPReady + s), kSoftmaxWarps * 32);
        }
        mbar_init(BAR(kPvDone), 1);
        mbar_init(BAR(kOReady), 1);
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    volatile int* abort_p = &abort_flag;

    if (w.n_tiles > 0 && warp == kProducerWarp && lane == 0) {
        // ---------------------------------------------------------------- TMA producer
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        for (int j = 0; j < w.n_tiles; ++j) {
            const int ks = j % C::kKStages, vs = j % C::kVStages;
            if (j >= C::kKStages && !mbar_wait(BAR(kKEmpty + ks), ((j / C::kKStages) - 1) & 1, abort_p, 1, p.status))
                break;
            mbar_arrive_expect_tx(BAR(kKFull + ks), C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c)
                tma_load_4d(sbase + C::kOffK + ks * C::kTileBytes + c * 16384, &tm_k, c * 64, w.kv_head, j * kBN,
                            w.kv_outer, BAR(kKFull + ks));
            if (j >= C::kVStages && !mbar_wait(BAR(kVEmpty + vs), ((j / C::kVStages) - 1) & 1, abort_p, 2, p.status))
                break;
            mbar_arrive_expect_tx(BAR(kVFull + vs), C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c)
                tma_load_4d(sbase + C::kOffV + vs * C::kTileBytes + c * 16384, &tm_v, c * 64, w.kv_head, j * kBN,
                            w.kv_outer, BAR(kVFull + vs));
        }
    } else if (w.n_tiles > 0 && warp == kMmaWarp && lane == 0) {
        // ---------------------------------------------------------------- MMA issuer
        constexpr uint32_t kIdS = idesc_bf16(kBM, kBN, 0, 0);  // S = Q K^T, both K-major
        constexpr uint32_t kIdO = idesc_bf16(kBM, D, 0, 1);    // O += P V, V MN-major
        auto issue_qk = [&](int j) -> bool {
            const int ks = j % C::kKStages;
            if (!mbar_wait(BAR(kKFull + ks), (j / C::kKStages) & 1, abort_p, 3, p.status)) return false;
            tc_fence_after();
            const uint64_t dk0 = sdesc_sw128(sbase + C::kOffK + ks * C::kTileBytes, 16, 1024);
            const uint32_t dcol = tmem + ((j & 1) ? C::kColS1 : C::kColS0);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = ((kk / 4) * 16384 + (kk % 4) * 32) >> 4;  // descriptor address units
                mma_ts(dcol, tmem + C::kColQ + kk * 8, dk0 + off, kIdS, kk > 0);  // A = Q from TMEM
            }
            mma_commit(BAR(kSFull + (j & 1)));
            mma_commit(BAR(kKEmpty + ks));
            return true;
        };
        bool ok = mbar_wait(BAR(kQFull), 0, abort_p, 4, p.status);
        ok = ok && issue_qk(0);
        if (ok && w.n_tiles > 1) ok = issue_qk(1);
        for (int j = 0; ok && j < w.n_tiles; ++j) {
            const int vs = j % C::kVStages;
            if (!mbar_wait(BAR(kPReady + (j & 1)), (j >> 1) & 1, abort_p, 5, p.status)) break;
            if (!mbar_wait(BAR(kVFull + vs), (j / C::kVStages) & 1, abort_p, 6, p.status)) break;
            tc_fence_after();
            const uint64_t dv0 = sdesc_sw128(sbase + C::kOffV + vs * C::kTileBytes, 16384, 1024);
            const uint32_t pcol = tmem + C::kColP;
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
                mma_ts(tmem + C::kColO, pcol + kk * 8, dv0 + (kk * 2048 >> 4), kIdO, (j > 0 || kk > 0) ? 1u : 0u);
            mma_commit(BAR(kVEmpty + vs));
            mma_commit(BAR(kPvDone));
            if (j + 2 < w.n_tiles) ok = issue_qk(j + 2);
        }
        if (ok) mma_commit(BAR(kOReady));
    } else if (warp < kSoftmaxWarps) {
        // ---------------------------------------------------------------- softmax warps
        const int row = threadIdx.x;  // query row within the tile = TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        const long q_pos = w.q_pos0 + w.r0 + row;
        float m_run = -INFINITY;  // running max of scale*log2(e)*S over the row (log2 units)
        float l_run = 0.f;        // running sum of 2^(scaled S - m_run)
        bool ok = true;
        if (w.n_tiles > 0) {
            // Q row -> TMEM (A operand of Q K^T): bf16 pairs packed per 32-bit column, zeros past q_len
            const int tok = w.r0 + row;
            const uint4* src = reinterpret_cast<const uint4*>(p.q + (int64_t)w.head * p.q_s_head +
                                                              (int64_t)tok * p.q_s_tok +
                                                              (int64_t)w.q_outer * p.q_s_outer);
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                uint32_t qr[32];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint4 v = tok < p.q_len ? __ldg(src + c * 8 + e) : make_uint4(0u, 0u, 0u, 0u);
                    qr[4 * e] = v.x;
                    qr[4 * e + 1] = v.y;
                    qr[4 * e + 2] = v.z;
                    qr[4 * e + 3] = v.w;
                }
                tmem_st32(lane_base + C::kColQ + c * 32, qr);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(BAR(kQFull));
        }
        for (int j = 0; j < w.n_tiles; ++j) {
            if (!mbar_wait(BAR(kSFull + (j & 1)), (j >> 1) & 1, abort_p, 7, p.status)) { ok = false; break; }
            tc_fence_after();
            const uint32_t scol = lane_base + ((j & 1) ? C::kColS1 : C::kColS0);
            uint32_t r0[32], r1[32], r2[32], r3[32];
            tmem_ld32(scol, r0);
            tmem_ld32(scol + 32, r1);
            tmem_ld32(scol + 64, r2);
            tmem_ld32(scol + 96, r3);
            tmem_wait_ld();
            float s[kBN];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                s[c] = __uint_as_float(r0[c]);
                s[32 + c] = __uint_as_float(r1[c]);
                s[64 + c] = __uint_as_float(r2[c]);
                s[96 + c] = __uint_as_float(r3[c]);
            }
            const long key0 = w.kv_pos0 + (long)j * kBN;
            const int kv_rem = p.kv_len - j * kBN;
            if ((p.causal && key0 + kBN - 1 > w.q_pos0 + w.r0) || kv_rem < kBN) {
                // last visible column of this row in this tile
                long lim = p.causal ? q_pos - key0 : (long)(kBN - 1);
                lim = min(lim, (long)kv_rem - 1);
                const int climit = (int)max(-1L, min(lim, (long)(kBN - 1)));
#pragma unroll
                for (int c = 0; c < kBN; ++c)
                    if (c > climit) s[c] = -INFINITY;
            }
            // row max as eight independent chains (a single chain would be 128 dependent ops)
            float m8[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) m8[c] = s[c];
#pragma unroll
            for (int c = 8; c < kBN; ++c) m8[c & 7] = fmaxf(m8[c & 7], s[c]);
            float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                             fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
            mx *= p.scale_log2;
            const float m_new = fmaxf(m_run, mx);
            const bool rescale = m_new > m_run + kRescaleThreshold;
            const float m_use = rescale ? m_new : m_run;
            const float alpha = rescale ? ex2_approx(m_run - m_new) : 1.f;
            const float msub = m_use == -INFINITY ? 0.f : m_use;
            float sum4[4] = {0.f, 0.f, 0.f, 0.f};  // four partial sums: independent chains
            uint32_t pk0[32], pk1[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float p0 = ex2_approx(fmaf(s[2 * c], p.scale_log2, -msub));
                const float p1 = ex2_approx(fmaf(s[2 * c + 1], p.scale_log2, -msub));
                const float p2 = ex2_approx(fmaf(s[64 + 2 * c], p.scale_log2, -msub));
                const float p3 = ex2_approx(fmaf(s[64 + 2 * c + 1], p.scale_log2, -msub));
                sum4[c & 3] += (p0 + p1) + (p2 + p3);
                pk0[c] = pack_bf16(p0, p1);
                pk1[c] = pack_bf16(p2, p3);
            }
            l_run = l_run * alpha + ((sum4[0] + sum4[1]) + (sum4[2] + sum4[3]));
            if (j > 0) {
                // P and O are read by PV of tile j-1: wait until it has completed (QK of tile j was
                // issued after PV of tile j-2, so at most PV j-1 is outstanding: the parity test is exact)
                if (!mbar_wait(BAR(kPvDone), (j - 1) & 1, abort_p, 8, p.status)) { ok = false; break; }
                tc_fence_after();
            }
            tmem_st32(lane_base + C::kColP, pk0);
            tmem_st32(lane_base + C::kColP + 32, pk1);
            if (rescale && j > 0) {
                // O holds PV of tiles < j (all complete): scale in place
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(lane_base + C::kColO + c * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st32(lane_base + C::kColO + c * 32, o);
                }
            }
            m_run = m_use;
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(BAR(kPReady + (j & 1)));
        }
        // ---------------------------------------------------------------- epilogue
        if (ok && w.n_tiles > 0) ok = mbar_wait(BAR(kOReady), 0, abort_p, 9, p.status);
        if (ok) {
            tc_fence_after();
            const bool has = w.n_tiles > 0 && l_run > 0.f;
            const float inv = has ? 1.f / l_run : 0.f;
            const float lse_v = has ? (m_run + lg2_approx(l_run)) * kLn2 : -INFINITY;
            const int tok = w.r0 + row;
            const bool valid = tok < p.q_len;
            const int64_t obase = (int64_t)w.head * p.o_s_head + (int64_t)tok * p.o_s_tok + (int64_t)w.q_outer * p.o_s_outer;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                if (w.n_tiles > 0) {
                    tmem_ld32(lane_base + C::kColO + c * 32, o);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = 0u;
                }
                if (valid) {
                    if constexpr (OUT_F32) {
                        float4* dst = reinterpret_cast<float4*>(p.o_f32 + obase + c * 32);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            dst[e] = make_float4(__uint_as_float(o[4 * e]) * inv, __uint_as_float(o[4 * e + 1]) * inv,
                                                 __uint_as_float(o[4 * e + 2]) * inv, __uint_as_float(o[4 * e + 3]) * inv);
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o_bf16) + obase + c * 32);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            uint4 v;
                            v.x = pack_bf16(__uint_as_float(o[8 * e + 0]) * inv, __uint_as_float(o[8 * e + 1]) * inv);
                            v.y = pack_bf16(__uint_as_float(o[8 * e + 2]) * inv, __uint_as_float(o[8 * e + 3]) * inv);
                            v.z = pack_bf16(__uint_as_float(o[8 * e + 4]) * inv, __uint_as_float(o[8 * e + 5]) * inv);
                            v.w = pack_bf16(__uint_as_float(o[8 * e + 6]) * inv, __uint_as_float(o[8 * e + 7]) * inv);
                            dst[e] = v;
                        }
                    }
                }
            }
            if (valid)
                p.lse[(int64_t)w.head * p.l_s_head + (int64_t)tok * p.l_s_tok + (int64_t)w.q_outer * p.l_s_outer] = lse_v;
        }
    }
    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D, bool OUT_F32>
cudaError_t launch_fwd_t(const FwdParams& f, cudaStream_t stream) {
    using C = FwdCfg<D>;
    CUtensorMap tk, tv;
    if (!make_tmap_bf16(&tk, f.k, D, kBN) || !make_tmap_bf16(&tv, f.v, D, kBN)) return cudaErrorInvalidValue;
    DevFwd p;
    p.q = static_cast<const uint16_t*>(f.q.ptr);
    p.q_s_head = f.q.s_head;
    p.q_s_tok = f.q.s_tok;
    p.q_s_outer = f.q.s_outer;
    p.d = D;
    p.g = f.g;
    p.n_heads = f.n_heads;
    p.n_outer = f.n_outer;
    p.q_len = f.q_len;
    p.kv_len = f.kv_len;
    p.ring_i0 = f.ring_i0;
    p.ring_t = f.ring_t;
    p.ring_p = f.ring_p;
    p.bsz = f.bsz;
    p.np = f.np;
    p.causal = f.causal;
    p.scale_log2 = f.scale * kLog2e;
    p.o_bf16 = f.o_bf16;
    p.o_f32 = f.o_f32;
    p.o_s_head = f.o_s_head;
    p.o_s_tok = f.o_s_tok;
    p.o_s_outer = f.o_s_outer;
    p.lse = f.lse;
    p.l_s_head = f.l_s_head;
    p.l_s_tok = f.l_s_tok;
    p.l_s_outer = f.l_s_outer;
    p.status = f.status;
    auto kern = attn_fwd_kernel<D, OUT_F32>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const long n_qt = (f.q_len + kBM - 1) / kBM;
    const long items = n_qt * (long)f.n_heads * (long)f.n_outer;
    if (items == 0) return cudaSuccess;
    kern<<<(unsigned)items, kThreads, C::kSmemBytes, stream>>>(tk, tv, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd_bf16(const FwdParams& f, cudaStream_t stream) {
    const bool f32 = f.o_f32 != nullptr;
    if (f.d == 64) return f32 ? launch_fwd_t<64, true>(f, stream) : launch_fwd_t<64, false>(f, stream);
    if (f.d == 128) return f32 ? launch_fwd_t<128, true>(f, stream) : launch_fwd_t<128, false>(f, stream);
    return cudaErrorInvalidValue;
}

}  // namespace usp

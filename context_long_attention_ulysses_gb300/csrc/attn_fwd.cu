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
// One CTA owns 256 query rows as two independent 128-row streams A and B
// that share every K/V tile it loads:
//   warp 8      TMA producer: both Q tiles once, then K_j and V_j into rings
//   warp 9      TMEM owner + single-thread tcgen05.mma issuer, per key tile j:
//                 PV_A(j), QK_A(j+1), PV_B(j), QK_B(j+1)
//               (S = Q K^T with both operands in shared memory, O += P V with
//               P from TMEM as bf16 and V MN-major)
//   warps 0-3   softmax of stream A, warps 4-7 softmax of stream B: thread =
//               query row = TMEM lane; online softmax in the log2 domain with
//               lazy rescaling of O (only when the running max grows by more
//               than 2^8), final normalisation, O and LSE stores.
// While one stream's softmax works on its S tile, the tensor core runs the
// other stream's products, so it always has queued work.
// TMEM columns: S_A [0,128), S_B [128,256), O_A [256,256+D), O_B [384,384+D).
// A stream's P (bf16) is written over the first 64 columns of its own S after
// the softmax has loaded S; the next QK^T into that S is issued after the PV
// that reads P (tcgen05.mma executes in issue order).  The commit that
// signals S(j) also covers PV(j-1), so P and O are free whenever the softmax
// sees its next S.
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"

namespace usp {

namespace {

constexpr int kBM = 128;           // query rows per stream
constexpr int kStreams = 2;        // query tiles per CTA
constexpr int kBN = 128;           // keys per tile
constexpr int kSoftmaxWarps = 8;   // 4 per stream (warpgroups 0 and 1)
constexpr int kProducerWarp = 8;   // warpgroup 2: producer, MMA issuer, two idle warps
constexpr int kMmaWarp = 9;
constexpr int kThreads = 12 * 32;
// Registers per thread after the set-up: the launch gives every warp 168 (65536 / 384, rounded down
// to 8). Warpgroup 2 gives some back so the softmax warps can hold a whole S row in registers. Per
// sub-partition (one warp of each warpgroup): 2 * 208 + 88 <= 3 * 168; per CTA 8 * 208 + 4 * 88 <= 12 * 168.
// With 88 (not 80) the producer and MMA issuer spill nothing in any instantiation (measured at
// 128K, d = 128: 85.1 ms against 85.7).
constexpr int kSoftmaxRegs = 208;
constexpr int kOtherRegs = 88;
static_assert(2 * kSoftmaxRegs + kOtherRegs <= 3 * 168, "register split exceeds the launch allocation");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8

template <int D>
struct FwdCfg {
    static constexpr int kChunks = D / 64;                 // 64-column (128-byte) swizzle atoms per row
    static constexpr int kTileBytes = kChunks * 128 * 128; // one 128-row bf16 tile
    static constexpr int kKStages = D == 64 ? 4 : 3;
    static constexpr int kVStages = D == 64 ? 4 : 2;
    static constexpr int kOffQ = 0;                        // Q_A, Q_B
    static constexpr int kOffK = kOffQ + kStreams * kTileBytes;
    static constexpr int kOffV = kOffK + kKStages * kTileBytes;
    static constexpr int kOffBar = kOffV + kVStages * kTileBytes;
    static constexpr int kNumBars = 1 + 2 * kKStages + 2 * kVStages + 3 * kStreams + 1;
    static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;  // + TMEM slot, + alignment slack
    static constexpr uint32_t kTmemCols = 512;
};

__device__ __forceinline__ uint32_t col_s(int st) { return st == 0 ? 0u : 128u; }
__device__ __forceinline__ uint32_t col_o(int st) { return st == 0 ? 256u : 384u; }

struct DevFwd {
    int d, g, n_heads, n_outer, q_len, kv_len;
    int ring_i0, ring_t, ring_p, bsz, np;
    int kv_gathered;
    int zigzag, zz_kh;
    int split_np, split_b;  // > 0: read and write in place in the sequence-sharded layout (split_pos)
    int causal;
    float scale_log2;
    void* o_bf16;
    float* o_f32;
    int64_t o_s_head, o_s_tok, o_s_outer;
    float* lse;
    int64_t l_s_head, l_s_tok, l_s_outer;
    int* status;
};

// Where a work item sits: query rows, heads, outer indices and token offsets.
struct WorkItem {
    int r0;                // first query row (local token) of the 256-row block
    int head, kv_head;
    int q_outer, kv_outer;
    long q_pos0, kv_pos0;  // global positions of local token 0
    int n_tiles[kStreams]; // visible key tiles of each 128-row stream (0: nothing visible)
    int n_max;
};

__device__ __forceinline__ WorkItem decode_item(const DevFwd& p) {
    const int n_qb = (p.q_len + kStreams * kBM - 1) / (kStreams * kBM);
    const int per_block = p.n_heads * p.n_outer;
    const int item = blockIdx.x;
    WorkItem w;
    // heaviest (last) query blocks first: causal work grows with the position
    // group-major: all query blocks of one (outer index, KV head) group -- heaviest first, the
    // group's query heads adjacent -- before the next group, so that the K/V tiles being read at any
    // time belong to few KV heads and stay in L2
    (void)per_block;
    const int n_kvh = p.n_heads / p.g;
    const int per_group = n_qb * p.g;
    const int grp = item / per_group, within = item % per_group;
    const int qb = n_qb - 1 - within / p.g;
    w.head = (grp % n_kvh) * p.g + within % p.g;
    const int o = grp / n_kvh;
    w.kv_head = w.head / p.g;
    if (p.zigzag) {
        // zigzag: rank i holds chunks i and 2P-1-i; o -> (i, b, query half)
        const int i = p.ring_i0 + o / (2 * p.bsz), b = (o / 2) % p.bsz, qh = o & 1;
        const int j = ((i - p.ring_t) % p.ring_p + p.ring_p) % p.ring_p;
        w.q_outer = (i * p.bsz + b) * 2 + qh;
        w.kv_outer = (j * p.bsz + b) * 2 + p.zz_kh;
        w.q_pos0 = (long)(qh ? 2 * p.ring_p - 1 - i : i) * p.np;
        w.kv_pos0 = (long)(p.zz_kh ? 2 * p.ring_p - 1 - j : j) * p.np;
    } else {
        const int i = p.ring_i0 + o / p.bsz;
        const int b = o % p.bsz;
        const int j = ((i - p.ring_t) % p.ring_p + p.ring_p) % p.ring_p;
        w.q_outer = i * p.bsz + b;
        w.kv_outer = p.kv_gathered ? b : j * p.bsz + b;
        w.q_pos0 = (long)i * p.np;
        w.kv_pos0 = p.kv_gathered ? 0L : (long)j * p.np;
    }
    w.r0 = qb * kStreams * kBM;
    w.n_max = 0;
#pragma unroll
    for (int st = 0; st < kStreams; ++st) {
        const int r0 = w.r0 + st * kBM;
        int kv_end = r0 < p.q_len ? p.kv_len : 0;
        if (p.causal && r0 < p.q_len) {
            const long last_q = w.q_pos0 + min(r0 + kBM, p.q_len) - 1;  // position of the stream's last row
            const long vis = last_q - w.kv_pos0 + 1;                   // keys with position <= last_q
            kv_end = (int)max(0L, min((long)p.kv_len, vis));
        }
        w.n_tiles[st] = (kv_end + kBN - 1) / kBN;
        w.n_max = max(w.n_max, w.n_tiles[st]);
    }
    return w;
}

// SPLIT: the sequence-sharded in-place addressing (split_pos); compiled out otherwise
template <int D, bool OUT_F32, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const DevFwd p) {
    using C = FwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + C::kNumBars * 8);
    __shared__ int abort_flag;

    const uint32_t bar0 = sbase + C::kOffBar;
    auto BAR = [&](int idx) { return bar0 + 8u * (uint32_t)idx; };
    const int kQFull = 0;
    const int kKFull = 1, kKEmpty = kKFull + C::kKStages;
    const int kVFull = kKEmpty + C::kKStages, kVEmpty = kVFull + C::kVStages;
    const int kSFull = kVEmpty + C::kVStages;  // per stream
    const int kPReady = kSFull + kStreams;     // per stream
    const int kOReady = kPReady + kStreams;    // per stream
    const int kDrain = kOReady + kStreams;     // the MMA issuer's last commit

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const WorkItem w = decode_item(p);
    const int snp = SPLIT ? p.split_np : 0;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(BAR(kQFull), 1);
        for (int s = 0; s < C::kKStages; ++s) { mbar_init(BAR(kKFull + s), 1); mbar_init(BAR(kKEmpty + s), 1); }
        for (int s = 0; s < C::kVStages; ++s) { mbar_init(BAR(kVFull + s), 1); mbar_init(BAR(kVEmpty + s), 1); }
        for (int st = 0; st < kStreams; ++st) {
            mbar_init(BAR(kSFull + st), 1);
            mbar_init(BAR(kPReady + st), 4 * 32);
            mbar_init(BAR(kOReady + st), 1);
        }
        mbar_init(BAR(kDrain), 1);
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
    // Each role's code sits inside the branch that set its register budget (so that the compiler
    // gives it that budget); every warp of a warpgroup executes the same setmaxnreg.
    if (warp >= kSoftmaxWarps) {
        setmaxnreg_dec<kOtherRegs>();
    if (w.n_max > 0 && warp == kProducerWarp && lane == 0) {
        // ---------------------------------------------------------------- TMA producer
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        mbar_arrive_expect_tx(BAR(kQFull), kStreams * C::kTileBytes);
        for (int st = 0; st < kStreams; ++st) {
            const TokOuter a = split_pos(w.r0 + st * kBM, w.q_outer, snp, p.split_b);
            for (int c = 0; c < C::kChunks; ++c)
                tma_load_4d(sbase + C::kOffQ + st * C::kTileBytes + c * 16384, &tm_q, c * 64, w.head, a.tok, a.outer,
                            BAR(kQFull));
        }
        // coordinates of key tile j; in split mode they step through the shards (whole tiles per shard)
        TokOuter kv = {0, w.kv_outer};
        int nk = 0, nv = 0;  // K and V tiles whose loads were issued
        for (int j = 0; j < w.n_max; ++j) {
            const int ks = j % C::kKStages, vs = j % C::kVStages;
            if (j >= C::kKStages && !mbar_wait(BAR(kKEmpty + ks), ((j / C::kKStages) - 1) & 1, abort_p, 1, p.status))
                break;
            mbar_arrive_expect_tx(BAR(kKFull + ks), C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c)
                tma_load_4d(sbase + C::kOffK + ks * C::kTileBytes + c * 16384, &tm_k, c * 64, w.kv_head, kv.tok,
                            kv.outer, BAR(kKFull + ks));
            nk = j + 1;
            if (j >= C::kVStages && !mbar_wait(BAR(kVEmpty + vs), ((j / C::kVStages) - 1) & 1, abort_p, 2, p.status))
                break;
            mbar_arrive_expect_tx(BAR(kVFull + vs), C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c)
                tma_load_4d(sbase + C::kOffV + vs * C::kTileBytes + c * 16384, &tm_v, c * 64, w.kv_head, kv.tok,
                            kv.outer, BAR(kVFull + vs));
            nv = j + 1;
            kv.tok += kBN;
            if (SPLIT && kv.tok == p.split_np) {
                kv.tok = 0;
                kv.outer += p.split_b;
            }
        }
        // every issued load lands before the CTA can exit (after an abort, too)
        mbar_drain(BAR(kQFull), 0, 10, p.status);
        drain_ring(BAR(kKFull), C::kKStages, nk, 11, p.status);
        drain_ring(BAR(kVFull), C::kVStages, nv, 12, p.status);
    } else if (w.n_max > 0 && warp == kMmaWarp && lane == 0) {
        // ---------------------------------------------------------------- MMA issuer
        constexpr uint32_t kIdS = idesc_bf16(kBM, kBN, 0, 0);  // S = Q K^T, both K-major
        constexpr uint32_t kIdO = idesc_bf16(kBM, D, 0, 1);    // O += P V, V MN-major
        // descriptors built once; each k-step adds its offset (address field, 16-byte units)
        const uint64_t dq0[kStreams] = {sdesc_sw128(sbase + C::kOffQ, 16, 1024),
                                        sdesc_sw128(sbase + C::kOffQ + C::kTileBytes, 16, 1024)};
        auto issue_qk = [&](int st, int j) {
            const uint64_t dk0 = sdesc_sw128(sbase + C::kOffK + (j % C::kKStages) * C::kTileBytes, 16, 1024);
            const uint32_t dcol = tmem + col_s(st);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = ((kk / 4) * 16384 + (kk % 4) * 32) >> 4;
                mma_ss(dcol, dq0[st] + off, dk0 + off, kIdS, kk > 0);
            }
            mma_commit(BAR(kSFull + st));
        };
        bool ok = mbar_wait(BAR(kQFull), 0, abort_p, 4, p.status);
        ok = ok && mbar_wait(BAR(kKFull), 0, abort_p, 3, p.status);
        if (ok) {
            tc_fence_after();
            for (int st = 0; st < kStreams; ++st)
                if (w.n_tiles[st] > 0) issue_qk(st, 0);
            mma_commit(BAR(kKEmpty));
        }
        for (int j = 0; ok && j < w.n_max; ++j) {
            const int vs = j % C::kVStages;
            const int ks1 = (j + 1) % C::kKStages;
            if (!mbar_wait(BAR(kVFull + vs), (j / C::kVStages) & 1, abort_p, 6, p.status)) break;
            bool k_waited = false;
            const uint64_t dv0 = sdesc_sw128(sbase + C::kOffV + vs * C::kTileBytes, 16384, 1024);
            for (int st = 0; ok && st < kStreams; ++st) {
                if (j >= w.n_tiles[st]) continue;
                if (!mbar_wait(BAR(kPReady + st), j & 1, abort_p, 5, p.status)) { ok = false; break; }
                tc_fence_after();
                const uint32_t pcol = tmem + col_s(st);  // P_st over the first 64 columns of S_st
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    mma_ts(tmem + col_o(st), pcol + kk * 8, dv0 + (kk * 2048 >> 4), kIdO, (j > 0 || kk > 0) ? 1u : 0u);
                if (j + 1 < w.n_tiles[st]) {
                    if (!k_waited) {
                        if (!mbar_wait(BAR(kKFull + ks1), ((j + 1) / C::kKStages) & 1, abort_p, 3, p.status)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        k_waited = true;
                    }
                    issue_qk(st, j + 1);  // in issue order after PV_st(j), which read P_st from these columns
                } else {
                    mma_commit(BAR(kOReady + st));
                }
            }
            if (!ok) break;
            mma_commit(BAR(kVEmpty + vs));
            if (k_waited) mma_commit(BAR(kKEmpty + ks1));
        }
        // every issued MMA completes before TMEM is freed (after an abort, too)
        mma_commit(BAR(kDrain));
        mbar_drain(BAR(kDrain), 0, 13, p.status);
    }
    } else {
        setmaxnreg_inc<kSoftmaxRegs>();
        // ---------------------------------------------------------------- softmax warps
        const int quad = warp & 3;           // TMEM lane quadrant
        const int st = warp >> 2;            // stream
        const int row = quad * 32 + lane;    // query row within the stream's tile = TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        const int r0 = w.r0 + st * kBM;
        const int n_tiles = w.n_tiles[st];
        const long q_pos = w.q_pos0 + r0 + row;
        float m_run = -INFINITY;  // running max of scale*log2(e)*S over the row (log2 units)
        float l_run = 0.f;        // running sum of 2^(scaled S - m_run)
        bool ok = true;
        for (int j = 0; j < n_tiles; ++j) {
            if (!mbar_wait(BAR(kSFull + st), j & 1, abort_p, 7, p.status)) { ok = false; break; }
            tc_fence_after();
            const uint32_t scol = lane_base + col_s(st);
            uint32_t r0r[32], r1r[32], r2r[32], r3r[32];
            tmem_ld32(scol, r0r);
            tmem_ld32(scol + 32, r1r);
            tmem_ld32(scol + 64, r2r);
            tmem_ld32(scol + 96, r3r);
            tmem_wait_ld();
            float s[kBN];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                s[c] = __uint_as_float(r0r[c]);
                s[32 + c] = __uint_as_float(r1r[c]);
                s[64 + c] = __uint_as_float(r2r[c]);
                s[96 + c] = __uint_as_float(r3r[c]);
            }
            const long key0 = w.kv_pos0 + (long)j * kBN;
            const int kv_rem = p.kv_len - j * kBN;
            if ((p.causal && key0 + kBN - 1 > w.q_pos0 + r0) || kv_rem < kBN) {
                // last visible column of this row in this tile
                long lim = p.causal ? q_pos - key0 : (long)(kBN - 1);
                lim = min(lim, (long)kv_rem - 1);
                const int climit = (int)max(-1L, min(lim, (long)(kBN - 1)));
#pragma unroll
                for (int c = 0; c < kBN; ++c)
                    if (c > climit) s[c] = -INFINITY;
            }
            // row max as eight independent chains of three-input maxima
            float m8[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) m8[c] = s[c];
#pragma unroll
            for (int c = 8; c < kBN; c += 2) m8[(c / 2) & 7] = max3f(m8[(c / 2) & 7], s[c], s[c + 1]);
            float mx = max3f(max3f(m8[0], m8[1], m8[2]), max3f(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
            mx *= p.scale_log2;
            const float m_new = fmaxf(m_run, mx);
            const bool rescale = m_new > m_run + kRescaleThreshold;
            const float m_use = rescale ? m_new : m_run;
            const float alpha = rescale ? ex2_approx(m_run - m_new) : 1.f;
            const float msub = m_use == -INFINITY ? 0.f : m_use;
            // column pairs in packed float32: x = S scale log2(e) - m, P = 2^x, two running pair sums
            const float2 c2 = make_float2(p.scale_log2, p.scale_log2), nm2 = make_float2(-msub, -msub);
            float2 sum2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                uint32_t pk[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const float2 x = fma2(make_float2(s[h * 32 + 2 * c], s[h * 32 + 2 * c + 1]), c2, nm2);
                    const float2 pv = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                    sum2[c & 1] = add2(sum2[c & 1], pv);
                    pk[c] = pack_bf16(pv.x, pv.y);
                }
                tmem_st16(scol + h * 16, pk);  // P over S: this row's S is already in registers
            }
            l_run = l_run * alpha + ((sum2[0].x + sum2[0].y) + (sum2[1].x + sum2[1].y));
            if (__any_sync(0xffffffffu, rescale) && j > 0) {
                // PV of tiles < j completed before S_j was signalled: scale O in place (warp-uniform
                // branch for the collective TMEM access; rows that keep their max have alpha = 1)
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    const uint32_t oc = lane_base + col_o(st) + c * 32;
                    tmem_ld32(oc, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st32(oc, o);
                }
            }
            m_run = m_use;
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(BAR(kPReady + st));
        }
        // ---------------------------------------------------------------- epilogue
        if (ok && n_tiles > 0) ok = mbar_wait(BAR(kOReady + st), 0, abort_p, 9, p.status);
        if (ok) {
            tc_fence_after();
            const bool has = n_tiles > 0 && l_run > 0.f;
            const float inv = has ? 1.f / l_run : 0.f;
            const float lse_v = has ? (m_run + lg2_approx(l_run)) * kLn2 : -INFINITY;
            const bool valid = r0 + row < p.q_len;
            // the stream's 128 rows lie in one shard (split mode): split its first row once
            const TokOuter a = split_pos(r0, w.q_outer, snp, p.split_b);
            const int64_t obase =
                (int64_t)w.head * p.o_s_head + (int64_t)(a.tok + row) * p.o_s_tok + (int64_t)a.outer * p.o_s_outer;
            const int64_t lbase =
                (int64_t)w.head * p.l_s_head + (int64_t)(a.tok + row) * p.l_s_tok + (int64_t)a.outer * p.l_s_outer;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                if (n_tiles > 0) {
                    tmem_ld32(lane_base + col_o(st) + c * 32, o);
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
                p.lse[lbase] = lse_v;
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

template <int D, bool OUT_F32, bool SPLIT>
cudaError_t launch_fwd_t(const FwdParams& f, cudaStream_t stream) {
    using C = FwdCfg<D>;
    CUtensorMap tq, tk, tv;
    if (!make_tmap_bf16(&tq, f.q, D, kBM) || !make_tmap_bf16(&tk, f.k, D, kBN) || !make_tmap_bf16(&tv, f.v, D, kBN))
        return cudaErrorInvalidValue;
    DevFwd p;
    p.d = D;
    p.g = f.g;
    p.n_heads = f.n_heads;
    p.n_outer = f.n_outer;
    p.q_len = f.q_len;
    p.kv_len = f.kv_len;
    p.ring_i0 = f.ring_i0;
    p.kv_gathered = f.kv_gathered;
    p.zigzag = f.zigzag;
    p.zz_kh = f.zz_kh;
    p.split_np = f.split_np;
    p.split_b = f.split_b;
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
    auto kern = attn_fwd_kernel<D, OUT_F32, SPLIT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const long n_qb = (f.q_len + kStreams * kBM - 1) / (kStreams * kBM);
    const long items = n_qb * (long)f.n_heads * (long)f.n_outer;
    if (items == 0) return cudaSuccess;
    kern<<<(unsigned)items, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd_bf16(const FwdParams& f, cudaStream_t stream) {
    const bool f32 = f.o_f32 != nullptr;
    if (f.split_np > 0) {  // in place in the sequence-sharded layout: bf16 output only
        if (f32) return cudaErrorInvalidValue;
        if (f.d == 64) return launch_fwd_t<64, false, true>(f, stream);
        if (f.d == 128) return launch_fwd_t<128, false, true>(f, stream);
        return cudaErrorInvalidValue;
    }
    if (f.d == 64) return f32 ? launch_fwd_t<64, true, false>(f, stream) : launch_fwd_t<64, false, false>(f, stream);
    if (f.d == 128) return f32 ? launch_fwd_t<128, true, false>(f, stream) : launch_fwd_t<128, false, false>(f, stream);
    return cudaErrorInvalidValue;
}

}  // namespace usp

// Attention backward on sm_103a tensor cores (the backward pass of the code
// example on the "Context Parallelism" glossary page, ultralytics.com,
// "Praktische Anwendung und Kompromisse": out.float().square().mean()
// .backward(); here for any upstream gradient dO).
//
//   P_ij  = exp(S_ij - lse_i)            S_ij = scale Q_i . K_j (causal: j <= i)
//   D_i   = dO_i . O_i
//   dV_j  = sum_{h in group} sum_i P_ij dO_i
//   dS_ij = P_ij (dO_i . V_j - D_i)
//   dK_j  = scale sum_{h in group} sum_i dS_ij Q_i
//   dQ_i  = scale sum_j dS_ij K_j
//
// Two forms. usp_attn_bwd runs the one-pass form: pre (below, which also zeroes
// a float32 dQ accumulator), then one kernel per (KV head, 128-key tile) that
// computes S^T and dP^T once per block pair and produces dK, dV and the pair's
// dQ partial (dkdvq_kernel, whose comment gives its design), then dQ rounded to
// bf16.  usp_attn_bwd_deterministic runs the three-pass form, no atomics,
// bit-reproducible:
//  1. pre:  D_i and lse_i*log2(e) into a workspace padded to 128-row tiles
//           (padding rows: lse = +inf, so their P is exactly 0), and -lse_i/scale
//           and -D_i each as a sum of three bf16 numbers: one extra k-step of
//           the dK/dV products subtracts them (see pass 2).
//  2. dK/dV: one CTA per (KV head, 128-key tile).  It walks every query head
//           of the GQA group and every 128-row query step that sees its keys:
//             S^T  = K Q^T,  dP^T = V dO^T          (tcgen05, shared-memory operands)
//             P^T, dS^T on CUDA cores (thread = key row = TMEM lane), bf16 into TMEM
//             dV  += P^T dO, dK += dS^T Q           (A from TMEM, B MN-major)
//           dK and dV stay in TMEM for the whole walk.
//  3. dQ:   one CTA per (query head, 128-row tile) walking its visible key
//           tiles: S = Q K^T, dP = dO V^T (dO held in TMEM), dS on CUDA
//           cores into TMEM, dQ += dS K.
// An MMA overwrites TMEM columns that another MMA reads only when it is issued
// after that MMA (tcgen05.mma executes in issue order); the element-wise warps
// overwrite TMEM only after their own loads of it have completed, or after a
// barrier says the MMA that reads it is done.  Each kernel's comment gives its
// column plan.
#include <algorithm>
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"

namespace usp {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------------ pass 1
// -x as three bf16 numbers a0 + a1 + a2 (each the rounded remainder of the
// previous ones; together about 24 significant bits), packed as the 16-byte
// row [a0, a1, a2, 0, 0, 0, 0, 0] that the dK/dV products' extra k-step reads.
__device__ __forceinline__ float bf16_round(float x) { return __uint_as_float(pack_bf16(x, 0.f) << 16); }
__device__ __forceinline__ uint4 neg_split3(float x) {
    const float a0 = bf16_round(-x);
    const float r1 = -x - a0;
    const float a1 = bf16_round(r1);
    const float a2 = bf16_round(r1 - a1);
    return make_uint4(pack_bf16(a0, a1), pack_bf16(a2, 0.f), 0u, 0u);
}

struct PreArgs {
    const uint16_t* o;     // shaped and strided as q
    const uint16_t* dout;  // likewise
    const float* lse;
    int64_t s_head, s_tok, s_outer;        // o / dout strides (elements)
    int64_t l_s_head, l_s_tok, l_s_outer;  // lse strides
    int heads, N, Npad, n_z;
    int split_np, split_b;  // in place in the sequence-sharded layout (split_pos)
    float scale;
    float *dvec, *lse2;
    uint4 *xl, *xd;
    float* dq_acc;  // one-pass backward: the float32 dQ accumulator, zeroed here (null: left alone)
};

// One block per 128 padded rows z * Npad + n (z = outer * heads + head; Npad is a multiple of
// 128): dvec = dO . O (fp32), lse2 = lse * log2(e), the split rows of lse / scale (xl) and of dvec
// (xd), and one 128-row tile of the dQ accumulator (tile = block) set to zero. Each row's O and dO
// are read as D/8 16-byte pieces by D/8 consecutive threads; every thread issues all of its loads
// (two per row it covers) before it uses one, and the zero stores while they are in flight.
//
// Which (outer, head, position) the block's row L (0 .. n_z * Npad - 1) covers: in the head-sharded
// layout head-major (L = z * Npad + n, one block = 128 positions of one head), in the sequence-
// sharded layout (SPLIT) token-major (L = (outer * Npad + n) * heads + head), so that a block's rows
// are the heads of a few tokens, contiguous there.
template <bool SPLIT>
__device__ __forceinline__ void pre_row(const PreArgs& a, int64_t L, int& outer, int& head, int& n) {
    if constexpr (SPLIT) {
        const int64_t per_outer = (int64_t)a.Npad * a.heads;
        outer = (int)(L / per_outer);
        const int64_t rem = L - (int64_t)outer * per_outer;
        n = (int)(rem / a.heads);
        head = (int)(rem - (int64_t)n * a.heads);
    } else {
        const int z = (int)(L / a.Npad);
        n = (int)(L - (int64_t)z * a.Npad);
        outer = z / a.heads;
        head = z - outer * a.heads;
    }
}

template <int D, bool SPLIT>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const PreArgs a) {
    constexpr int kPieces = D / 8;             // 16-byte pieces per row: 16 or 8
    constexpr int kRowsPerPass = 256 / kPieces;  // 16 or 32
    constexpr int kPasses = 128 / kRowsPerPass;  // 8 or 4
    __shared__ float dot[128];
    const int64_t row0 = (int64_t)blockIdx.x * 128;
    const int piece = threadIdx.x % kPieces;
    const int sub = threadIdx.x / kPieces;
    const int N = a.N;
    uint4 ov[kPasses], dv[kPasses];
#pragma unroll
    for (int i = 0; i < kPasses; ++i) {
        int outer, head, n;
        pre_row<SPLIT>(a, row0 + i * kRowsPerPass + sub, outer, head, n);
        ov[i] = make_uint4(0u, 0u, 0u, 0u);
        dv[i] = ov[i];
        if (n < N) {
            const TokOuter at = split_pos(n, outer, SPLIT ? a.split_np : 0, a.split_b);
            const int64_t base =
                (int64_t)at.outer * a.s_outer + (int64_t)head * a.s_head + (int64_t)at.tok * a.s_tok + piece * 8;
            ov[i] = __ldg(reinterpret_cast<const uint4*>(a.o + base));
            dv[i] = __ldg(reinterpret_cast<const uint4*>(a.dout + base));
        }
    }
    if (a.dq_acc) {
        float4* t = reinterpret_cast<float4*>(a.dq_acc + row0 * D);
        const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int j = threadIdx.x; j < 128 * D / 4; j += 256) t[j] = zero;
    }
#pragma unroll
    for (int i = 0; i < kPasses; ++i) {
        const uint32_t* x = &ov[i].x;
        const uint32_t* y = &dv[i].x;
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e)
            acc += __uint_as_float(x[e] << 16) * __uint_as_float(y[e] << 16) +
                   __uint_as_float(x[e] & 0xFFFF0000u) * __uint_as_float(y[e] & 0xFFFF0000u);
#pragma unroll
        for (int off = kPieces / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (piece == 0) dot[i * kRowsPerPass + sub] = acc;
    }
    __syncthreads();
    if (threadIdx.x < 128) {
        const int r = threadIdx.x;
        int outer, head, n;
        pre_row<SPLIT>(a, row0 + r, outer, head, n);
        const int64_t row = ((int64_t)outer * a.heads + head) * a.Npad + n;  // the workspace row
        if (n >= N) {
            a.dvec[row] = 0.f;
            a.lse2[row] = INFINITY;
            a.xl[row] = make_uint4(0x0000FF7Fu, 0u, 0u, 0u);  // -(largest finite bf16): P underflows to 0
            a.xd[row] = make_uint4(0u, 0u, 0u, 0u);
        } else {
            const TokOuter at = split_pos(n, outer, SPLIT ? a.split_np : 0, a.split_b);
            const float l = a.lse[(int64_t)at.outer * a.l_s_outer + (int64_t)head * a.l_s_head + (int64_t)at.tok * a.l_s_tok];
            const float acc = dot[r];
            a.dvec[row] = acc;
            a.lse2[row] = l * kLog2e;
            a.xl[row] = neg_split3(l / a.scale);
            a.xd[row] = neg_split3(acc);
        }
    }
}

// ------------------------------------------------------------------ common
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
                 : "memory");
}

struct DevBwd {
    int Hq, g, N, Npad, causal;  // Hq: query heads per outer index; N: query tokens per block
    int Nkv;                     // key tokens per block
    int ring_i0, ring_t, ring_p, bsz, n_outer, kv_gathered;
    int zigzag, zz_kh, zz_qh;  // zigzag ring: KV half of the launch, fixed query half or -1
    int split_np, split_b;     // in place in the sequence-sharded layout (split_pos); N, Nkv global
    float scale, scale_log2;
    const float* lse2;  // [n_z][Npad], z = query outer * Hq + head
    const float* dvec;  // [n_z][Npad]
    const uint4* xl;    // [n_z][Npad]: -lse / scale as three bf16 (a 16-byte row)
    const uint4* xd;    // [n_z][Npad]: -D as three bf16
    const uint16_t* q;       // queries (pass 3 loads its tile into TMEM)
    const uint16_t* dout;    // upstream gradient, strided as q
    uint16_t *dq, *dk, *dv;  // bf16 results, or
    float *dq_f, *dk_f, *dv_f;  // float32 results (non-null), added to when acc != 0
    int acc;
    int64_t q_s_head, q_s_tok, q_s_outer;  // dq strides (elements)
    int64_t k_s_head, k_s_tok, k_s_outer;  // dk, dv strides
    int* status;
    float* dq_acc;  // one-pass backward: float32 dQ accumulator (BwdParams::dq_acc layout)
};

// Outer index o of a launch -> query outer (rank i, batch b), KV outer (rank
// j = (i - t) mod P and batch b; batch b alone when K/V are gathered) and the
// causal shift: the position of the query block's first token minus that of
// the key block's (query q sees key k, both block-local, iff q + shift >= k).
// The Ulysses path has one outer index, 0, and shift 0.
__device__ __forceinline__ void bwd_outer(const DevBwd& p, int o, int& q_outer, int& kv_outer, int& shift) {
    if (p.zigzag) {
        // zigzag: rank i holds chunks i and 2P-1-i of N tokens each (outer (i*bsz + b)*2 + half)
        int i, b, qh;
        if (p.zz_qh >= 0) {
            i = p.ring_i0 + o / p.bsz;
            b = o % p.bsz;
            qh = p.zz_qh;
        } else {
            i = p.ring_i0 + o / (2 * p.bsz);
            b = (o / 2) % p.bsz;
            qh = o & 1;
        }
        const int j = ((i - p.ring_t) % p.ring_p + p.ring_p) % p.ring_p;
        q_outer = (i * p.bsz + b) * 2 + qh;
        kv_outer = (j * p.bsz + b) * 2 + p.zz_kh;
        const int qc = qh ? 2 * p.ring_p - 1 - i : i, kc = p.zz_kh ? 2 * p.ring_p - 1 - j : j;
        shift = (qc - kc) * p.N;
        return;
    }
    const int i = p.ring_i0 + o / p.bsz, b = o % p.bsz;
    const int j = ((i - p.ring_t) % p.ring_p + p.ring_p) % p.ring_p;
    q_outer = i * p.bsz + b;
    kv_outer = p.kv_gathered ? b : j * p.bsz + b;
    shift = p.kv_gathered ? i * p.N : (i - j) * p.N;
}

// 32 consecutive values of one result row, times mul: a bf16 store, or a
// float32 store / accumulate.
__device__ __forceinline__ void store_row32(uint16_t* o16, float* o32, int acc, int64_t off, const uint32_t (&r)[32],
                                            float mul) {
    if (o32) {
        float4* dst = reinterpret_cast<float4*>(o32 + off);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float4 v = make_float4(__uint_as_float(r[4 * e]) * mul, __uint_as_float(r[4 * e + 1]) * mul,
                                   __uint_as_float(r[4 * e + 2]) * mul, __uint_as_float(r[4 * e + 3]) * mul);
            if (acc) {
                const float4 a = dst[e];
                v.x += a.x;
                v.y += a.y;
                v.z += a.z;
                v.w += a.w;
            }
            dst[e] = v;
        }
    } else {
        uint4* dst = reinterpret_cast<uint4*>(o16 + off);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            uint4 v;
            v.x = pack_bf16(__uint_as_float(r[8 * e + 0]) * mul, __uint_as_float(r[8 * e + 1]) * mul);
            v.y = pack_bf16(__uint_as_float(r[8 * e + 2]) * mul, __uint_as_float(r[8 * e + 3]) * mul);
            v.z = pack_bf16(__uint_as_float(r[8 * e + 4]) * mul, __uint_as_float(r[8 * e + 5]) * mul);
            v.w = pack_bf16(__uint_as_float(r[8 * e + 6]) * mul, __uint_as_float(r[8 * e + 7]) * mul);
            dst[e] = v;
        }
    }
}

// ------------------------------------------------------------------ pass 2: dK, dV
// One 128-key tile per CTA, walked over 128-row query steps, so that every
// product is a full 128 x 128 x 16 tcgen05.mma.  TMEM holds S^T, dP^T, dV and
// dK (128 columns each); P^T and dS^T (bf16) are written in place over the
// first half of each 64-column block of S^T and dP^T.  Per step the tensor
// core runs
//     S^T(i)  dP^T(i)  | dV(i)  S^T(i+1)  | dK(i)  dP^T(i+1) | dV(i+1) ...
// and the element-wise warps compute P(i) while dP^T(i) runs and dS(i)
// while dV(i) and S^T(i+1) run.  A product that overwrites S^T or dP^T is
// issued after the one that reads the bf16 operand stored there
// (tcgen05.mma executes in issue order).
// Eight element-wise warps: warp w owns TMEM lanes 32 (w % 4) .. + 31 (its
// key rows) and query columns 64 (w / 4) .. + 63 of each step.
// The per-query values lse and D reach the element-wise warps through the
// products rather than through per-element shared-memory loads: a ninth
// k-step with A = a 128 x 16 tile of rows [1, 1, 1, 0, ...] and B = the
// query rows of -lse/scale (resp. -D) split into three bf16 numbers leaves
//     S'^T  = K Q^T - lse/scale      dP'^T = V dO^T - D
// in TMEM, so that P = 2^(S' scale log2 e) and dS = P dP'.  Those small
// operands are K-major without swizzle; the second 16-byte half of their
// 32-byte rows (K = 16) is a shared block of zeros.
constexpr int kKvEwWarps = 8;
constexpr int kKvProducerWarp = 8;
constexpr int kKvMmaWarp = 9;
constexpr int kKvThreads = 10 * 32;

template <int D>
struct KvCfg {
    static constexpr int kBK = 128;  // keys per CTA (TMEM lanes)
    static constexpr int kBQ = 128;  // query rows per step
    static constexpr int kChunks = D / 64;
    static constexpr int kTile = kChunks * 128 * 128;  // one 128-row bf16 tile (K, V, Q or dO)
    static constexpr int kStages = 2;
    static constexpr int kXBytes = kBQ * 16;  // one 16-byte row per query: -lse/scale or -D as 3 bf16
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kTile;
    static constexpr int kOffQ = 2 * kTile;
    static constexpr int kOffDO = kOffQ + kStages * kTile;
    static constexpr int kOffX = kOffDO + kStages * kTile;  // per stage: lse rows, then D rows
    static constexpr int kOffOnes = kOffX + kStages * 2 * kXBytes;
    static constexpr int kOffZero = kOffOnes + kBK * 16;
    static constexpr int kOffBar = kOffZero + 2048;
    static constexpr int kNumBars = 1 + 2 * kStages + 6;
    static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;
    static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 384;
};

// SPLIT (this and dq_kernel): the sequence-sharded in-place addressing, compiled out otherwise
template <int D, bool SPLIT>
__global__ void __launch_bounds__(kKvThreads, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v, const DevBwd p) {
    using C = KvCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + C::kNumBars * 8);
    __shared__ int abort_flag;
    const uint32_t bar0 = sbase + C::kOffBar;
    auto BAR = [&](int idx) { return bar0 + 8u * (uint32_t)idx; };
    const int kKvFull = 0, kQFull = 1, kQEmpty = 1 + C::kStages, kSFull = 1 + 2 * C::kStages, kDPFull = kSFull + 1,
              kPReady = kSFull + 2, kDSReady = kSFull + 3, kOReady = kSFull + 4, kDrain = kSFull + 5;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int Hkv = p.Hq / p.g;
    // group-major: all key tiles of one (outer index, KV head) -- low key tiles first, they carry the
    // most causal work -- before the next, so that the CTAs in flight stream the same Q/dO tiles
    const int n_kt = (p.Nkv + C::kBK - 1) / C::kBK;
    const int grp = blockIdx.x / n_kt;
    const int kt = blockIdx.x % n_kt;
    const int hk = grp % Hkv;
    int q_outer, kv_outer, shift;
    bwd_outer(p, grp / Hkv, q_outer, kv_outer, shift);
    const int n_qt = (p.N + C::kBQ - 1) / C::kBQ;
    // causal: query steps before the one holding the first query that reaches key kt * kBK see none
    // of these keys
    const int first_q = kt * C::kBK - shift;
    const int qt_lo = (p.causal && first_q > 0) ? first_q / C::kBQ : 0;
    const int nq = max(0, n_qt - qt_lo);
    const int n_it = p.g * nq;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(BAR(kKvFull), 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(BAR(kQFull + s), 1);
            mbar_init(BAR(kQEmpty + s), 1);
        }
        mbar_init(BAR(kSFull), 1);
        mbar_init(BAR(kDPFull), 1);
        mbar_init(BAR(kPReady), kKvEwWarps * 32);
        mbar_init(BAR(kDSReady), kKvEwWarps * 32);
        mbar_init(BAR(kOReady), 1);
        mbar_init(BAR(kDrain), 1);
        fence_mbar_init();
    }
    if (warp == kKvMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    if (threadIdx.x < C::kBK) {
        // row t of the ones operand (bf16 1.0 = 0x3F80 in its first three columns) and 16 bytes of zeros
        *reinterpret_cast<uint4*>(smem + C::kOffOnes + threadIdx.x * 16) = make_uint4(0x3F803F80u, 0x3F80u, 0u, 0u);
        *reinterpret_cast<uint4*>(smem + C::kOffZero + threadIdx.x * 16) = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    volatile int* abort_p = &abort_flag;

    if (n_it > 0 && warp == kKvProducerWarp && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_do);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        mbar_arrive_expect_tx(BAR(kKvFull), 2 * C::kTile);
        const TokOuter kv = split_pos(kt * C::kBK, kv_outer, SPLIT ? p.split_np : 0, p.split_b);
        for (int c = 0; c < C::kChunks; ++c) {
            tma_load_4d(sbase + C::kOffK + c * 16384, &tm_k, c * 64, hk, kv.tok, kv.outer, BAR(kKvFull));
            tma_load_4d(sbase + C::kOffV + c * 16384, &tm_v, c * 64, hk, kv.tok, kv.outer, BAR(kKvFull));
        }
        TokOuter q_next = {0, 0};  // split mode: the next query tile's coordinates, stepped through the shards
        int issued = 0;            // query steps whose loads were issued
        for (int it = 0; it < n_it; ++it) {
            const int s = it % C::kStages;
            const int hq = hk * p.g + it / nq;
            const int qt = qt_lo + it % nq;
            if (it >= C::kStages &&
                !mbar_wait(BAR(kQEmpty + s), ((it / C::kStages) - 1) & 1, abort_p, 21, p.status))
                break;
            mbar_arrive_expect_tx(BAR(kQFull + s), 2 * C::kTile + 2 * C::kXBytes);
            TokOuter qa;
            if constexpr (SPLIT) {
                // one division per query head (the walk restarts at qt_lo), then whole tiles per shard
                if (it % nq == 0) q_next = split_pos(qt * C::kBQ, q_outer, p.split_np, p.split_b);
                qa = q_next;
                q_next.tok += C::kBQ;
                if (q_next.tok == p.split_np) {
                    q_next.tok = 0;
                    q_next.outer += p.split_b;
                }
            } else {
                qa = {qt * C::kBQ, q_outer};
            }
            for (int c = 0; c < C::kChunks; ++c) {
                tma_load_4d(sbase + C::kOffQ + s * C::kTile + c * 16384, &tm_q, c * 64, hq, qa.tok, qa.outer,
                            BAR(kQFull + s));
                tma_load_4d(sbase + C::kOffDO + s * C::kTile + c * 16384, &tm_do, c * 64, hq, qa.tok, qa.outer,
                            BAR(kQFull + s));
            }
            const int64_t voff = ((int64_t)q_outer * p.Hq + hq) * p.Npad + (int64_t)qt * C::kBQ;
            bulk_load(sbase + C::kOffX + s * 2 * C::kXBytes, p.xl + voff, C::kXBytes, BAR(kQFull + s));
            bulk_load(sbase + C::kOffX + s * 2 * C::kXBytes + C::kXBytes, p.xd + voff, C::kXBytes, BAR(kQFull + s));
            issued = it + 1;
        }
        // every issued load lands before the CTA can exit (after an abort, too)
        mbar_drain(BAR(kKvFull), 0, 40, p.status);
        drain_ring(BAR(kQFull), C::kStages, issued, 41, p.status);
    } else if (n_it > 0 && warp == kKvMmaWarp && lane == 0) {
        constexpr uint32_t kIdS = idesc_bf16(C::kBK, C::kBQ, 0, 0);  // S^T = K Q^T, dP^T = V dO^T
        constexpr uint32_t kIdG = idesc_bf16(C::kBK, D, 0, 1);       // dV += P^T dO, dK += dS^T Q
        // descriptors built once; each k-step adds its offset (address field, 16-byte units)
        const uint64_t dk0 = sdesc_sw128(sbase + C::kOffK, 16, 1024), dv0 = sdesc_sw128(sbase + C::kOffV, 16, 1024);
        // the extra k-step's operands: rows of ones (A) and the stage's split rows (B); 8-row
        // groups 128 bytes apart, the zero half of every row at the shared zero block
        auto plain = [&](int off) {
            return sdesc_plain(sbase + off, (uint32_t)(C::kOffZero - off), 128);
        };
        const uint64_t dones = plain(C::kOffOnes);
        // S'^T (A = K, x = 0: lse rows) or dP'^T (A = V, x = 1: D rows) of step it: B = Q or dO of
        // its stage, both K-major
        auto issue_t = [&](int it, uint64_t a0, int off_b, uint32_t col, int x) {
            const int s = it % C::kStages;
            const uint64_t b0 = sdesc_sw128(sbase + off_b + s * C::kTile, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = ((kk / 4) * 16384 + (kk % 4) * 32) >> 4;
                mma_ss(tmem + col, a0 + off, b0 + off, kIdS, kk > 0);
            }
            mma_ss(tmem + col, dones, plain(C::kOffX + (2 * s + x) * C::kXBytes), kIdS, 1u);
        };
        // dV (A = P^T) or dK (A = dS^T) of step it: A from TMEM, B = dO or Q MN-major
        auto issue_g = [&](int it, uint32_t col_a, int off_b, uint32_t col_d) {
            const uint64_t b0 = sdesc_sw128(sbase + off_b + (it % C::kStages) * C::kTile, 16384, 1024);
#pragma unroll
            for (int kk = 0; kk < C::kBQ / 16; ++kk) {
                // queries 16 kk .. + 15 sit in the bf16 half of 64-column block kk / 4
                const uint32_t a = tmem + col_a + (kk / 4) * 64 + (kk % 4) * 8;
                mma_ts(tmem + col_d, a, b0 + (kk * 2048 >> 4), kIdG, (it > 0 || kk > 0) ? 1u : 0u);
            }
        };
        bool ok = mbar_wait(BAR(kKvFull), 0, abort_p, 23, p.status);
        ok = ok && mbar_wait(BAR(kQFull), 0, abort_p, 22, p.status);
        if (ok) {
            tc_fence_after();
            issue_t(0, dk0, C::kOffQ, C::kColS, 0);
            mma_commit(BAR(kSFull));
            issue_t(0, dv0, C::kOffDO, C::kColDP, 1);
            mma_commit(BAR(kDPFull));
        }
        for (int it = 0; ok && it < n_it; ++it) {
            const bool more = it + 1 < n_it;
            if (!mbar_wait(BAR(kPReady), it & 1, abort_p, 25, p.status)) break;
            tc_fence_after();
            issue_g(it, C::kColS, C::kOffDO, C::kColDV);
            if (more) {
                if (!mbar_wait(BAR(kQFull + (it + 1) % C::kStages), ((it + 1) / C::kStages) & 1, abort_p, 22,
                               p.status))
                    break;
                tc_fence_after();
                issue_t(it + 1, dk0, C::kOffQ, C::kColS, 0);  // after dV(it), which read P^T from these columns
                mma_commit(BAR(kSFull));
            }
            if (!mbar_wait(BAR(kDSReady), it & 1, abort_p, 24, p.status)) break;
            tc_fence_after();
            issue_g(it, C::kColDP, C::kOffQ, C::kColDK);
            mma_commit(BAR(kQEmpty + it % C::kStages));
            if (more) {
                issue_t(it + 1, dv0, C::kOffDO, C::kColDP, 1);  // after dK(it), which read dS^T from these columns
                mma_commit(BAR(kDPFull));
            } else {
                mma_commit(BAR(kOReady));
            }
        }
        // every issued MMA completes before TMEM is freed (after an abort, too)
        mma_commit(BAR(kDrain));
        mbar_drain(BAR(kDrain), 0, 42, p.status);
    } else if (warp < kKvEwWarps) {
        // ---------------------------------------------------------------- element-wise warps
        const int quad = warp & 3, half = warp >> 2;
        const int key = kt * C::kBK + quad * 32 + lane;  // key row = TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        const uint32_t col_s = C::kColS + half * 64, col_dp = C::kColDP + half * 64;
        bool ok = true;
        for (int it = 0; it < n_it; ++it) {
            const int qt = qt_lo + it % nq;
            // ---- P = exp2(S * scale * log2(e) - lse * log2(e)) on this warp's 64 query columns
            if (!mbar_wait(BAR(kSFull), it & 1, abort_p, 26, p.status)) { ok = false; break; }
            tc_fence_after();
            uint32_t ra[32], rb[32];
            tmem_ld32(lane_base + col_s, ra);
            tmem_ld32(lane_base + col_s + 32, rb);
            tmem_wait_ld();
            const int q0 = qt * C::kBQ + half * 64;  // query of column 0
            const bool need_mask = p.causal && q0 + shift < kt * C::kBK + C::kBK - 1;
            const int qmin_ok = key - shift - q0;  // columns e with q0 + e + shift >= key are visible
            float pf[64];
            uint32_t pk[32];
            const float2 c2 = make_float2(p.scale_log2, p.scale_log2);
#pragma unroll
            for (int e = 0; e < 64; e += 2) {
                // S' already holds S - lse / scale: P = 2^(S' scale log2 e), column pairs in packed float32
                const float2 x = mul2(make_float2(__uint_as_float(e < 32 ? ra[e] : rb[e - 32]),
                                                  __uint_as_float(e < 32 ? ra[e + 1] : rb[e - 31])),
                                      c2);
                pf[e] = ex2_approx(x.x);
                pf[e + 1] = ex2_approx(x.y);
                if (need_mask) {
                    if (e < qmin_ok) pf[e] = 0.f;
                    if (e + 1 < qmin_ok) pf[e + 1] = 0.f;
                }
                pk[e / 2] = pack_bf16(pf[e], pf[e + 1]);
            }
            tmem_st32(lane_base + col_s, pk);  // P^T over the first 32 of this warp's S^T columns
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(BAR(kPReady));
            // ---- dS = P (dP - D)
            if (!mbar_wait(BAR(kDPFull), it & 1, abort_p, 28, p.status)) { ok = false; break; }
            tc_fence_after();
            tmem_ld32(lane_base + col_dp, ra);
            tmem_ld32(lane_base + col_dp + 32, rb);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 64; e += 2) {
                // dP' already holds dP - D
                const float2 ds = mul2(make_float2(pf[e], pf[e + 1]),
                                       make_float2(__uint_as_float(e < 32 ? ra[e] : rb[e - 32]),
                                                   __uint_as_float(e < 32 ? ra[e + 1] : rb[e - 31])));
                pk[e / 2] = pack_bf16(ds.x, ds.y);
            }
            tmem_st32(lane_base + col_dp, pk);  // dS^T over the first 32 of this warp's dP^T columns
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(BAR(kDSReady));
        }
        if (ok && n_it > 0) ok = mbar_wait(BAR(kOReady), 0, abort_p, 29, p.status);
        if (ok) {
            // warps 0-3 write dV, warps 4-7 write dK (scale applied here)
            tc_fence_after();
            const bool valid = key < p.Nkv;
            const TokOuter ka = split_pos(key, kv_outer, SPLIT ? p.split_np : 0, p.split_b);
            const int64_t base = (int64_t)ka.outer * p.k_s_outer + (int64_t)hk * p.k_s_head + (int64_t)ka.tok * p.k_s_tok;
            const uint32_t col = half == 0 ? C::kColDV : C::kColDK;
            const float mul = half == 0 ? 1.f : p.scale;
            uint16_t* out16 = half == 0 ? p.dv : p.dk;
            float* out32 = half == 0 ? p.dv_f : p.dk_f;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t r[32];
                if (n_it > 0) {
                    tmem_ld32(lane_base + col + cc * 32, r);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) r[e] = 0u;
                }
                if (valid) store_row32(out16, out32, p.acc, base + cc * 32, r, mul);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kKvMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ pass 3: dQ
// One CTA per (query head, 128-row query tile), walking its visible key
// tiles.  Q and dO are constant for the CTA: they live in TMEM (loaded once
// by the element-wise warps) as the A operands of S = Q K^T and dP = dO V^T,
// so the shared memory holds only the K and V rings.  K is the deeper ring:
// a K tile serves S(j) and, a step later, dQ(j).
// TMEM: S, dP (128 columns each), Q and dO (bf16, D/2 columns each), dQ (D).
// dS (bf16) is written in place over the first half of each warp's 64-column
// block of dP.  Per step the tensor core runs
//     S(j+1) | dQ(j)  dP(j+1) | S(j+2) ...
// and the element-wise warps compute P(j+1) from S(j+1) while dQ(j) and
// dP(j+1) run, then dS(j+1) while S(j+2) runs.  dP(j+1) overwrites the
// columns dQ(j) reads, so it is issued after dQ(j) (tcgen05.mma executes in
// issue order).
// Eight element-wise warps: warp w owns TMEM lanes 32 (w % 4) .. + 31 (its
// query rows) and key columns 64 (w / 4) .. + 63 of each step, so two warps
// share each sub-partition and hide each other's latency.
constexpr int kDqEwWarps = 8;
constexpr int kDqProducerWarp = 8;
constexpr int kDqMmaWarp = 9;
constexpr int kDqThreads = 10 * 32;

template <int D>
struct DqCfg {
    static constexpr int kBM = 128;  // query rows per CTA (TMEM lanes)
    static constexpr int kBN = 128;  // keys per step
    static constexpr int kChunks = D / 64;
    static constexpr int kTile = kChunks * 128 * 128;
    static constexpr int kKStages = D == 64 ? 8 : 5;
    static constexpr int kVStages = D == 64 ? 4 : 2;
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kKStages * kTile;
    static constexpr int kOffBar = kOffV + kVStages * kTile;
    static constexpr int kNumBars = 2 * kKStages + 2 * kVStages + 7;
    static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;
    static constexpr uint32_t kColS = 0, kColDP = 128, kColQ = 256, kColDO = 256 + D / 2, kColDQ = 384;
};

// One 128-row operand (Q or dO) of this CTA into TMEM as packed bf16: thread
// (lane quadrant, half) stores its row's values half * D/2 .. + D/2 - 1, zeros
// past the last row.
template <int D>
__device__ __forceinline__ void rows_to_tmem(const uint16_t* base, bool valid, uint32_t taddr) {
    constexpr int kW = D / 4;  // 32-bit words
    uint32_t w[kW];
    if (valid) {
        const uint4* src = reinterpret_cast<const uint4*>(base);
#pragma unroll
        for (int e = 0; e < kW / 4; ++e) {
            const uint4 v = src[e];
            w[4 * e] = v.x;
            w[4 * e + 1] = v.y;
            w[4 * e + 2] = v.z;
            w[4 * e + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int e = 0; e < kW; ++e) w[e] = 0u;
    }
    if constexpr (kW == 32) {
        tmem_st32(taddr, w);
    } else {
        tmem_st16(taddr, w);
    }
}

template <int D, bool SPLIT>
__global__ void __launch_bounds__(kDqThreads, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v, const DevBwd p) {
    using C = DqCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + C::kNumBars * 8);
    __shared__ int abort_flag;
    const uint32_t bar0 = sbase + C::kOffBar;
    auto BAR = [&](int idx) { return bar0 + 8u * (uint32_t)idx; };
    const int kKFull = 0, kKEmpty = C::kKStages, kVFull = 2 * C::kKStages, kVEmpty = kVFull + C::kVStages,
              kSFull = kVEmpty + C::kVStages, kSFree = kSFull + 1, kDPFull = kSFull + 2, kDsReady = kSFull + 3,
              kQdoReady = kSFull + 4, kOReady = kSFull + 5, kDrain = kSFull + 6;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int n_qt = (p.N + C::kBM - 1) / C::kBM;
    // group-major: all query tiles of one (outer index, KV head) group -- heaviest first, the group's
    // query heads adjacent -- before the next group, so that the K/V tiles in flight stay in L2
    const int n_kvh = p.Hq / p.g;
    const int per_group = n_qt * p.g;
    const int grp = (int)(blockIdx.x / per_group), within = (int)(blockIdx.x % per_group);
    const int qt = n_qt - 1 - within / p.g;
    const int hq = (grp % n_kvh) * p.g + within % p.g;
    const int hk = hq / p.g;
    int q_outer, kv_outer, shift;
    bwd_outer(p, grp / n_kvh, q_outer, kv_outer, shift);
    // causal: keys up to the position of the tile's last query
    const int kv_end = p.causal ? max(0, min(p.Nkv, min(p.N, (qt + 1) * C::kBM) + shift)) : p.Nkv;
    const int n_it = (kv_end + C::kBN - 1) / C::kBN;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < C::kKStages; ++s) {
            mbar_init(BAR(kKFull + s), 1);
            mbar_init(BAR(kKEmpty + s), 1);
        }
        for (int s = 0; s < C::kVStages; ++s) {
            mbar_init(BAR(kVFull + s), 1);
            mbar_init(BAR(kVEmpty + s), 1);
        }
        mbar_init(BAR(kSFull), 1);
        mbar_init(BAR(kSFree), kDqEwWarps * 32);
        mbar_init(BAR(kDPFull), 1);
        mbar_init(BAR(kDsReady), kDqEwWarps * 32);
        mbar_init(BAR(kQdoReady), kDqEwWarps * 32);
        mbar_init(BAR(kOReady), 1);
        mbar_init(BAR(kDrain), 1);
        fence_mbar_init();
    }
    if (warp == kDqMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    volatile int* abort_p = &abort_flag;

    if (n_it > 0 && warp == kDqProducerWarp && lane == 0) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        int nk = 0, nv = 0;  // K and V tiles whose loads were issued
        for (int j = 0; j < n_it; ++j) {
            const int ks = j % C::kKStages, vs = j % C::kVStages;
            if (j >= C::kKStages &&
                !mbar_wait(BAR(kKEmpty + ks), ((j / C::kKStages) - 1) & 1, abort_p, 31, p.status))
                break;
            const TokOuter kv = split_pos(j * C::kBN, kv_outer, SPLIT ? p.split_np : 0, p.split_b);
            mbar_arrive_expect_tx(BAR(kKFull + ks), C::kTile);
            for (int c = 0; c < C::kChunks; ++c)
                tma_load_4d(sbase + C::kOffK + ks * C::kTile + c * 16384, &tm_k, c * 64, hk, kv.tok, kv.outer,
                            BAR(kKFull + ks));
            nk = j + 1;
            if (j >= C::kVStages &&
                !mbar_wait(BAR(kVEmpty + vs), ((j / C::kVStages) - 1) & 1, abort_p, 38, p.status))
                break;
            mbar_arrive_expect_tx(BAR(kVFull + vs), C::kTile);
            for (int c = 0; c < C::kChunks; ++c)
                tma_load_4d(sbase + C::kOffV + vs * C::kTile + c * 16384, &tm_v, c * 64, hk, kv.tok, kv.outer,
                            BAR(kVFull + vs));
            nv = j + 1;
        }
        // every issued load lands before the CTA can exit (after an abort, too)
        drain_ring(BAR(kKFull), C::kKStages, nk, 43, p.status);
        drain_ring(BAR(kVFull), C::kVStages, nv, 44, p.status);
    } else if (n_it > 0 && warp == kDqMmaWarp && lane == 0) {
        constexpr uint32_t kIdS = idesc_bf16(C::kBM, C::kBN, 0, 0);  // S = Q K^T, dP = dO V^T (B K-major)
        constexpr uint32_t kIdG = idesc_bf16(C::kBM, D, 0, 1);       // dQ += dS K, K MN-major
        // S(j) = Q K_j^T: A = Q from TMEM (16 values = 8 columns per k-step), B = K_j
        auto issue_s = [&](int j) -> bool {
            const int ks = j % C::kKStages;
            if (!mbar_wait(BAR(kKFull + ks), (j / C::kKStages) & 1, abort_p, 32, p.status)) return false;
            tc_fence_after();
            const uint64_t dk0 = sdesc_sw128(sbase + C::kOffK + ks * C::kTile, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = ((kk / 4) * 16384 + (kk % 4) * 32) >> 4;
                mma_ts(tmem + C::kColS, tmem + C::kColQ + kk * 8, dk0 + off, kIdS, kk > 0);
            }
            mma_commit(BAR(kSFull));
            return true;
        };
        // dP(j) = dO V_j^T: A = dO from TMEM, B = V_j
        auto issue_dp = [&](int j) -> bool {
            const int vs = j % C::kVStages;
            if (!mbar_wait(BAR(kVFull + vs), (j / C::kVStages) & 1, abort_p, 39, p.status)) return false;
            tc_fence_after();
            const uint64_t dv0 = sdesc_sw128(sbase + C::kOffV + vs * C::kTile, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = ((kk / 4) * 16384 + (kk % 4) * 32) >> 4;
                mma_ts(tmem + C::kColDP, tmem + C::kColDO + kk * 8, dv0 + off, kIdS, kk > 0);
            }
            mma_commit(BAR(kDPFull));
            mma_commit(BAR(kVEmpty + vs));  // V_j is no longer needed once dP_j is done
            return true;
        };
        bool ok = mbar_wait(BAR(kQdoReady), 0, abort_p, 33, p.status);
        if (ok) tc_fence_after();
        ok = ok && issue_s(0) && issue_dp(0);
        for (int j = 0; ok && j < n_it; ++j) {
            const int ks = j % C::kKStages;
            const bool more = j + 1 < n_it;
            if (more) {
                // S(j+1) overwrites S(j): after the element-wise warps have loaded it
                if (!mbar_wait(BAR(kSFree), j & 1, abort_p, 34, p.status)) break;
                if (!issue_s(j + 1)) break;
            }
            if (!mbar_wait(BAR(kDsReady), j & 1, abort_p, 35, p.status)) break;
            tc_fence_after();
            const uint64_t bk = sdesc_sw128(sbase + C::kOffK + ks * C::kTile, 16384, 1024);
#pragma unroll
            for (int kk = 0; kk < C::kBN / 16; ++kk) {
                // keys 16 kk .. + 15: the bf16 half of dP's 64-column block kk / 4
                const uint32_t a = tmem + C::kColDP + (kk / 4) * 64 + (kk % 4) * 8;
                mma_ts(tmem + C::kColDQ, a, bk + (kk * 2048 >> 4), kIdG, (j > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(BAR(kKEmpty + ks));
            if (more) {
                if (!issue_dp(j + 1)) break;  // after dQ(j), which read dS from these columns
            } else {
                mma_commit(BAR(kOReady));
            }
        }
        // every issued MMA completes before TMEM is freed (after an abort, too)
        mma_commit(BAR(kDrain));
        mbar_drain(BAR(kDrain), 0, 45, p.status);
    } else if (warp < kDqEwWarps) {
        const int quad = warp & 3, half = warp >> 2;
        const int r = quad * 32 + lane;  // query row within the tile = TMEM lane
        const int q = qt * C::kBM + r;
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        const int64_t vrow = ((int64_t)q_outer * p.Hq + hq) * p.Npad + q;  // q < Npad always
        const TokOuter qa = split_pos(q, q_outer, SPLIT ? p.split_np : 0, p.split_b);
        const float lse2_r = p.lse2[vrow];
        const float dv_r = p.dvec[vrow];
        if (n_it > 0) {
            // this row's Q and dO (values half * D/2 .. + D/2 - 1) into TMEM
            const int64_t row = (int64_t)qa.outer * p.q_s_outer + (int64_t)hq * p.q_s_head + (int64_t)qa.tok * p.q_s_tok +
                                half * (D / 2);
            rows_to_tmem<D>(p.q + row, q < p.N, lane_base + C::kColQ + half * (D / 4));
            rows_to_tmem<D>(p.dout + row, q < p.N, lane_base + C::kColDO + half * (D / 4));
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(BAR(kQdoReady));
        }
        const uint32_t col_s = C::kColS + half * 64, col_dp = C::kColDP + half * 64;
        bool ok = true;
        for (int j = 0; j < n_it; ++j) {
            // ---- P = exp2(S * scale * log2(e) - lse * log2(e)) on this warp's 64 key columns
            if (!mbar_wait(BAR(kSFull), j & 1, abort_p, 36, p.status)) { ok = false; break; }
            tc_fence_after();
            uint32_t ra[32], rb[32];
            tmem_ld32(lane_base + col_s, ra);
            tmem_ld32(lane_base + col_s + 32, rb);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(BAR(kSFree));  // S(j) is in registers: S(j+1) may overwrite it
            const int key0 = j * C::kBN + half * 64;  // key of this warp's column 0
            // visible columns: key0 + c <= q (causal, block-local plus shift) and key0 + c < Nkv
            int climit = p.Nkv - 1 - key0;
            if (p.causal) climit = min(climit, q + shift - key0);
            const bool need_mask = climit < 63;
            float pf[64];
            const float2 c2 = make_float2(p.scale_log2, p.scale_log2);
            const float2 nl2 = make_float2(-lse2_r, -lse2_r);
#pragma unroll
            for (int e = 0; e < 64; e += 2) {
                const float2 x = fma2(make_float2(__uint_as_float(e < 32 ? ra[e] : rb[e - 32]),
                                                  __uint_as_float(e < 32 ? ra[e + 1] : rb[e - 31])),
                                      c2, nl2);
                pf[e] = ex2_approx(x.x);
                pf[e + 1] = ex2_approx(x.y);
                if (need_mask) {
                    if (e > climit) pf[e] = 0.f;
                    if (e + 1 > climit) pf[e + 1] = 0.f;
                }
            }
            // ---- dS = P (dP - D), bf16, over the first 32 of this warp's dP columns
            if (!mbar_wait(BAR(kDPFull), j & 1, abort_p, 28, p.status)) { ok = false; break; }
            tc_fence_after();
            tmem_ld32(lane_base + col_dp, ra);
            tmem_ld32(lane_base + col_dp + 32, rb);
            tmem_wait_ld();
            const float2 nd2 = make_float2(-dv_r, -dv_r);
            uint32_t dsp[32];
#pragma unroll
            for (int e = 0; e < 64; e += 2) {
                const float2 dp = make_float2(__uint_as_float(e < 32 ? ra[e] : rb[e - 32]),
                                              __uint_as_float(e < 32 ? ra[e + 1] : rb[e - 31]));
                const float2 ds = mul2(make_float2(pf[e], pf[e + 1]), add2(dp, nd2));
                dsp[e / 2] = pack_bf16(ds.x, ds.y);
            }
            tmem_st32(lane_base + col_dp, dsp);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(BAR(kDsReady));
        }
        if (ok && n_it > 0) ok = mbar_wait(BAR(kOReady), 0, abort_p, 37, p.status);
        if (ok) {
            // each warp writes half of the row's dQ columns
            tc_fence_after();
            const bool valid = q < p.N;
            const int64_t base =
                (int64_t)qa.outer * p.q_s_outer + (int64_t)hq * p.q_s_head + (int64_t)qa.tok * p.q_s_tok + half * (D / 2);
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) {
                uint32_t rr[32];
                if (n_it > 0) {
                    tmem_ld32(lane_base + C::kColDQ + half * (D / 2) + cc * 32, rr);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) rr[e] = 0u;
                }
                if (valid) store_row32(p.dq, p.dq_f, p.acc, base + cc * 32, rr, p.scale);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kDqMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}


// ------------------------------------------------------------------ one pass: dK, dV and dQ
// The dK/dV walk of pass 2 with the dQ product added, so that S and dP are
// computed (and their exponentials taken) once per visible block pair: five
// 128 x 128 products per step (S^T, dP^T, dV, dK, dQ) instead of the four of
// pass 2 plus the three of pass 3.
//   dQ_i (+)= dS_i K   over this CTA's 128 keys is a partial of dQ_i; it is
//   added in float32 into the workspace accumulator with red.global.add.v4
//   (the CTAs of the other key tiles add theirs; the order of the additions
//   varies from run to run, so dQ is not bit-reproducible, unlike dK and dV,
//   which stay in TMEM for the whole walk).
// dS^T (bf16) goes over the first half of each 64-column block of dP^T in
// TMEM, the A operand of dK += dS^T Q, and to shared memory, where its bytes
// read M-major are the A operand of dQ = dS K.  At d = 128 the shared copy is
// written over the dO tile of its own step once dV, the last product reading
// that tile, is done (no room for a buffer of its own).
// TMEM: S^T (P^T in place, bf16), dP^T (dS^T in place), dV, dK; at d = 128 dQ(i)
// lands in the dP^T columns after dK(i) has read dS^T(i) there, and dP^T(i+1) is
// issued after the reducers have drained dQ(i) (at d = 64 dQ has columns of its
// own, and only dQ(i+1) waits for that).  Per step the tensor core runs
//     dK(i)  dQ(i)  | dP^T(i+1)  dV(i+1)  S^T(i+2) | dK(i+1) ...
// and the element-wise warps compute P(i+1) while dK(i) and dQ(i) run and
// dS(i+1) while dV(i+1) runs; the reducer warps drain dQ(i) from TMEM right
// after dQ(i), then add it into the accumulator.  Q tiles
// are released after dK, dO tiles (with dS^T) after dQ, so the next Q tile
// loads while dQ and dV run.  The lse / D rows enter S^T and dP^T as the
// ninth k-step of pass 2.
// Sixteen warps in four warpgroups: 0 and 1 element-wise (P, dS), 2 the TMA producer (warp 8) and
// the MMA issuer (warp 9), 3 the dQ reducers (warp w drains the TMEM lanes 32 (w % 4) .. + 31 of
// dQ and adds them into the accumulator).  The reductions are throttled by the L2's atomic rate
// (about 22 bytes per clock per SM against 64 KiB per step): on warps of their own they stall
// only themselves, not the computation of P and dS.  Registers per thread after the set-up (the
// launch gives 128, 65536 / 512): warpgroup 2 keeps KqCfg::kOtherRegs, the reducers take
// kRedRegs (each holds its 32 rows' d values of dQ) and the two element-wise warpgroups kEwRegs.
constexpr int kKqEwWarps = 8;
constexpr int kKqProducerWarp = 8;
constexpr int kKqMmaWarp = 9;
constexpr int kKqRedWarp0 = 12;
constexpr int kKqThreads = 16 * 32;
constexpr int kKqLaunchRegs = 65536 / kKqThreads;

template <int D>
struct KqCfg {
    static constexpr int kBK = 128;  // keys per CTA (TMEM lanes of S^T, dP^T, dV, dK)
    static constexpr int kBQ = 128;  // query rows per step (TMEM lanes of dQ)
    static constexpr int kChunks = D / 64;
    static constexpr int kTile = kChunks * 128 * 128;   // one 128-row bf16 tile (K, V, Q or dO)
    static constexpr int kDsBytes = 128 * 128 * 2;     // dS^T: 128 keys x 128 queries, bf16
    static constexpr bool kDsInDo = kTile == kDsBytes;  // d = 128: dS^T over its step's dO tile
    static constexpr int kStages = 2;
    static constexpr int kXBytes = kBQ * 16;
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kTile;
    static constexpr int kOffQ = 2 * kTile;
    static constexpr int kOffDO = kOffQ + kStages * kTile;
    static constexpr int kOffDS = kOffDO + kStages * kTile;             // d = 64: dS^T's own buffer
    // dQ's column groups (4 columns of 128 rows each) reach the accumulator two ways: the last
    // kRedGroups by red.global from the reducers' registers (through the SM's L1TEX unit, which the
    // tensor core's operand reads also use), the others staged in shared memory and reduced by the
    // TMA engine (which costs shared-memory bandwidth twice): splitting the traffic loads both paths
    static constexpr int kGroups = D / 4;
    static constexpr int kRedGroups = D == 128 ? 16 : 0;  // measured: 274 ms at d = 128 (0 or 32: 294, 311); none at d = 64
    static constexpr bool kRedFirst = false;
    // the staging buffer, up to 16 column groups (32 KiB) per round: at d = 128 the dO tile of the
    // step (dS^T's shared copy, free once dQ is done), at d = 64 kStageBufs buffers of their own used
    // in turn, each waited for (its bulk reduction's read) only when the reducers next fill it.
    // Measured at 128K, d = 64: one buffer 204.3 ms, two 206.4 ms, one with a third Q/dO stage
    // 206.5 ms.
    static constexpr int kStageBytes = 128 * 64 * 4;
    static constexpr int kStageBufs = kDsInDo ? 0 : 1;
    static constexpr int kOffStage = kOffDS + (kDsInDo ? 0 : kDsBytes);
    static constexpr int kOffX = kOffStage + kStageBufs * kStageBytes;  // per stage: lse rows, D rows
    static_assert(kDsInDo || kGroups - kRedGroups <= 16, "d = 64: one staging round per step");
    static constexpr int kOffOnes = kOffX + kStages * 2 * kXBytes;
    static constexpr int kOffZero = kOffOnes + kBK * 16;
    static constexpr int kOffBar = kOffZero + 2048;
    static constexpr int kNumBars = 1 + 4 * kStages + 9;
    static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;
    static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 384;
    // register budgets (setmaxnreg): warpgroup 2 gives 32 back, which the reducers take; the
    // element-wise warps keep the launch's 128 (measured at d = 64: 144 for the reducers and 136 for
    // the element-wise warps, 206.5 ms against 206.2)
    static constexpr int kOtherRegs = 96, kRedRegs = 160;
    static constexpr int kEwRegs = (4 * kKqLaunchRegs - kOtherRegs - kRedRegs) / 2 / 8 * 8;
    // dQ's columns: at d = 128 the dP^T columns (TMEM is full), so that dP^T(it+1) waits until the
    // reducers have drained dQ(it); at d = 64 columns of its own (448 .. 511), so that only dQ(it+1)
    // waits for that (measured at 128K: 206.3 ms against 212.2)
    static constexpr bool kDqOwn = D == 64;
    static constexpr uint32_t kColDQ = kDqOwn ? 448 : kColDP;
};
static_assert(KqCfg<128>::kSmemBytes <= 227 * 1024 && KqCfg<64>::kSmemBytes <= 227 * 1024, "shared memory");
static_assert(2 * KqCfg<128>::kEwRegs + KqCfg<128>::kOtherRegs + KqCfg<128>::kRedRegs <= 4 * kKqLaunchRegs &&
                  2 * KqCfg<64>::kEwRegs + KqCfg<64>::kOtherRegs + KqCfg<64>::kRedRegs <= 4 * kKqLaunchRegs,
              "register split exceeds the launch allocation of a sub-partition");

// bytes of shared memory (16-byte aligned, a multiple of 16) added into global float32 memory by the
// TMA engine, completion tracked by this thread's bulk-async group
__device__ __forceinline__ void bulk_reduce_add_f32(float* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(dst), "r"(src),
                 "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// the four reducer warps (named barrier 1): every thread's flag ANDed
__device__ __forceinline__ bool reducers_all(bool ok) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)ok)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void reducers_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

template <int D, bool SPLIT>
__global__ void __launch_bounds__(kKqThreads, 1)
    dkdvq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                 const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v, const DevBwd p) {
    using C = KqCfg<D>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + C::kNumBars * 8);
    __shared__ int abort_flag;
    const uint32_t bar0 = sbase + C::kOffBar;
    auto BAR = [&](int idx) { return bar0 + 8u * (uint32_t)idx; };
    const int kKvFull = 0, kQFull = 1, kQEmpty = 1 + S, kOFull = 1 + 2 * S, kOEmpty = 1 + 3 * S,
              kSFull = 1 + 4 * S, kDPFull = kSFull + 1, kPReady = kSFull + 2, kDVDone = kSFull + 3,
              kDSReady = kSFull + 4, kDQFull = kSFull + 5, kDQFree = kSFull + 6, kOReady = kSFull + 7,
              kDrain = kSFull + 8;
    // shared-memory offset of step it's dS^T
    auto ds_off = [](int it) { return C::kDsInDo ? C::kOffDO + (it % S) * C::kTile : C::kOffDS; };

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int Hkv = p.Hq / p.g;
    // group-major: all key tiles of one (outer index, KV head), low key tiles first (as pass 2)
    const int n_kt = (p.Nkv + C::kBK - 1) / C::kBK;
    const int grp = blockIdx.x / n_kt;
    const int kt = blockIdx.x % n_kt;
    const int hk = grp % Hkv;
    int q_outer, kv_outer, shift;
    bwd_outer(p, grp / Hkv, q_outer, kv_outer, shift);
    const int n_qt = (p.N + C::kBQ - 1) / C::kBQ;
    const int first_q = kt * C::kBK - shift;
    const int qt_lo = (p.causal && first_q > 0) ? first_q / C::kBQ : 0;
    const int nq = max(0, n_qt - qt_lo);
    const int n_it = p.g * nq;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(BAR(kKvFull), 1);
        for (int s = 0; s < S; ++s) {
            mbar_init(BAR(kQFull + s), 1);
            mbar_init(BAR(kQEmpty + s), 1);
            mbar_init(BAR(kOFull + s), 1);
            mbar_init(BAR(kOEmpty + s), 1);
        }
        mbar_init(BAR(kSFull), 1);
        mbar_init(BAR(kDPFull), 1);
        mbar_init(BAR(kPReady), kKqEwWarps * 32);
        mbar_init(BAR(kDVDone), 1);
        mbar_init(BAR(kDSReady), kKqEwWarps * 32);
        mbar_init(BAR(kDQFull), 1);
        mbar_init(BAR(kDQFree), 4 * 32);  // the four reducer warps
        mbar_init(BAR(kOReady), 1);
        mbar_init(BAR(kDrain), 1);
        fence_mbar_init();
    }
    if (warp == kKqMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    if (threadIdx.x < C::kBK) {
        // row t of the ones operand (bf16 1.0 in its first three columns) and 16 bytes of zeros
        *reinterpret_cast<uint4*>(smem + C::kOffOnes + threadIdx.x * 16) = make_uint4(0x3F803F80u, 0x3F80u, 0u, 0u);
        *reinterpret_cast<uint4*>(smem + C::kOffZero + threadIdx.x * 16) = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    volatile int* abort_p = &abort_flag;

    // Each role's code sits inside the branch that set its register budget; every warp of a
    // warpgroup executes the same setmaxnreg.
    if (warp >= kKqProducerWarp && warp < kKqRedWarp0) {
        setmaxnreg_dec<C::kOtherRegs>();
    if (n_it > 0 && warp == kKqProducerWarp && lane == 0) {
        // ---------------------------------------------------------------- TMA producer
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_do);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        mbar_arrive_expect_tx(BAR(kKvFull), 2 * C::kTile);
        const TokOuter kv = split_pos(kt * C::kBK, kv_outer, SPLIT ? p.split_np : 0, p.split_b);
        for (int c = 0; c < C::kChunks; ++c) {
            tma_load_4d(sbase + C::kOffK + c * 16384, &tm_k, c * 64, hk, kv.tok, kv.outer, BAR(kKvFull));
            tma_load_4d(sbase + C::kOffV + c * 16384, &tm_v, c * 64, hk, kv.tok, kv.outer, BAR(kKvFull));
        }
        TokOuter q_next = {0, 0};  // split mode: the next query tile's coordinates, stepped through the shards
        int nq_issued = 0, no_issued = 0;  // Q and dO tiles whose loads were issued
        for (int it = 0; it < n_it; ++it) {
            const int s = it % S;
            const int hq = hk * p.g + it / nq;
            const int qt = qt_lo + it % nq;
            TokOuter qa;
            if constexpr (SPLIT) {
                if (it % nq == 0) q_next = split_pos(qt * C::kBQ, q_outer, p.split_np, p.split_b);
                qa = q_next;
                q_next.tok += C::kBQ;
                if (q_next.tok == p.split_np) {
                    q_next.tok = 0;
                    q_next.outer += p.split_b;
                }
            } else {
                qa = {qt * C::kBQ, q_outer};
            }
            const int64_t voff = ((int64_t)q_outer * p.Hq + hq) * p.Npad + (int64_t)qt * C::kBQ;
            // Q (with the lse rows): its stage is free once dK of step it - S is done
            if (it >= S && !mbar_wait(BAR(kQEmpty + s), ((it / S) - 1) & 1, abort_p, 50, p.status)) break;
            mbar_arrive_expect_tx(BAR(kQFull + s), C::kTile + C::kXBytes);
            for (int c = 0; c < C::kChunks; ++c)
                tma_load_4d(sbase + C::kOffQ + s * C::kTile + c * 16384, &tm_q, c * 64, hq, qa.tok, qa.outer,
                            BAR(kQFull + s));
            bulk_load(sbase + C::kOffX + s * 2 * C::kXBytes, p.xl + voff, C::kXBytes, BAR(kQFull + s));
            nq_issued = it + 1;
            // dO (with the D rows): its stage (and the dS^T over it) is free once dQ of step it - S is done
            if (it >= S && !mbar_wait(BAR(kOEmpty + s), ((it / S) - 1) & 1, abort_p, 51, p.status)) break;
            mbar_arrive_expect_tx(BAR(kOFull + s), C::kTile + C::kXBytes);
            for (int c = 0; c < C::kChunks; ++c)
                tma_load_4d(sbase + C::kOffDO + s * C::kTile + c * 16384, &tm_do, c * 64, hq, qa.tok, qa.outer,
                            BAR(kOFull + s));
            bulk_load(sbase + C::kOffX + s * 2 * C::kXBytes + C::kXBytes, p.xd + voff, C::kXBytes, BAR(kOFull + s));
            no_issued = it + 1;
        }
        // every issued load lands before the CTA can exit (after an abort, too)
        mbar_drain(BAR(kKvFull), 0, 53, p.status);
        drain_ring(BAR(kQFull), S, nq_issued, 54, p.status);
        drain_ring(BAR(kOFull), S, no_issued, 55, p.status);
    } else if (n_it > 0 && warp == kKqMmaWarp && lane == 0) {
        // ---------------------------------------------------------------- MMA issuer
        constexpr uint32_t kIdS = idesc_bf16(C::kBK, C::kBQ, 0, 0);  // S^T = K Q^T, dP^T = V dO^T
        constexpr uint32_t kIdG = idesc_bf16(C::kBK, D, 0, 1);       // dV += P^T dO, dK += dS^T Q
        constexpr uint32_t kIdQ = idesc_bf16(C::kBQ, D, 1, 1);       // dQ = dS K: A and B M/N-major
        const uint64_t dk0 = sdesc_sw128(sbase + C::kOffK, 16, 1024), dv0 = sdesc_sw128(sbase + C::kOffV, 16, 1024);
        const uint64_t k_mn = sdesc_sw128(sbase + C::kOffK, 16384, 1024);  // K as the N-major B of dQ
        auto plain = [&](int off) { return sdesc_plain(sbase + off, (uint32_t)(C::kOffZero - off), 128); };
        const uint64_t dones = plain(C::kOffOnes);
        // S'^T (A = K, x = 0: lse rows, B = Q) or dP'^T (A = V, x = 1: D rows, B = dO) of step it
        auto issue_t = [&](int it, uint64_t a0, int off_b, uint32_t col, int x) {
            const int s = it % S;
            const uint64_t b0 = sdesc_sw128(sbase + off_b + s * C::kTile, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = ((kk / 4) * 16384 + (kk % 4) * 32) >> 4;
                mma_ss(tmem + col, a0 + off, b0 + off, kIdS, kk > 0);
            }
            mma_ss(tmem + col, dones, plain(C::kOffX + (2 * s + x) * C::kXBytes), kIdS, 1u);
        };
        // dV += P^T dO: A = P^T from TMEM (the bf16 half of each 64-column block of S^T), B = dO N-major
        auto issue_dv = [&](int it) {
            const uint64_t b0 = sdesc_sw128(sbase + C::kOffDO + (it % S) * C::kTile, 16384, 1024);
#pragma unroll
            for (int kk = 0; kk < C::kBQ / 16; ++kk) {
                const uint32_t a = tmem + C::kColS + (kk / 4) * 64 + (kk % 4) * 8;
                mma_ts(tmem + C::kColDV, a, b0 + (kk * 2048 >> 4), kIdG, (it > 0 || kk > 0) ? 1u : 0u);
            }
        };
        // dK += dS^T Q: A = dS^T from TMEM (the bf16 half of each 64-column block of dP^T), B = Q N-major
        auto issue_dk = [&](int it) {
            const uint64_t b0 = sdesc_sw128(sbase + C::kOffQ + (it % S) * C::kTile, 16384, 1024);
#pragma unroll
            for (int kk = 0; kk < C::kBQ / 16; ++kk) {
                const uint32_t a = tmem + C::kColDP + (kk / 4) * 64 + (kk % 4) * 8;
                mma_ts(tmem + C::kColDK, a, b0 + (kk * 2048 >> 4), kIdG, (it > 0 || kk > 0) ? 1u : 0u);
            }
        };
        // dQ = dS K into its columns: A = the dS^T bytes read M-major (keys 16 kk .. + 15), B = K N-major
        auto issue_dq = [&](int it) {
            const uint64_t a0 = sdesc_sw128(sbase + ds_off(it), 16384, 1024);
#pragma unroll
            for (int kk = 0; kk < C::kBK / 16; ++kk)
                mma_ss(tmem + C::kColDQ, a0 + (kk * 2048 >> 4), k_mn + (kk * 2048 >> 4), kIdQ, kk > 0 ? 1u : 0u);
        };
        bool ok = mbar_wait(BAR(kKvFull), 0, abort_p, 56, p.status);
        ok = ok && mbar_wait(BAR(kQFull), 0, abort_p, 57, p.status);
        ok = ok && mbar_wait(BAR(kOFull), 0, abort_p, 58, p.status);
        if (ok) {
            tc_fence_after();
            issue_t(0, dk0, C::kOffQ, C::kColS, 0);
            mma_commit(BAR(kSFull));
            issue_t(0, dv0, C::kOffDO, C::kColDP, 1);
            mma_commit(BAR(kDPFull));
        }
        ok = ok && mbar_wait(BAR(kPReady), 0, abort_p, 59, p.status);
        if (ok) {
            tc_fence_after();
            issue_dv(0);
            mma_commit(BAR(kDVDone));
        }
        if (ok && n_it > 1) {
            ok = mbar_wait(BAR(kQFull + 1 % S), (1 / S) & 1, abort_p, 57, p.status);
            if (ok) {
                tc_fence_after();
                issue_t(1, dk0, C::kOffQ, C::kColS, 0);  // after dV(0), which read P^T from these columns
                mma_commit(BAR(kSFull));
            }
        }
        for (int it = 0; ok && it < n_it; ++it) {
            const int s = it % S;
            if (!mbar_wait(BAR(kDSReady), it & 1, abort_p, 60, p.status)) break;
            tc_fence_after();
            issue_dk(it);
            mma_commit(BAR(kQEmpty + s));
            // d = 64: dQ(it-1) drained from dQ's own columns; d = 128: over the dP^T columns, after
            // dK(it), which read dS^T from them
            if (C::kDqOwn && it > 0 && !mbar_wait(BAR(kDQFree), (it - 1) & 1, abort_p, 61, p.status)) break;
            issue_dq(it);
            mma_commit(BAR(kDQFull));
            if constexpr (!C::kDsInDo) mma_commit(BAR(kOEmpty + s));  // d = 128: the reducers release it
            if (it + 1 < n_it) {
                const int s1 = (it + 1) % S;
                // d = 128: dP^T(it+1) overwrites dQ(it), after the reducers have drained it. It goes
                // before dV(it+1), so that dS(it+1) is computed while dV(it+1) runs.
                if (!C::kDqOwn && !mbar_wait(BAR(kDQFree), it & 1, abort_p, 61, p.status)) break;
                if (!mbar_wait(BAR(kOFull + s1), ((it + 1) / S) & 1, abort_p, 58, p.status)) break;
                tc_fence_after();
                issue_t(it + 1, dv0, C::kOffDO, C::kColDP, 1);
                mma_commit(BAR(kDPFull));
                if (!mbar_wait(BAR(kPReady), (it + 1) & 1, abort_p, 59, p.status)) break;
                tc_fence_after();
                issue_dv(it + 1);
                mma_commit(BAR(kDVDone));
                if (it + 2 < n_it) {
                    if (!mbar_wait(BAR(kQFull + (it + 2) % S), ((it + 2) / S) & 1, abort_p, 57, p.status)) break;
                    tc_fence_after();
                    issue_t(it + 2, dk0, C::kOffQ, C::kColS, 0);  // after dV(it+1), which read P^T here
                    mma_commit(BAR(kSFull));
                }
            } else {
                mma_commit(BAR(kOReady));
            }
        }
        // every issued MMA completes before TMEM is freed (after an abort, too)
        mma_commit(BAR(kDrain));
        mbar_drain(BAR(kDrain), 0, 62, p.status);
    }
    } else if (warp >= kKqRedWarp0) {
        if constexpr (C::kRedRegs > kKqLaunchRegs) setmaxnreg_inc<C::kRedRegs>();
        // ---------------------------------------------------------------- dQ reducers
        // warp w: query rows 32 (w % 4) .. + 31 of the step's tile (TMEM lanes), every column.  dQ(it)
        // goes from TMEM to registers (then dQ(it+1), or at d = 128 dP^T(it+1), may overwrite it);
        // kRedGroups of its column
        // groups go from there into the accumulator by red.global, the others through the shared
        // staging buffer ([groups][128 rows][4]) and the TMA engine's bulk reduction (the same bytes
        // are contiguous in the accumulator).
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        const bool elected = warp == kKqRedWarp0 && lane == 0;
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16) + C::kColDQ;
        for (int it = 0; it < n_it; ++it) {
            const bool ok_w = __all_sync(0xffffffffu, mbar_wait(BAR(kDQFull), it & 1, abort_p, 66, p.status));
            if (!reducers_all(ok_w)) break;  // all four warps leave together (they share named barrier 1)
            tc_fence_after();
            uint32_t v[D / 32][32];
#pragma unroll
            for (int c = 0; c < D / 32; ++c) tmem_ld32(lane_base + c * 32, v[c]);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(BAR(kDQFree));  // in registers: the MMA may overwrite these columns
            const int hq = hk * p.g + it / nq;
            const int qt = qt_lo + it % nq;
            float* tile = p.dq_acc + (((int64_t)q_outer * p.Hq + hq) * p.Npad + (int64_t)qt * C::kBQ) * D;
            const uint32_t stage =
                sbase + (C::kDsInDo ? ds_off(it)
                                    : C::kOffStage + (it % (C::kStageBufs > 1 ? C::kStageBufs : 1)) * C::kStageBytes);
            if (!C::kDsInDo) {
                // the buffer's previous step (it - kStageBufs): its bulk reduction has read it (with two
                // buffers, the other step's group may still be in flight)
                if (elected) {
                    if constexpr (C::kStageBufs == 2) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
                    else asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                }
                reducers_sync();
            }
            // column group g of row r sits at (g * 128 + r) * 4 floats of the tile
            auto red_groups = [&]() {
                float* rowp = tile + r * 4;
#pragma unroll
                for (int g = C::kGroups - C::kRedGroups; g < C::kGroups; ++g) {
                    const uint32_t* x = &v[g / 8][4 * (g % 8)];
                    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(rowp + g * C::kBQ * 4),
                                 "f"(__uint_as_float(x[0])), "f"(__uint_as_float(x[1])), "f"(__uint_as_float(x[2])),
                                 "f"(__uint_as_float(x[3]))
                                 : "memory");
                }
            };
            if (C::kRedFirst) red_groups();
#pragma unroll
            for (int g0 = 0; g0 < C::kGroups - C::kRedGroups; g0 += 16) {
                const int ng = C::kGroups - C::kRedGroups - g0 < 16 ? C::kGroups - C::kRedGroups - g0 : 16;
                // groups g0 .. g0 + ng - 1 of row r: the warp's 32 rows of one group are 512 bytes
#pragma unroll
                for (int g = 0; g < ng; ++g) {
                    const uint32_t* x = &v[(g0 + g) / 8][4 * ((g0 + g) % 8)];
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(stage + (g * C::kBQ + r) * 16),
                                 "r"(x[0]), "r"(x[1]), "r"(x[2]), "r"(x[3])
                                 : "memory");
                }
                fence_proxy_async_smem();
                reducers_sync();
                if (elected) {
                    bulk_reduce_add_f32(tile + g0 * C::kBQ * 4, stage, (uint32_t)ng * C::kBQ * 16);
                    if (C::kDsInDo) bulk_wait_read_all();  // the staging buffer may be written again
                }
                if (C::kDsInDo) reducers_sync();
            }
            // d = 128: the staging was this step's dO tile; the producer may load the next one into it
            // (before the red.global issue, which can wait on the L1TEX queue)
            if (C::kDsInDo && elected) mbar_arrive(BAR(kOEmpty + it % S));
            if (!C::kRedFirst) red_groups();
        }
        if (elected) bulk_wait_all();  // every reduction issued has reached global memory
    } else {
        if constexpr (C::kEwRegs > kKqLaunchRegs) setmaxnreg_inc<C::kEwRegs>();
        // ---------------------------------------------------------------- element-wise warps
        // warp w: TMEM lanes 32 (w % 4) .. + 31 (its key rows of S^T / dP^T), query columns of half w / 4
        const int quad = warp & 3, half = warp >> 2;
        const int krow = quad * 32 + lane;  // key row of S^T, dP^T and dS^T
        const int key = kt * C::kBK + krow;
        const bool key_ok = key < p.Nkv;
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        const uint32_t col_s = C::kColS + half * 64, col_dp = C::kColDP + half * 64;
        float pf[64];
        bool ok = true;
        // a wait whose outcome is the same for the whole warp (the TMEM loads and stores after it
        // are warp-collective): a warp gives up if any of its lanes did
        auto ew_wait = [&](int idx, uint32_t parity, int site) {
            return __all_sync(0xffffffffu, mbar_wait(BAR(idx), parity, abort_p, site, p.status));
        };
        // P = exp2(S' scale log2 e) of step j (S' = S - lse / scale), bf16 over S^T for dV
        auto do_p = [&](int j) -> bool {
            const int qt = qt_lo + j % nq;
            if (!ew_wait(kSFull, j & 1, 63)) return false;
            tc_fence_after();
            uint32_t ra[32], rb[32];
            tmem_ld32(lane_base + col_s, ra);
            tmem_ld32(lane_base + col_s + 32, rb);
            tmem_wait_ld();
            const int q0 = qt * C::kBQ + half * 64;  // query of column 0
            const bool need_mask = (p.causal && q0 + shift < kt * C::kBK + C::kBK - 1) || !key_ok;
            const int qmin_ok = key_ok ? (p.causal ? key - shift - q0 : 0) : 64;  // first visible column
            uint32_t pk[32];
            const float2 c2 = make_float2(p.scale_log2, p.scale_log2);
#pragma unroll
            for (int e = 0; e < 64; e += 2) {
                const float2 x = mul2(make_float2(__uint_as_float(e < 32 ? ra[e] : rb[e - 32]),
                                                  __uint_as_float(e < 32 ? ra[e + 1] : rb[e - 31])),
                                      c2);
                pf[e] = ex2_approx(x.x);
                pf[e + 1] = ex2_approx(x.y);
                if (need_mask) {
                    if (e < qmin_ok) pf[e] = 0.f;
                    if (e + 1 < qmin_ok) pf[e + 1] = 0.f;
                }
                pk[e / 2] = pack_bf16(pf[e], pf[e + 1]);
            }
            tmem_st32(lane_base + col_s, pk);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(BAR(kPReady));
            return true;
        };
        // dS = P (dP - D) of step j (dP' = dP - D), bf16, as this thread's row of dS^T in shared memory
        auto do_ds = [&](int j) -> bool {
            if (!ew_wait(kDPFull, j & 1, 64)) return false;
            tc_fence_after();
            uint32_t ra[32], rb[32];
            tmem_ld32(lane_base + col_dp, ra);
            tmem_ld32(lane_base + col_dp + 32, rb);
            tmem_wait_ld();
            uint32_t pk[32];
#pragma unroll
            for (int e = 0; e < 64; e += 2) {
                const float2 ds = mul2(make_float2(pf[e], pf[e + 1]),
                                       make_float2(__uint_as_float(e < 32 ? ra[e] : rb[e - 32]),
                                                   __uint_as_float(e < 32 ? ra[e + 1] : rb[e - 31])));
                pk[e / 2] = pack_bf16(ds.x, ds.y);
            }
            // dS^T over the first 32 of this warp's dP^T columns: the A operand of dK (dP^T is in registers)
            tmem_st32(lane_base + col_dp, pk);
            // at d = 128 dS^T also goes over this step's dO tile (the A operand of dQ): wait until
            // dV(j), its last reader, is done
            if (C::kDsInDo && !ew_wait(kDVDone, j & 1, 65)) return false;
            // row krow, queries 64 half .. + 63: one 128-byte row of the 128-byte-swizzled K-major tile
            uint8_t* row = smem + ds_off(j) + half * 16384 + krow * 128;
#pragma unroll
            for (int u = 0; u < 8; ++u)
                *reinterpret_cast<uint4*>(row + ((u ^ (krow & 7)) << 4)) =
                    make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
            fence_proxy_async_smem();
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(BAR(kDSReady));
            return true;
        };
        if (n_it > 0) ok = do_p(0) && do_ds(0);
        for (int it = 0; ok && it + 1 < n_it; ++it) {
            if (!do_p(it + 1)) { ok = false; break; }
            if (!do_ds(it + 1)) { ok = false; break; }
        }
        if (ok && n_it > 0) ok = ew_wait(kOReady, 0, 67);
        if (ok) {
            // warps 0-3 write dV, warps 4-7 write dK (scale applied here)
            tc_fence_after();
            const bool valid = key < p.Nkv;
            const TokOuter ka = split_pos(key, kv_outer, SPLIT ? p.split_np : 0, p.split_b);
            const int64_t base = (int64_t)ka.outer * p.k_s_outer + (int64_t)hk * p.k_s_head + (int64_t)ka.tok * p.k_s_tok;
            const uint32_t col = half == 0 ? C::kColDV : C::kColDK;
            const float mul = half == 0 ? 1.f : p.scale;
            uint16_t* out16 = half == 0 ? p.dv : p.dk;
            float* out32 = half == 0 ? p.dv_f : p.dk_f;  // ring schedules: float32, added to when acc != 0
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t r[32];
                if (n_it > 0) {
                    tmem_ld32(lane_base + col + cc * 32, r);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) r[e] = 0u;
                }
                if (valid) store_row32(out16, out32, p.acc, base + cc * 32, r, mul);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kKqMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// The dQ accumulator to zero: 16-byte stores, grid-stride (n4 = float4 count).
// dQ = scale * accumulator, rounded to bf16: thread (tile, part, row) converts columns 32 part .. + 31
// of one query row (reads of consecutive threads are consecutive 16-byte groups of the tile).
template <int D, bool SPLIT>
__global__ void __launch_bounds__(256) dq_store_kernel(const DevBwd p, int64_t n_threads) {
    const int64_t t = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (t >= n_threads) return;
    constexpr int kParts = D / 32;
    const int r = (int)(t % 128);
    const int part = (int)((t / 128) % kParts);
    const int64_t tile = t / (128 * kParts);  // z * (Npad / 128) + query tile
    const int64_t tiles_per_z = p.Npad / 128;
    const int z = (int)(tile / tiles_per_z);
    const int n = (int)(tile % tiles_per_z) * 128 + r;
    if (n >= p.N) return;
    const float* src = p.dq_acc + tile * 128 * D;
    uint32_t v[32];
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        const float4 x = *reinterpret_cast<const float4*>(src + ((part * 8 + g) * 128 + r) * 4);
        v[4 * g] = __float_as_uint(x.x);
        v[4 * g + 1] = __float_as_uint(x.y);
        v[4 * g + 2] = __float_as_uint(x.z);
        v[4 * g + 3] = __float_as_uint(x.w);
    }
    const int outer = z / p.Hq, head = z % p.Hq;
    const TokOuter at = split_pos(n, outer, SPLIT ? p.split_np : 0, p.split_b);
    const int64_t off = (int64_t)at.outer * p.q_s_outer + (int64_t)head * p.q_s_head + (int64_t)at.tok * p.q_s_tok +
                        part * 32;
    store_row32(p.dq, nullptr, 0, off, v, p.scale);
}

struct BwdMaps {
    CUtensorMap q, dout, k, v;
};

template <int D>
bool make_bwd_maps(const BwdParams& b, int q_rows, BwdMaps* m) {
    return make_tmap_bf16(&m->q, b.q, D, q_rows) && make_tmap_bf16(&m->dout, b.dout, D, q_rows) &&
           make_tmap_bf16(&m->k, b.k, D, 128) && make_tmap_bf16(&m->v, b.v, D, 128);
}

// query and key positions per outer index: the tensors' token extents, or in the sequence-sharded
// in-place mode the whole sequence (every shard of one batch)
int q_len_of(const BwdParams& b) { return b.split_np ? b.q.n_tok * (b.q.n_outer / b.split_b) : b.q.n_tok; }
int kv_len_of(const BwdParams& b) { return b.split_np ? b.k.n_tok * (b.k.n_outer / b.split_b) : b.k.n_tok; }

int npad_of(const BwdParams& b) { return (q_len_of(b) + 127) / 128 * 128; }

DevBwd dev_params(const BwdParams& b) {
    const int Npad = npad_of(b);
    const size_t rows = (size_t)b.n_z * Npad;
    DevBwd p;
    p.Hq = b.q.n_head;
    p.g = b.g;
    p.N = q_len_of(b);
    p.Nkv = kv_len_of(b);
    p.split_np = b.split_np;
    p.split_b = b.split_b;
    p.kv_gathered = b.kv_gathered;
    p.zigzag = b.zigzag;
    p.zz_kh = b.zz_kh;
    p.zz_qh = b.zz_qh;
    p.Npad = Npad;
    p.causal = b.causal;
    p.ring_i0 = b.ring_i0;
    p.ring_t = b.ring_t;
    p.ring_p = b.ring_p;
    p.bsz = b.bsz;
    p.n_outer = b.n_outer;
    p.scale = b.scale;
    p.scale_log2 = b.scale * kLog2e;
    p.dvec = b.ws;
    p.lse2 = b.ws + rows;
    p.xl = reinterpret_cast<const uint4*>(b.ws + 2 * rows);
    p.xd = p.xl + rows;
    p.q = static_cast<const uint16_t*>(b.q.ptr);
    p.dout = static_cast<const uint16_t*>(b.dout.ptr);
    p.dq = static_cast<uint16_t*>(b.dq);
    p.dk = static_cast<uint16_t*>(b.dk);
    p.dv = static_cast<uint16_t*>(b.dv);
    p.dq_f = b.dq_f32;
    p.dk_f = b.dk_f32;
    p.dv_f = b.dv_f32;
    p.acc = b.accumulate;
    p.q_s_head = b.q.s_head;
    p.q_s_tok = b.q.s_tok;
    p.q_s_outer = b.q.s_outer;
    p.k_s_head = b.k.s_head;
    p.k_s_tok = b.k.s_tok;
    p.k_s_outer = b.k.s_outer;
    p.status = b.status;
    p.dq_acc = b.dq_acc;
    return p;
}

template <int D, bool SPLIT>
cudaError_t pre_t(const BwdParams& b, cudaStream_t stream) {
    const DevBwd p = dev_params(b);
    PreArgs a;
    a.o = static_cast<const uint16_t*>(b.o.ptr);
    a.dout = static_cast<const uint16_t*>(b.dout.ptr);
    a.lse = b.lse;
    a.s_head = b.o.s_head;
    a.s_tok = b.o.s_tok;
    a.s_outer = b.o.s_outer;
    a.l_s_head = b.l_s_head;
    a.l_s_tok = b.l_s_tok;
    a.l_s_outer = b.l_s_outer;
    a.heads = b.q.n_head;
    a.N = q_len_of(b);
    a.split_np = b.split_np;
    a.split_b = b.split_b;
    a.Npad = p.Npad;
    a.n_z = b.n_z;
    a.scale = b.scale;
    a.dvec = const_cast<float*>(p.dvec);
    a.lse2 = const_cast<float*>(p.lse2);
    a.xl = const_cast<uint4*>(p.xl);
    a.xd = const_cast<uint4*>(p.xd);
    a.dq_acc = b.dq_acc;
    const int64_t tiles = (int64_t)b.n_z * p.Npad / 128;
    if (tiles == 0) return cudaSuccess;
    bwd_pre_kernel<D, SPLIT><<<(unsigned)tiles, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

template <int D, bool SPLIT>
cudaError_t dkdv_t(const BwdParams& b, cudaStream_t stream) {
    BwdMaps m;
    if (!make_bwd_maps<D>(b, KvCfg<D>::kBQ, &m)) return cudaErrorInvalidValue;
    auto kern = dkdv_kernel<D, SPLIT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, KvCfg<D>::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int64_t n_kt = (kv_len_of(b) + 127) / 128;
    const int64_t grid = n_kt * b.n_outer * (b.q.n_head / b.g);
    if (grid == 0) return cudaSuccess;
    kern<<<(unsigned)grid, kKvThreads, KvCfg<D>::kSmemBytes, stream>>>(m.q, m.dout, m.k, m.v, dev_params(b));
    return cudaGetLastError();
}

template <int D, bool SPLIT>
cudaError_t dq_t(const BwdParams& b, cudaStream_t stream) {
    BwdMaps m;
    if (!make_bwd_maps<D>(b, DqCfg<D>::kBM, &m)) return cudaErrorInvalidValue;
    auto kern = dq_kernel<D, SPLIT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DqCfg<D>::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int64_t n_qt = (q_len_of(b) + 127) / 128;
    const int64_t grid = n_qt * b.n_outer * b.q.n_head;
    if (grid == 0) return cudaSuccess;
    kern<<<(unsigned)grid, kDqThreads, DqCfg<D>::kSmemBytes, stream>>>(m.k, m.v, dev_params(b));
    return cudaGetLastError();
}

template <int D, bool SPLIT>
cudaError_t dkdvq_t(const BwdParams& b, cudaStream_t stream) {
    if (!b.dq_acc) return cudaErrorInvalidValue;
    BwdMaps m;
    if (!make_bwd_maps<D>(b, KqCfg<D>::kBQ, &m)) return cudaErrorInvalidValue;
    auto kern = dkdvq_kernel<D, SPLIT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, KqCfg<D>::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int64_t n_kt = (kv_len_of(b) + 127) / 128;
    const int64_t grid = n_kt * b.n_outer * (b.q.n_head / b.g);
    if (grid == 0) return cudaSuccess;
    kern<<<(unsigned)grid, kKqThreads, KqCfg<D>::kSmemBytes, stream>>>(m.q, m.dout, m.k, m.v, dev_params(b));
    return cudaGetLastError();
}

template <int D, bool SPLIT>
cudaError_t dq_store_t(const BwdParams& b, cudaStream_t stream) {
    if (!b.dq_acc || !b.dq) return cudaErrorInvalidValue;
    const DevBwd p = dev_params(b);
    const int64_t n_threads = (int64_t)b.n_z * p.Npad * (D / 32);
    if (n_threads == 0) return cudaSuccess;
    dq_store_kernel<D, SPLIT><<<(unsigned)((n_threads + 255) / 256), 256, 0, stream>>>(p, n_threads);
    return cudaGetLastError();
}

// each pass in two forms: the sequence-sharded in-place addressing (split_np > 0) or not
template <template <int, bool> class F>
cudaError_t dispatch(const BwdParams& b, cudaStream_t stream) {
    const bool split = b.split_np > 0;
    if (b.d == 64) return split ? F<64, true>::run(b, stream) : F<64, false>::run(b, stream);
    if (b.d == 128) return split ? F<128, true>::run(b, stream) : F<128, false>::run(b, stream);
    return cudaErrorInvalidValue;
}
template <int D, bool S>
struct PreF {
    static cudaError_t run(const BwdParams& b, cudaStream_t s) { return pre_t<D, S>(b, s); }
};
template <int D, bool S>
struct DkdvF {
    static cudaError_t run(const BwdParams& b, cudaStream_t s) { return dkdv_t<D, S>(b, s); }
};
template <int D, bool S>
struct DqF {
    static cudaError_t run(const BwdParams& b, cudaStream_t s) { return dq_t<D, S>(b, s); }
};
template <int D, bool S>
struct DkdvqF {
    static cudaError_t run(const BwdParams& b, cudaStream_t s) { return dkdvq_t<D, S>(b, s); }
};
template <int D, bool S>
struct DqStoreF {
    static cudaError_t run(const BwdParams& b, cudaStream_t s) { return dq_store_t<D, S>(b, s); }
};

}  // namespace

cudaError_t launch_bwd_pre(const BwdParams& b, cudaStream_t stream) { return dispatch<PreF>(b, stream); }
cudaError_t launch_bwd_dkdv(const BwdParams& b, cudaStream_t stream) { return dispatch<DkdvF>(b, stream); }
cudaError_t launch_bwd_dq(const BwdParams& b, cudaStream_t stream) { return dispatch<DqF>(b, stream); }
cudaError_t launch_bwd_dkdvq(const BwdParams& b, cudaStream_t stream) { return dispatch<DkdvqF>(b, stream); }
cudaError_t launch_bwd_dq_store(const BwdParams& b, cudaStream_t stream) { return dispatch<DqStoreF>(b, stream); }

}  // namespace usp

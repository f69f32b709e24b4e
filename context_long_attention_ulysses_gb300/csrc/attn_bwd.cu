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
// Three launches, no atomics, deterministic:
//  1. pre:  D_i and lse_i*log2(e) into a workspace padded to 128-row tiles
//           (padding rows: lse = +inf, so their P is exactly 0).
//  2. dK/dV: one CTA per (KV head, 128-key tile).  It walks every query head
//           of the GQA group and every 64-row query tile that sees its keys:
//             S^T  = K Q^T,  dP^T = V dO^T          (tcgen05, shared-memory operands)
//             P^T, dS^T on CUDA cores (thread = key row = TMEM lane), bf16 into TMEM
//             dV  += P^T dO, dK += dS^T Q           (A from TMEM, B MN-major)
//           dK and dV stay in TMEM for the whole walk.
//  3. dQ:   one CTA per (query head, 128-row tile) walking its visible key
//           tiles: S = Q K^T, dP = dO V^T, dS on CUDA cores into TMEM,
//           dQ += dS K.
// TMEM columns are laid out so that no MMA ever writes columns that another
// MMA may still be reading: S/dP are single-buffered (the next S is issued
// only after the softmax warps have loaded the previous one) and the bf16
// operands P^T, dS^T (dS in pass 3) are double-buffered.
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"

namespace usp {

namespace {

constexpr int kThreads = 6 * 32;
constexpr int kSoftmaxWarps = 4;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------------ pass 1
// One warp per padded row: dvec = dO . O (fp32), lse2 = lse * log2(e).
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dout,
                                                      const float* __restrict__ lse, float* __restrict__ dvec,
                                                      float* __restrict__ lse2, int Zq, int N, int Npad) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * 8 + threadIdx.x / 32;
    if (row >= (int64_t)Zq * Npad) return;
    const int z = (int)(row / Npad);
    const int n = (int)(row % Npad);
    if (n >= N) {
        if (lane == 0) {
            dvec[row] = 0.f;
            lse2[row] = INFINITY;
        }
        return;
    }
    constexpr int kPer = D / 32;  // elements per lane (2 or 4)
    const int64_t base = ((int64_t)z * N + n) * D + lane * kPer;
    float acc = 0.f;
    if constexpr (kPer == 4) {
        const uint2 a = *reinterpret_cast<const uint2*>(o + base);
        const uint2 b = *reinterpret_cast<const uint2*>(dout + base);
        acc = __uint_as_float(a.x << 16) * __uint_as_float(b.x << 16) +
              __uint_as_float(a.x & 0xFFFF0000u) * __uint_as_float(b.x & 0xFFFF0000u) +
              __uint_as_float(a.y << 16) * __uint_as_float(b.y << 16) +
              __uint_as_float(a.y & 0xFFFF0000u) * __uint_as_float(b.y & 0xFFFF0000u);
    } else {
        const uint32_t a = *reinterpret_cast<const uint32_t*>(o + base);
        const uint32_t b = *reinterpret_cast<const uint32_t*>(dout + base);
        acc = __uint_as_float(a << 16) * __uint_as_float(b << 16) +
              __uint_as_float(a & 0xFFFF0000u) * __uint_as_float(b & 0xFFFF0000u);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) {
        dvec[row] = acc;
        lse2[row] = lse[(int64_t)z * N + n] * kLog2e;
    }
}

// ------------------------------------------------------------------ common
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
                 : "memory");
}

struct DevBwd {
    int Zq, g, N, Npad, causal;
    float scale, scale_log2;
    const float* lse2;  // [Zq][Npad]
    const float* dvec;  // [Zq][Npad]
    uint16_t *dq, *dk, *dv;
    int* status;
};

// ------------------------------------------------------------------ pass 2: dK, dV
template <int D>
struct KvCfg {
    static constexpr int kBK = 128;  // keys per CTA (TMEM lanes)
    static constexpr int kBQ = 64;   // query rows per step
    static constexpr int kChunks = D / 64;
    static constexpr int kKVBytes = kChunks * kBK * 128;
    static constexpr int kQBytes = kChunks * kBQ * 128;
    static constexpr int kStages = 4;
    static constexpr int kVecBytes = 2 * kBQ * 4;  // lse2 then dvec of one query tile
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kKVBytes;
    static constexpr int kOffQ = 2 * kKVBytes;
    static constexpr int kOffDO = kOffQ + kStages * kQBytes;
    static constexpr int kOffVec = kOffDO + kStages * kQBytes;
    static constexpr int kOffBar = kOffVec + kStages * kVecBytes;
    static constexpr int kNumBars = 1 + 2 * kStages + 2 + 2 + 1;
    static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;
    static constexpr uint32_t kColS = 0, kColDP = 64, kColPt0 = 128, kColPt1 = 160, kColDSt0 = 192, kColDSt1 = 224,
                              kColDV = 256, kColDK = 384;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
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
    const int kKvFull = 0, kQFull = 1, kQEmpty = 1 + C::kStages, kSFull = 1 + 2 * C::kStages, kSFree = kSFull + 1,
              kPReady = kSFree + 1, kOReady = kPReady + 2;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int Zk = p.Zq / p.g;
    const int kt = blockIdx.x / Zk;  // low key tiles carry the most causal work: they go first
    const int zk = blockIdx.x % Zk;
    const int n_qt = (p.N + C::kBQ - 1) / C::kBQ;
    const int qt_lo = p.causal ? (kt * C::kBK) / C::kBQ : 0;
    const int nq = n_qt - qt_lo;
    const int n_it = p.g * nq;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(BAR(kKvFull), 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(BAR(kQFull + s), 1);
            mbar_init(BAR(kQEmpty + s), 1);
        }
        mbar_init(BAR(kSFull), 1);
        mbar_init(BAR(kSFree), kSoftmaxWarps * 32);
        mbar_init(BAR(kPReady), kSoftmaxWarps * 32);
        mbar_init(BAR(kPReady + 1), kSoftmaxWarps * 32);
        mbar_init(BAR(kOReady), 1);
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    volatile int* abort_p = &abort_flag;

    if (n_it > 0 && warp == kProducerWarp && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_do);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        mbar_arrive_expect_tx(BAR(kKvFull), 2 * C::kKVBytes);
        for (int c = 0; c < C::kChunks; ++c) {
            tma_load_4d(sbase + C::kOffK + c * (C::kBK * 128), &tm_k, c * 64, zk, kt * C::kBK, 0, BAR(kKvFull));
            tma_load_4d(sbase + C::kOffV + c * (C::kBK * 128), &tm_v, c * 64, zk, kt * C::kBK, 0, BAR(kKvFull));
        }
        for (int it = 0; it < n_it; ++it) {
            const int s = it % C::kStages;
            const int zq = zk * p.g + it / nq;
            const int qt = qt_lo + it % nq;
            if (it >= C::kStages &&
                !mbar_wait(BAR(kQEmpty + s), ((it / C::kStages) - 1) & 1, abort_p, 21, p.status))
                break;
            mbar_arrive_expect_tx(BAR(kQFull + s), 2 * C::kQBytes + C::kVecBytes);
            for (int c = 0; c < C::kChunks; ++c) {
                tma_load_4d(sbase + C::kOffQ + s * C::kQBytes + c * (C::kBQ * 128), &tm_q, c * 64, zq, qt * C::kBQ, 0,
                            BAR(kQFull + s));
                tma_load_4d(sbase + C::kOffDO + s * C::kQBytes + c * (C::kBQ * 128), &tm_do, c * 64, zq, qt * C::kBQ,
                            0, BAR(kQFull + s));
            }
            const int64_t voff = (int64_t)zq * p.Npad + (int64_t)qt * C::kBQ;
            bulk_load(sbase + C::kOffVec + s * C::kVecBytes, p.lse2 + voff, C::kBQ * 4, BAR(kQFull + s));
            bulk_load(sbase + C::kOffVec + s * C::kVecBytes + C::kBQ * 4, p.dvec + voff, C::kBQ * 4, BAR(kQFull + s));
        }
    } else if (n_it > 0 && warp == kMmaWarp && lane == 0) {
        constexpr uint32_t kIdS = idesc_bf16(C::kBK, C::kBQ, 0, 0);  // S^T = K Q^T, dP^T = V dO^T
        constexpr uint32_t kIdG = idesc_bf16(C::kBK, D, 0, 1);       // dV += P^T dO, dK += dS^T Q
        // descriptors built once; each k-step adds its offset (address field, 16-byte units)
        const uint64_t dk0 = sdesc_sw128(sbase + C::kOffK, 16, 1024), dv0 = sdesc_sw128(sbase + C::kOffV, 16, 1024);
        auto issue_s = [&](int it) -> bool {
            const int s = it % C::kStages;
            if (!mbar_wait(BAR(kQFull + s), (it / C::kStages) & 1, abort_p, 22, p.status)) return false;
            tc_fence_after();
            const uint64_t dq0 = sdesc_sw128(sbase + C::kOffQ + s * C::kQBytes, 16, 1024);
            const uint64_t ddo0 = sdesc_sw128(sbase + C::kOffDO + s * C::kQBytes, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t a_off = ((kk / 4) * (C::kBK * 128) + (kk % 4) * 32) >> 4;
                const uint32_t b_off = ((kk / 4) * (C::kBQ * 128) + (kk % 4) * 32) >> 4;
                mma_ss(tmem + C::kColS, dk0 + a_off, dq0 + b_off, kIdS, kk > 0);
            }
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t a_off = ((kk / 4) * (C::kBK * 128) + (kk % 4) * 32) >> 4;
                const uint32_t b_off = ((kk / 4) * (C::kBQ * 128) + (kk % 4) * 32) >> 4;
                mma_ss(tmem + C::kColDP, dv0 + a_off, ddo0 + b_off, kIdS, kk > 0);
            }
            mma_commit(BAR(kSFull));
            return true;
        };
        bool ok = mbar_wait(BAR(kKvFull), 0, abort_p, 23, p.status);
        ok = ok && issue_s(0);
        for (int it = 0; ok && it < n_it; ++it) {
            const int s = it % C::kStages;
            if (it + 1 < n_it) {
                if (!mbar_wait(BAR(kSFree), it & 1, abort_p, 24, p.status)) break;
                if (!issue_s(it + 1)) break;
            }
            if (!mbar_wait(BAR(kPReady + (it & 1)), (it >> 1) & 1, abort_p, 25, p.status)) break;
            tc_fence_after();
            const uint64_t bdo = sdesc_sw128(sbase + C::kOffDO + s * C::kQBytes, C::kBQ * 128, 1024);
            const uint64_t bq = sdesc_sw128(sbase + C::kOffQ + s * C::kQBytes, C::kBQ * 128, 1024);
            const uint32_t pt = tmem + ((it & 1) ? C::kColPt1 : C::kColPt0);
            const uint32_t dst = tmem + ((it & 1) ? C::kColDSt1 : C::kColDSt0);
#pragma unroll
            for (int kk = 0; kk < C::kBQ / 16; ++kk)
                mma_ts(tmem + C::kColDV, pt + kk * 8, bdo + (kk * 2048 >> 4), kIdG, (it > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < C::kBQ / 16; ++kk)
                mma_ts(tmem + C::kColDK, dst + kk * 8, bq + (kk * 2048 >> 4), kIdG, (it > 0 || kk > 0) ? 1u : 0u);
            mma_commit(BAR(kQEmpty + s));
            if (it + 1 == n_it) mma_commit(BAR(kOReady));
        }
    } else if (warp < kSoftmaxWarps) {
        // ---------------------------------------------------------------- element-wise warps
        const int c = threadIdx.x;  // key row within the tile = TMEM lane
        const int key = kt * C::kBK + c;
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        bool ok = true;
        for (int it = 0; it < n_it; ++it) {
            const int s = it % C::kStages;
            const int qt = qt_lo + it % nq;
            if (!mbar_wait(BAR(kSFull), it & 1, abort_p, 26, p.status)) { ok = false; break; }
            tc_fence_after();
            uint32_t sa[32], sb[32], da[32], db[32];
            tmem_ld32(lane_base + C::kColS, sa);
            tmem_ld32(lane_base + C::kColS + 32, sb);
            tmem_ld32(lane_base + C::kColDP, da);
            tmem_ld32(lane_base + C::kColDP + 32, db);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(BAR(kSFree));
            if (!mbar_wait(BAR(kQFull + s), (it / C::kStages) & 1, abort_p, 27, p.status)) { ok = false; break; }
            const float* vl = reinterpret_cast<const float*>(smem + C::kOffVec + s * C::kVecBytes);
            const float* vd = vl + C::kBQ;
            const int q0 = qt * C::kBQ;
            const bool need_mask = p.causal && q0 < kt * C::kBK + C::kBK - 1;
            const int qmin_ok = key - q0;  // columns e with q0 + e >= key are visible
            uint32_t pk[32], dk[32];
#pragma unroll
            for (int e = 0; e < C::kBQ; e += 2) {
                float sv0 = __uint_as_float(e < 32 ? sa[e] : sb[e - 32]);
                float sv1 = __uint_as_float(e < 32 ? sa[e + 1] : sb[e - 31]);
                float dp0 = __uint_as_float(e < 32 ? da[e] : db[e - 32]);
                float dp1 = __uint_as_float(e < 32 ? da[e + 1] : db[e - 31]);
                float p0 = ex2_approx(fmaf(sv0, p.scale_log2, -vl[e]));
                float p1 = ex2_approx(fmaf(sv1, p.scale_log2, -vl[e + 1]));
                if (need_mask) {
                    if (e < qmin_ok) p0 = 0.f;
                    if (e + 1 < qmin_ok) p1 = 0.f;
                }
                const float ds0 = p0 * (dp0 - vd[e]);
                const float ds1 = p1 * (dp1 - vd[e + 1]);
                pk[e / 2] = pack_bf16(p0, p1);
                dk[e / 2] = pack_bf16(ds0, ds1);
            }
            const uint32_t pt = lane_base + ((it & 1) ? C::kColPt1 : C::kColPt0);
            const uint32_t dst = lane_base + ((it & 1) ? C::kColDSt1 : C::kColDSt0);
            tmem_st32(pt, pk);
            tmem_st32(dst, dk);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(BAR(kPReady + (it & 1)));
        }
        if (ok && n_it > 0) ok = mbar_wait(BAR(kOReady), 0, abort_p, 28, p.status);
        if (ok) {
            tc_fence_after();
            const bool valid = key < p.N;
            const int64_t base = ((int64_t)zk * p.N + key) * D;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const uint32_t col = half == 0 ? C::kColDV : C::kColDK;
                const float mul = half == 0 ? 1.f : p.scale;
                uint16_t* out = half == 0 ? p.dv : p.dk;
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
                    if (valid) {
                        uint4* dstp = reinterpret_cast<uint4*>(out + base + cc * 32);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            uint4 v;
                            v.x = pack_bf16(__uint_as_float(r[8 * e + 0]) * mul, __uint_as_float(r[8 * e + 1]) * mul);
                            v.y = pack_bf16(__uint_as_float(r[8 * e + 2]) * mul, __uint_as_float(r[8 * e + 3]) * mul);
                            v.z = pack_bf16(__uint_as_float(r[8 * e + 4]) * mul, __uint_as_float(r[8 * e + 5]) * mul);
                            v.w = pack_bf16(__uint_as_float(r[8 * e + 6]) * mul, __uint_as_float(r[8 * e + 7]) * mul);
                            dstp[e] = v;
                        }
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ pass 3: dQ
template <int D>
struct DqCfg {
    static constexpr int kBM = 128;  // query rows per CTA (TMEM lanes)
    static constexpr int kBN = 128;  // keys per step
    static constexpr int kChunks = D / 64;
    static constexpr int kTile = kChunks * 128 * 128;
    // K is held until dQ's product, V only until dP's: separate rings, K deeper
    static constexpr int kKStages = D == 64 ? 4 : 3;
    static constexpr int kVStages = D == 64 ? 3 : 2;
    static constexpr int kOffQ = 0;
    static constexpr int kOffDO = kTile;
    static constexpr int kOffK = 2 * kTile;
    static constexpr int kOffV = kOffK + kKStages * kTile;
    static constexpr int kOffBar = kOffV + kVStages * kTile;
    static constexpr int kNumBars = 1 + 2 * kKStages + 2 * kVStages + 2 + 2 + 1;
    static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;
    static constexpr uint32_t kColS = 0, kColDP = 128, kColDS0 = 256, kColDS1 = 320, kColDQ = 384;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
              const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v, const DevBwd p) {
    using C = DqCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + C::kNumBars * 8);
    __shared__ int abort_flag;
    const uint32_t bar0 = sbase + C::kOffBar;
    auto BAR = [&](int idx) { return bar0 + 8u * (uint32_t)idx; };
    const int kQFull = 0, kKFull = 1, kKEmpty = kKFull + C::kKStages, kVFull = kKEmpty + C::kKStages,
              kVEmpty = kVFull + C::kVStages, kSFull = kVEmpty + C::kVStages, kSFree = kSFull + 1,
              kDsReady = kSFree + 1, kOReady = kDsReady + 2;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int n_qt = (p.N + C::kBM - 1) / C::kBM;
    const int qt = n_qt - 1 - (int)(blockIdx.x / p.Zq);  // heaviest query tiles first
    const int zq = blockIdx.x % p.Zq;
    const int zk = zq / p.g;
    const int kv_end = p.causal ? min(p.N, (qt + 1) * C::kBM) : p.N;
    const int n_it = (kv_end + C::kBN - 1) / C::kBN;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(BAR(kQFull), 1);
        for (int s = 0; s < C::kKStages; ++s) {
            mbar_init(BAR(kKFull + s), 1);
            mbar_init(BAR(kKEmpty + s), 1);
        }
        for (int s = 0; s < C::kVStages; ++s) {
            mbar_init(BAR(kVFull + s), 1);
            mbar_init(BAR(kVEmpty + s), 1);
        }
        mbar_init(BAR(kSFull), 1);
        mbar_init(BAR(kSFree), kSoftmaxWarps * 32);
        mbar_init(BAR(kDsReady), kSoftmaxWarps * 32);
        mbar_init(BAR(kDsReady + 1), kSoftmaxWarps * 32);
        mbar_init(BAR(kOReady), 1);
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    volatile int* abort_p = &abort_flag;

    if (n_it > 0 && warp == kProducerWarp && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_do);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        mbar_arrive_expect_tx(BAR(kQFull), 2 * C::kTile);
        for (int c = 0; c < C::kChunks; ++c) {
            tma_load_4d(sbase + C::kOffQ + c * 16384, &tm_q, c * 64, zq, qt * C::kBM, 0, BAR(kQFull));
            tma_load_4d(sbase + C::kOffDO + c * 16384, &tm_do, c * 64, zq, qt * C::kBM, 0, BAR(kQFull));
        }
        for (int j = 0; j < n_it; ++j) {
            const int ks = j % C::kKStages, vs = j % C::kVStages;
            if (j >= C::kKStages &&
                !mbar_wait(BAR(kKEmpty + ks), ((j / C::kKStages) - 1) & 1, abort_p, 31, p.status))
                break;
            mbar_arrive_expect_tx(BAR(kKFull + ks), C::kTile);
            for (int c = 0; c < C::kChunks; ++c)
                tma_load_4d(sbase + C::kOffK + ks * C::kTile + c * 16384, &tm_k, c * 64, zk, j * C::kBN, 0,
                            BAR(kKFull + ks));
            if (j >= C::kVStages &&
                !mbar_wait(BAR(kVEmpty + vs), ((j / C::kVStages) - 1) & 1, abort_p, 38, p.status))
                break;
            mbar_arrive_expect_tx(BAR(kVFull + vs), C::kTile);
            for (int c = 0; c < C::kChunks; ++c)
                tma_load_4d(sbase + C::kOffV + vs * C::kTile + c * 16384, &tm_v, c * 64, zk, j * C::kBN, 0,
                            BAR(kVFull + vs));
        }
    } else if (n_it > 0 && warp == kMmaWarp && lane == 0) {
        constexpr uint32_t kIdS = idesc_bf16(C::kBM, C::kBN, 0, 0);  // S = Q K^T, dP = dO V^T
        constexpr uint32_t kIdG = idesc_bf16(C::kBM, D, 0, 1);       // dQ += dS K, K MN-major
        // descriptors built once; each k-step adds its offset (address field, 16-byte units)
        const uint64_t dq0 = sdesc_sw128(sbase + C::kOffQ, 16, 1024), ddo0 = sdesc_sw128(sbase + C::kOffDO, 16, 1024);
        auto issue_s = [&](int j) -> bool {
            const int ks = j % C::kKStages, vs = j % C::kVStages;
            if (!mbar_wait(BAR(kKFull + ks), (j / C::kKStages) & 1, abort_p, 32, p.status)) return false;
            if (!mbar_wait(BAR(kVFull + vs), (j / C::kVStages) & 1, abort_p, 39, p.status)) return false;
            tc_fence_after();
            const uint64_t dk0 = sdesc_sw128(sbase + C::kOffK + ks * C::kTile, 16, 1024);
            const uint64_t dv0 = sdesc_sw128(sbase + C::kOffV + vs * C::kTile, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = ((kk / 4) * 16384 + (kk % 4) * 32) >> 4;
                mma_ss(tmem + C::kColS, dq0 + off, dk0 + off, kIdS, kk > 0);
            }
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = ((kk / 4) * 16384 + (kk % 4) * 32) >> 4;
                mma_ss(tmem + C::kColDP, ddo0 + off, dv0 + off, kIdS, kk > 0);
            }
            mma_commit(BAR(kSFull));
            mma_commit(BAR(kVEmpty + vs));  // V_j is no longer needed once dP_j is done
            return true;
        };
        bool ok = mbar_wait(BAR(kQFull), 0, abort_p, 33, p.status);
        ok = ok && issue_s(0);
        for (int j = 0; ok && j < n_it; ++j) {
            const int ks = j % C::kKStages;
            if (j + 1 < n_it) {
                if (!mbar_wait(BAR(kSFree), j & 1, abort_p, 34, p.status)) break;
                if (!issue_s(j + 1)) break;
            }
            if (!mbar_wait(BAR(kDsReady + (j & 1)), (j >> 1) & 1, abort_p, 35, p.status)) break;
            tc_fence_after();
            const uint64_t bk = sdesc_sw128(sbase + C::kOffK + ks * C::kTile, 16384, 1024);
            const uint32_t ds = tmem + ((j & 1) ? C::kColDS1 : C::kColDS0);
#pragma unroll
            for (int kk = 0; kk < C::kBN / 16; ++kk)
                mma_ts(tmem + C::kColDQ, ds + kk * 8, bk + (kk * 2048 >> 4), kIdG, (j > 0 || kk > 0) ? 1u : 0u);
            mma_commit(BAR(kKEmpty + ks));
            if (j + 1 == n_it) mma_commit(BAR(kOReady));
        }
    } else if (warp < kSoftmaxWarps) {
        const int r = threadIdx.x;  // query row within the tile = TMEM lane
        const int q = qt * C::kBM + r;
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        const int64_t vrow = (int64_t)zq * p.Npad + q;  // q < Npad always
        const float lse2_r = p.lse2[vrow];
        const float dv_r = p.dvec[vrow];
        bool ok = true;
        for (int j = 0; j < n_it; ++j) {
            if (!mbar_wait(BAR(kSFull), j & 1, abort_p, 36, p.status)) { ok = false; break; }
            tc_fence_after();
            const int key0 = j * C::kBN;
            // visible columns: key0 + c <= q (causal) and key0 + c < N
            int climit = p.N - 1 - key0;
            if (p.causal) climit = min(climit, q - key0);
            const bool need_mask = climit < C::kBN - 1;
            uint32_t dsp[64];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t sa[32], sb[32], da[32], db[32];
                tmem_ld32(lane_base + C::kColS + half * 64, sa);
                tmem_ld32(lane_base + C::kColS + half * 64 + 32, sb);
                tmem_ld32(lane_base + C::kColDP + half * 64, da);
                tmem_ld32(lane_base + C::kColDP + half * 64 + 32, db);
                tmem_wait_ld();
                if (half == 1) {
                    tc_fence_before();
                    mbar_arrive(BAR(kSFree));
                }
#pragma unroll
                for (int e = 0; e < 64; e += 2) {
                    const int col = half * 64 + e;
                    const float sv0 = __uint_as_float(e < 32 ? sa[e] : sb[e - 32]);
                    const float sv1 = __uint_as_float(e < 32 ? sa[e + 1] : sb[e - 31]);
                    const float dp0 = __uint_as_float(e < 32 ? da[e] : db[e - 32]);
                    const float dp1 = __uint_as_float(e < 32 ? da[e + 1] : db[e - 31]);
                    float p0 = ex2_approx(fmaf(sv0, p.scale_log2, -lse2_r));
                    float p1 = ex2_approx(fmaf(sv1, p.scale_log2, -lse2_r));
                    if (need_mask) {
                        if (col > climit) p0 = 0.f;
                        if (col + 1 > climit) p1 = 0.f;
                    }
                    dsp[half * 32 + e / 2] = pack_bf16(p0 * (dp0 - dv_r), p1 * (dp1 - dv_r));
                }
            }
            const uint32_t ds = lane_base + ((j & 1) ? C::kColDS1 : C::kColDS0);
            uint32_t lo[32], hi[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                lo[e] = dsp[e];
                hi[e] = dsp[32 + e];
            }
            tmem_st32(ds, lo);
            tmem_st32(ds + 32, hi);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(BAR(kDsReady + (j & 1)));
        }
        if (ok && n_it > 0) ok = mbar_wait(BAR(kOReady), 0, abort_p, 37, p.status);
        if (ok) {
            tc_fence_after();
            const bool valid = q < p.N;
            const int64_t base = ((int64_t)zq * p.N + q) * D;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t rr[32];
                if (n_it > 0) {
                    tmem_ld32(lane_base + C::kColDQ + cc * 32, rr);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) rr[e] = 0u;
                }
                if (valid) {
                    uint4* dstp = reinterpret_cast<uint4*>(p.dq + base + cc * 32);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        uint4 v;
                        v.x = pack_bf16(__uint_as_float(rr[8 * e + 0]) * p.scale, __uint_as_float(rr[8 * e + 1]) * p.scale);
                        v.y = pack_bf16(__uint_as_float(rr[8 * e + 2]) * p.scale, __uint_as_float(rr[8 * e + 3]) * p.scale);
                        v.z = pack_bf16(__uint_as_float(rr[8 * e + 4]) * p.scale, __uint_as_float(rr[8 * e + 5]) * p.scale);
                        v.w = pack_bf16(__uint_as_float(rr[8 * e + 6]) * p.scale, __uint_as_float(rr[8 * e + 7]) * p.scale);
                        dstp[e] = v;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

struct BwdMaps {
    CUtensorMap q, dout, k, v;
};

template <int D>
bool make_bwd_maps(const BwdParams& b, int q_rows, BwdMaps* m) {
    const int Zk = b.Zq / b.g;
    const int64_t nd = (int64_t)b.N * D;
    Tensor4 tq{const_cast<void*>(b.q), nd, D, nd * b.Zq, b.Zq, b.N, 1};
    Tensor4 tdo{const_cast<void*>(b.dout), nd, D, nd * b.Zq, b.Zq, b.N, 1};
    Tensor4 tk{const_cast<void*>(b.k), nd, D, nd * Zk, Zk, b.N, 1};
    Tensor4 tv{const_cast<void*>(b.v), nd, D, nd * Zk, Zk, b.N, 1};
    return make_tmap_bf16(&m->q, tq, D, q_rows) && make_tmap_bf16(&m->dout, tdo, D, q_rows) &&
           make_tmap_bf16(&m->k, tk, D, 128) && make_tmap_bf16(&m->v, tv, D, 128);
}

DevBwd dev_params(const BwdParams& b) {
    const int Npad = (b.N + 127) / 128 * 128;
    DevBwd p;
    p.Zq = b.Zq;
    p.g = b.g;
    p.N = b.N;
    p.Npad = Npad;
    p.causal = b.causal;
    p.scale = b.scale;
    p.scale_log2 = b.scale * kLog2e;
    p.dvec = b.dvec;
    p.lse2 = b.dvec + (size_t)b.Zq * Npad;
    p.dq = static_cast<uint16_t*>(b.dq);
    p.dk = static_cast<uint16_t*>(b.dk);
    p.dv = static_cast<uint16_t*>(b.dv);
    p.status = b.status;
    return p;
}

template <int D>
cudaError_t pre_t(const BwdParams& b, cudaStream_t stream) {
    const DevBwd p = dev_params(b);
    const int64_t rows = (int64_t)b.Zq * p.Npad;
    bwd_pre_kernel<D><<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(
        static_cast<const uint16_t*>(b.o), static_cast<const uint16_t*>(b.dout), b.lse, const_cast<float*>(p.dvec),
        const_cast<float*>(p.lse2), b.Zq, b.N, p.Npad);
    return cudaGetLastError();
}

template <int D>
cudaError_t dkdv_t(const BwdParams& b, cudaStream_t stream) {
    BwdMaps m;
    if (!make_bwd_maps<D>(b, KvCfg<D>::kBQ, &m)) return cudaErrorInvalidValue;
    auto kern = dkdv_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, KvCfg<D>::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int n_kt = (b.N + 127) / 128;
    kern<<<(unsigned)(n_kt * (b.Zq / b.g)), kThreads, KvCfg<D>::kSmemBytes, stream>>>(m.q, m.dout, m.k, m.v,
                                                                                      dev_params(b));
    return cudaGetLastError();
}

template <int D>
cudaError_t dq_t(const BwdParams& b, cudaStream_t stream) {
    BwdMaps m;
    if (!make_bwd_maps<D>(b, DqCfg<D>::kBM, &m)) return cudaErrorInvalidValue;
    auto kern = dq_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DqCfg<D>::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int n_qt = (b.N + 127) / 128;
    kern<<<(unsigned)(n_qt * b.Zq), kThreads, DqCfg<D>::kSmemBytes, stream>>>(m.q, m.dout, m.k, m.v, dev_params(b));
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_pre(const BwdParams& b, cudaStream_t stream) {
    return b.d == 64 ? pre_t<64>(b, stream) : (b.d == 128 ? pre_t<128>(b, stream) : cudaErrorInvalidValue);
}
cudaError_t launch_bwd_dkdv(const BwdParams& b, cudaStream_t stream) {
    return b.d == 64 ? dkdv_t<64>(b, stream) : (b.d == 128 ? dkdv_t<128>(b, stream) : cudaErrorInvalidValue);
}
cudaError_t launch_bwd_dq(const BwdParams& b, cudaStream_t stream) {
    return b.d == 64 ? dq_t<64>(b, stream) : (b.d == 128 ? dq_t<128>(b, stream) : cudaErrorInvalidValue);
}

}  // namespace usp

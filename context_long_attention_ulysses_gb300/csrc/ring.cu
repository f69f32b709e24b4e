// Ring attention support: exact log-sum-exp merge of partial attentions.
//
// "Context Parallelism" (ultralytics.com), section "So funktioniert
// Kontextparallelitaet": in ring attention every device computes partial
// attention against the KV block it holds, passes the block on and repeats
// until the whole sequence is covered; the result equals full-sequence
// attention.  Two partials over disjoint key sets, each normalised over its
// own keys and carrying its LSE, combine exactly as
//   lse = ln(e^{lse_a} + e^{lse_b}),  o = e^{lse_a - lse} o_a + e^{lse_b - lse} o_b.
// These kernels are HBM-bound element-wise passes: one warp per row, 16-byte
// vectors, full-precision expf/logf.
#include <cmath>

#include "kernels.h"

namespace usp {

namespace {

__global__ void __launch_bounds__(256) lse_merge_kernel(int64_t rows, int d, const float* o_a, const float* lse_a,
                                                        const float* o_b, const float* lse_b, float* o,
                                                        float* lse) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    if (row >= rows) return;
    const float la = lse_a[row], lb = lse_b[row];
    float wa, wb, l;
    if (la == -INFINITY && lb == -INFINITY) {
        wa = wb = 0.f;
        l = -INFINITY;
    } else {
        const float m = fmaxf(la, lb);
        l = m + logf(expf(la - m) + expf(lb - m));
        wa = expf(la - l);
        wb = expf(lb - l);
    }
    // every lane has read lse_a/lse_b before lane 0 may overwrite them in place
    __syncwarp();
    const int nv = d / 4;
    const float4* a4 = reinterpret_cast<const float4*>(o_a + row * d);
    const float4* b4 = reinterpret_cast<const float4*>(o_b + row * d);
    float4* o4 = reinterpret_cast<float4*>(o + row * d);
    for (int c = lane; c < nv; c += 32) {
        const float4 a = a4[c], b = b4[c];
        float4 r;
        r.x = (wa == 0.f ? 0.f : wa * a.x) + (wb == 0.f ? 0.f : wb * b.x);
        r.y = (wa == 0.f ? 0.f : wa * a.y) + (wb == 0.f ? 0.f : wb * b.y);
        r.z = (wa == 0.f ? 0.f : wa * a.z) + (wb == 0.f ? 0.f : wb * b.z);
        r.w = (wa == 0.f ? 0.f : wa * a.w) + (wb == 0.f ? 0.f : wb * b.w);
        o4[c] = r;
    }
    if (lane == 0) lse[row] = l;
}

__global__ void f32_to_bf16_kernel(const float4* __restrict__ src, uint2* __restrict__ dst, int64_t n4) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
        const float4 f = src[i];
        uint32_t lo, hi;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(lo) : "f"(f.y), "f"(f.x));
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(hi) : "f"(f.w), "f"(f.z));
        dst[i] = make_uint2(lo, hi);
    }
}

__global__ void fill_f32_kernel(float* dst, float value, int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = value;
}

unsigned grid_for(int64_t n, int threads) {
    int64_t b = (n + threads - 1) / threads;
    const int64_t cap = 152 * 16;
    return (unsigned)(b < 1 ? 1 : (b > cap ? cap : b));
}

}  // namespace

cudaError_t launch_lse_merge(int64_t rows, int d, const float* o_a, const float* lse_a, const float* o_b,
                             const float* lse_b, float* o, float* lse, cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    const int64_t blocks = (rows + 7) / 8;
    lse_merge_kernel<<<(unsigned)blocks, 256, 0, stream>>>(rows, d, o_a, lse_a, o_b, lse_b, o, lse);
    return cudaGetLastError();
}

cudaError_t launch_f32_to_bf16(const float* src, void* dst, int64_t n, cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    const int64_t n4 = n / 4;
    f32_to_bf16_kernel<<<grid_for(n4, 256), 256, 0, stream>>>(reinterpret_cast<const float4*>(src),
                                                              static_cast<uint2*>(dst), n4);
    return cudaGetLastError();
}

cudaError_t launch_fill_f32(float* dst, float value, int64_t n, cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    fill_f32_kernel<<<grid_for(n, 256), 256, 0, stream>>>(dst, value, n);
    return cudaGetLastError();
}

}  // namespace usp

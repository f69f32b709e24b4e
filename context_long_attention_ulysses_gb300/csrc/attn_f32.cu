// Float32 attention forward on CUDA cores.
//
// Causal (or full) scaled dot product attention as in the code example of
// "Context Parallelism" (ultralytics.com), section "Praktische Anwendung und
// Kompromisse", for float32 inputs that must match float64 to ~1e-5: true
// FP32 FMA arithmetic (tensor-core TF32 would not), one thread per query
// row, an online softmax over 32-key tiles staged in shared memory, and the
// natural-log LSE of each row.
#include <cmath>

#include "kernels.h"

namespace usp {

namespace {

constexpr int kRows = 64;   // query rows (threads) per CTA
constexpr int kKeys = 32;   // keys per shared-memory tile

template <int D>
__global__ void __launch_bounds__(kRows) attn_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                                                         const float* __restrict__ v, float* __restrict__ o,
                                                         float* __restrict__ lse, int g, int N, int causal,
                                                         float scale) {
    __shared__ float sK[kKeys][D];
    __shared__ float sV[kKeys][D];
    const int z = blockIdx.y;
    const int zk = z / g;
    const int row0 = blockIdx.x * kRows;
    const int i = row0 + threadIdx.x;
    const bool valid = i < N;
    const float* qrow = q + ((size_t)z * N + (valid ? i : 0)) * D;
    const float* kz = k + (size_t)zk * N * D;
    const float* vz = v + (size_t)zk * N * D;

    float qr[D];
#pragma unroll
    for (int c = 0; c < D; ++c) qr[c] = qrow[c] * scale;
    float acc[D];
#pragma unroll
    for (int c = 0; c < D; ++c) acc[c] = 0.f;
    float m = -INFINITY, l = 0.f;

    int key_end = N;
    if (causal) key_end = min(N, row0 + kRows);
    for (int j0 = 0; j0 < key_end; j0 += kKeys) {
        __syncthreads();
        for (int e = threadIdx.x; e < kKeys * D; e += kRows) {
            const int jj = e / D, c = e % D;
            const int j = j0 + jj;
            sK[jj][c] = j < N ? kz[(size_t)j * D + c] : 0.f;
            sV[jj][c] = j < N ? vz[(size_t)j * D + c] : 0.f;
        }
        __syncthreads();
        if (!valid) continue;
        const int jmax = min(kKeys, (causal ? i + 1 : N) - j0);
        for (int jj = 0; jj < jmax; ++jj) {
            float s = 0.f;
#pragma unroll
            for (int c = 0; c < D; ++c) s = fmaf(qr[c], sK[jj][c], s);
            if (s > m) {
                const float alpha = expf(m - s);
                l *= alpha;
#pragma unroll
                for (int c = 0; c < D; ++c) acc[c] *= alpha;
                m = s;
            }
            const float p = expf(s - m);
            l += p;
#pragma unroll
            for (int c = 0; c < D; ++c) acc[c] = fmaf(p, sV[jj][c], acc[c]);
        }
    }
    if (!valid) return;
    const float inv = 1.f / l;
    float* orow = o + ((size_t)z * N + i) * D;
#pragma unroll
    for (int c = 0; c < D; ++c) orow[c] = acc[c] * inv;
    lse[(size_t)z * N + i] = m + logf(l);
}

}  // namespace

cudaError_t launch_attn_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse, int Zq,
                                int g, int N, int d, int causal, float scale, cudaStream_t stream) {
    dim3 grid((unsigned)((N + kRows - 1) / kRows), (unsigned)Zq);
    if (d == 64)
        attn_f32_kernel<64><<<grid, kRows, 0, stream>>>(q, k, v, o, lse, g, N, causal, scale);
    else if (d == 128)
        attn_f32_kernel<128><<<grid, kRows, 0, stream>>>(q, k, v, o, lse, g, N, causal, scale);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace usp

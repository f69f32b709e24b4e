// Ulysses all-to-all as an on-device layout remap.
//
// "Million-Token-Kontexte im Training" (bytewire.ai), section "Ulysses: Die
// Sequenz als Verteilungseinheit": before attention Q, K, V are exchanged by
// an all-to-all so that each device sees the whole sequence; "Context
// Parallelism" (ultralytics.com), section "So funktioniert": token-local
// layers afterwards run on the local shard, hence the inverse remap.
//
// With the P ranks living on one GPU the exchange is a permutation of
// d-element rows (128-512 contiguous bytes):
//   sequence side row (p, b, n', h)  <->  head side row (r, b, h', n)
//   n = p*N/P + n',  h = r*Hx/P + h'.
// Each CTA owns one head-side (r, b, h') and a run of tokens n, so the
// head-side accesses are one contiguous run and the sequence-side accesses
// are whole rows at stride Hx*row_bytes.  Data moves in 16-byte vectors,
// four per thread in flight, with streaming cache hints (each byte is touched
// once).
#include "kernels.h"

namespace usp {

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

template <int CHUNKS>  // 16-byte chunks per row
__global__ void __launch_bounds__(kThreads) remap_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                         int dir, int B, int Hx, int N, int P) {
    constexpr int kRowsPerPass = kThreads / CHUNKS;
    constexpr int kRowsPerBlock = kRowsPerPass * kUnroll;
    const int Hl = Hx / P;
    const int Np = N / P;
    const int hr = blockIdx.y;  // (r*B + b)*Hl + hl
    const int r = hr / (B * Hl);
    const int rem = hr - r * (B * Hl);
    const int b = rem / Hl;
    const int hl = rem - b * Hl;
    const int h = r * Hl + hl;
    const int chunk = threadIdx.x % CHUNKS;
    const int row_in_pass = threadIdx.x / CHUNKS;
    const int n_base = blockIdx.x * kRowsPerBlock;

    uint4 buf[kUnroll];
    size_t dst_off[kUnroll];
    bool live[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const int n = n_base + u * kRowsPerPass + row_in_pass;
        live[u] = n < N;
        const int nn = live[u] ? n : 0;
        const int p = nn / Np;
        const int npr = nn - p * Np;
        const size_t head_row = (size_t)hr * (size_t)N + (size_t)nn;
        const size_t seq_row = ((size_t)(p * B + b) * (size_t)Np + (size_t)npr) * (size_t)Hx + (size_t)h;
        const size_t s_row = dir == 0 ? seq_row : head_row;
        const size_t d_row = dir == 0 ? head_row : seq_row;
        dst_off[u] = d_row * CHUNKS + chunk;
        if (live[u]) buf[u] = __ldcs(src + s_row * CHUNKS + chunk);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
        if (live[u]) __stcs(dst + dst_off[u], buf[u]);
}

template <int CHUNKS>
cudaError_t launch_t(int dir, const void* src, void* dst, int B, int Hx, int N, int P, cudaStream_t s) {
    constexpr int kRowsPerBlock = (kThreads / CHUNKS) * kUnroll;
    dim3 grid((unsigned)((N + kRowsPerBlock - 1) / kRowsPerBlock), (unsigned)(B * Hx));
    remap_kernel<CHUNKS><<<grid, kThreads, 0, s>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst), dir,
                                                   B, Hx, N, P);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_remap(int dir, const void* src, void* dst, int B, int Hx, int N, int P, int row_bytes,
                         cudaStream_t stream) {
    switch (row_bytes) {
        case 64: return launch_t<4>(dir, src, dst, B, Hx, N, P, stream);
        case 128: return launch_t<8>(dir, src, dst, B, Hx, N, P, stream);
        case 256: return launch_t<16>(dir, src, dst, B, Hx, N, P, stream);
        case 512: return launch_t<32>(dir, src, dst, B, Hx, N, P, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace usp

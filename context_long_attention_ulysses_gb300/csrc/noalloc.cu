// Attention backward for callers that cannot allocate device memory.
//
// The backward needs a caller-provided workspace: the deterministic
// three-pass backward (usp_attn_bwd_deterministic) 40 bytes per query row,
// rows padded to 128-row tiles.  Some callers cannot obtain one: code running inside a
// framework that owns every device allocation and forbids raw cudaMalloc,
// plugins loaded into a host process that has no allocator to hand them, or
// code that must not touch the allocator at all once set up.  This file gives
// them usp_attn_bwd_noalloc, the deterministic backward with a fixed scratch
// array compiled into the library as its workspace.
//
// The scratch is a file-scope __device__ array of USP_NOALLOC_SCRATCH_BYTES.
// Every GPU that loads the library holds it until the process exits.  Host
// code cannot use the array's name as a device address (it names a host-side
// stand-in), so the address is looked up with cudaGetSymbolAddress once per
// device, with that device current, on the first call made on it, and kept
// for the life of the process: after cudaDeviceReset the array may sit at a
// new address, which this cache does not see (the library's status word is
// looked up the same way).
#include <mutex>

#include "../../include/usp.h"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = USP_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up on first use).
usp_status scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return USP_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return USP_ERR_CUDA;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return USP_OK;
}

}  // namespace

extern "C" usp_status usp_attn_bwd_noalloc(const usp_problem* p, const void* q, const void* k, const void* v,
                                           const void* o, const float* lse, const void* dout, void* dq, void* dk,
                                           void* dv, usp_stream stream) {
    // Every argument check, then the size check, before any CUDA call: a problem the backward does
    // not support, or one the scratch cannot hold, is refused with nothing looked up or enqueued.
    usp_status st = usp::attn_bwd_check(p, q, k, v, o, lse, dout, dq, dk, dv);
    if (st != USP_OK) return st;
    const size_t need = usp_attn_bwd_deterministic_workspace_size(p);
    if (need == 0) return USP_OK;  // an empty problem: nothing to do
    if (need > kScratchBytes) return USP_ERR_WORKSPACE;
    void* scratch = nullptr;
    st = scratch_address(&scratch);
    if (st != USP_OK) return st;
    // The backward's first pass rewrites every scratch entry the later passes
    // read, so the previous call's contents never matter.
    return usp_attn_bwd_deterministic(p, q, k, v, o, lse, dout, dq, dk, dv, scratch, kScratchBytes, stream);
}

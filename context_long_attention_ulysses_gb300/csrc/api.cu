// C-ABI layer of libusp: host-side validation, tensor-map encoding and
// dispatch to the kernels.  Nothing is enqueued unless every argument checks
// out; the library never allocates device memory.
#include <cmath>
#include <cstring>
#include <initializer_list>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include <cudaTypedefs.h>

#include "../../include/usp.h"
#include "kernels.h"

namespace usp {

// Device status word (see ptx.cuh); one per device context.
__device__ int g_status_word = 0;

namespace {

constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices] = {};
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Address of the status word on the current device (looked up once per device).
int* status_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int*>(p);
    }
    return g_status_ptr[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    return g_encode;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_size(int dtype) { return dtype == USP_F32 ? 4 : (dtype == USP_BF16 ? 2 : 0); }

// Sizes and divisibility shared by every problem-based entry point.  The
// Ulysses path splits heads over ranks (Hq, Hkv divisible by P); ring mode
// keeps every head on every rank and only splits tokens.
usp_status check_problem(const usp_problem* p, bool split_heads = true) {
    if (!p) return USP_ERR_INVALID_ARG;
    if (p->B < 0 || p->N < 0 || p->Hq < 1 || p->Hkv < 1 || p->P < 1) return USP_ERR_INVALID_ARG;
    if (p->N % p->P != 0 || p->Hq % p->Hkv != 0) return USP_ERR_INVALID_ARG;
    if (split_heads && (p->Hq % p->P != 0 || p->Hkv % p->P != 0)) return USP_ERR_INVALID_ARG;
    if (p->dtype != USP_F32 && p->dtype != USP_BF16) return USP_ERR_INVALID_ARG;
    if (p->d < 1) return USP_ERR_INVALID_ARG;
    if (!(p->scale >= 0.f) || std::isinf(p->scale)) return USP_ERR_INVALID_ARG;
    if ((int64_t)p->B * p->Hq > 65535) return USP_ERR_UNSUPPORTED;  // grid.y limit
    return USP_OK;
}

float eff_scale(const usp_problem* p) { return p->scale == 0.f ? 1.0f / std::sqrt((float)p->d) : p->scale; }

bool empty(const usp_problem* p) { return p->B == 0 || p->N == 0; }

usp_status cuda_status(cudaError_t e) { return e == cudaSuccess ? USP_OK : USP_ERR_CUDA; }

// ---------------------------------------------------------------- tracing
// When enabled, every kernel launch is bracketed by two CUDA events on its
// stream; usp_trace_report() resolves them into per-kernel totals.
struct TraceSlot {
    const char* name;
    cudaEvent_t a, b;
};
struct TraceAcc {
    int64_t launches = 0;
    double ms = 0.0;
};
std::mutex g_trace_mu;
bool g_trace_on = false;
std::vector<TraceSlot> g_trace_pending;
std::vector<cudaEvent_t> g_trace_pool;
std::map<std::string, TraceAcc> g_trace_acc;

cudaEvent_t trace_event() {
    if (!g_trace_pool.empty()) {
        cudaEvent_t e = g_trace_pool.back();
        g_trace_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

template <class F>
cudaError_t traced(const char* name, cudaStream_t s, F&& launch) {
    std::unique_lock<std::mutex> lock(g_trace_mu);
    if (!g_trace_on) {
        lock.unlock();
        return launch();
    }
    cudaEvent_t a = trace_event(), b = trace_event();
    if (!a || !b) return cudaErrorMemoryAllocation;
    cudaEventRecord(a, s);
    cudaError_t e = launch();
    cudaEventRecord(b, s);
    g_trace_pending.push_back({name, a, b});
    return e;
}

}  // namespace

bool make_tmap_bf16(CUtensorMap* map, const Tensor4& t, int d, int box_rows) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)t.n_head, (cuuint64_t)t.n_tok, (cuuint64_t)t.n_outer};
    cuuint64_t strides[3] = {(cuuint64_t)t.s_head * 2, (cuuint64_t)t.s_tok * 2, (cuuint64_t)t.s_outer * 2};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, t.ptr, dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace usp

using namespace usp;

extern "C" {

const char* usp_status_string(usp_status s) {
    switch (s) {
        case USP_OK: return "USP_OK";
        case USP_ERR_INVALID_ARG: return "USP_ERR_INVALID_ARG";
        case USP_ERR_UNSUPPORTED: return "USP_ERR_UNSUPPORTED";
        case USP_ERR_MISALIGNED: return "USP_ERR_MISALIGNED";
        case USP_ERR_WORKSPACE: return "USP_ERR_WORKSPACE";
        case USP_ERR_CUDA: return "USP_ERR_CUDA";
        case USP_ERR_TIMEOUT: return "USP_ERR_TIMEOUT";
    }
    return "USP_ERR_UNKNOWN";
}

const char* usp_build_info(void) { return "libusp 0.1 sm_103a (tcgen05/TMEM/TMA attention, on-device all-to-all)"; }

usp_status usp_device_status(usp_stream stream) {
    int* sp = status_ptr();
    if (!sp) return USP_ERR_CUDA;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return USP_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, sp, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return USP_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpy(sp, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return USP_ERR_CUDA;
        return USP_ERR_TIMEOUT;
    }
    return USP_OK;
}

usp_status usp_diag_wait_timeout(usp_stream stream) {
    int* sp = status_ptr();
    if (!sp) return USP_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return cuda_status(traced("diag_wait_timeout", s, [&] { return launch_wait_timeout_probe(sp, s); }));
}

usp_status usp_diag_raise_status(usp_stream stream) {
    int* sp = status_ptr();
    if (!sp) return USP_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return cuda_status(traced("diag_raise_status", s, [&] { return launch_raise_status(sp, s); }));
}

static usp_status a2a(int dir, const usp_problem* p, int Hx, const void* src, void* dst, usp_stream stream) {
    usp_status st = check_problem(p);
    if (st != USP_OK) return st;
    if (Hx != p->Hq && Hx != p->Hkv) return USP_ERR_INVALID_ARG;
    const int row_bytes = p->d * elem_size(p->dtype);
    if (row_bytes != 64 && row_bytes != 128 && row_bytes != 256 && row_bytes != 512) return USP_ERR_UNSUPPORTED;
    if (empty(p)) return USP_OK;
    if (!aligned16(src) || !aligned16(dst)) return USP_ERR_MISALIGNED;
    const size_t bytes = (size_t)p->B * Hx * (size_t)p->N * row_bytes;
    const char* sb = static_cast<const char*>(src);
    const char* tb = static_cast<const char*>(dst);
    if (sb < tb + bytes && tb < sb + bytes) return USP_ERR_INVALID_ARG;  // overlap
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return cuda_status(traced(dir == 0 ? "a2a_seq2head" : "a2a_head2seq", s, [&] {
        return launch_remap(dir, src, dst, p->B, Hx, p->N, p->P, row_bytes, s);
    }));
}

usp_status usp_a2a_seq2head(const usp_problem* p, int Hx, const void* src, void* dst, usp_stream stream) {
    return a2a(0, p, Hx, src, dst, stream);
}

usp_status usp_a2a_head2seq(const usp_problem* p, int Hx, const void* src, void* dst, usp_stream stream) {
    return a2a(1, p, Hx, src, dst, stream);
}

// Head-sharded forward parameters: every (rank, batch, local head) is one
// "head slot"; slots are contiguous [N][d] blocks.
static FwdParams head_sharded_fwd(const usp_problem* p, const void* q, const void* k, const void* v, void* o,
                                  float* lse, int* status) {
    FwdParams f{};
    const int Zq = p->B * p->Hq;  // = P * B * Hq/P
    const int Zk = p->B * p->Hkv;
    const int64_t nd = (int64_t)p->N * p->d;
    f.q = Tensor4{const_cast<void*>(q), nd, p->d, nd * Zq, Zq, p->N, 1};
    f.k = Tensor4{const_cast<void*>(k), nd, p->d, nd * Zk, Zk, p->N, 1};
    f.v = Tensor4{const_cast<void*>(v), nd, p->d, nd * Zk, Zk, p->N, 1};
    f.d = p->d;
    f.g = p->Hq / p->Hkv;
    f.n_heads = Zq;
    f.n_outer = 1;
    f.q_len = p->N;
    f.kv_len = p->N;
    f.ring_i0 = 0;
    f.ring_t = 0;
    f.ring_p = 1;
    f.bsz = 1;
    f.np = 0;
    f.causal = p->causal ? 1 : 0;
    f.scale = eff_scale(p);
    f.o_bf16 = o;
    f.o_f32 = nullptr;
    f.o_s_head = nd;
    f.o_s_tok = p->d;
    f.o_s_outer = nd * Zq;
    f.lse = lse;
    f.l_s_head = p->N;
    f.l_s_tok = 1;
    f.l_s_outer = (int64_t)p->N * Zq;
    f.status = status;
    return f;
}

usp_status usp_attn_fwd(const usp_problem* p, const void* q, const void* k, const void* v, void* o, float* lse,
                        usp_stream stream) {
    usp_status st = check_problem(p);
    if (st != USP_OK) return st;
    if (p->d != 64 && p->d != 128) return USP_ERR_UNSUPPORTED;
    if (empty(p)) return USP_OK;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return USP_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int Zq = p->B * p->Hq;
    if (p->dtype == USP_F32)
        return cuda_status(traced("attn_fwd_f32", s, [&] {
            return launch_attn_fwd_f32(static_cast<const float*>(q), static_cast<const float*>(k),
                                       static_cast<const float*>(v), static_cast<float*>(o), lse, Zq, p->Hq / p->Hkv,
                                       p->N, p->d, p->causal ? 1 : 0, eff_scale(p), s);
        }));
    int* sp = status_ptr();
    if (!sp) return USP_ERR_CUDA;
    FwdParams f = head_sharded_fwd(p, q, k, v, o, lse, sp);
    return cuda_status(traced("attn_fwd", s, [&] { return launch_attn_fwd_bf16(f, s); }));
}

// Backward workspace rows: per query row, rows padded to whole 128-row tiles, D_i and lse_i*log2(e)
// (float32), then -lse_i/scale and -D_i each as a 16-byte row of three bf16 numbers.
static size_t bwd_rows_bytes(const usp_problem* p) {
    const size_t npad = ((size_t)p->N + 127) / 128 * 128;
    return (((size_t)p->B * p->Hq * npad * (2 * sizeof(float) + 2 * 16)) + 255) & ~(size_t)255;
}

// The one-pass backward adds the float32 dQ accumulator: d values per padded query row.
size_t usp_attn_bwd_workspace_size(const usp_problem* p) {
    if (check_problem(p) != USP_OK) return 0;
    const size_t npad = ((size_t)p->N + 127) / 128 * 128;
    return bwd_rows_bytes(p) + (size_t)p->B * p->Hq * npad * (size_t)p->d * sizeof(float);
}

size_t usp_attn_bwd_deterministic_workspace_size(const usp_problem* p) {
    if (check_problem(p) != USP_OK) return 0;
    return bwd_rows_bytes(p);
}

}  // extern "C"

namespace usp {
usp_status attn_bwd_check(const usp_problem* p, const void* q, const void* k, const void* v, const void* o,
                          const float* lse, const void* dout, const void* dq, const void* dk, const void* dv) {
    usp_status st = check_problem(p);
    if (st != USP_OK) return st;
    if (p->d != 64 && p->d != 128) return USP_ERR_UNSUPPORTED;
    if (p->dtype != USP_BF16) return USP_ERR_UNSUPPORTED;
    if (empty(p)) return USP_OK;
    const void* ptrs[] = {q, k, v, o, lse, dout, dq, dk, dv};
    for (const void* ptr : ptrs)
        if (!aligned16(ptr)) return USP_ERR_MISALIGNED;
    return USP_OK;
}
}  // namespace usp

extern "C" {

// Head-sharded buffers as Z = B*Hq query heads (Z/g KV heads) of N tokens, one outer index.
static BwdParams head_sharded_bwd(const usp_problem* p, const void* q, const void* k, const void* v, const void* o,
                                  const float* lse, const void* dout, void* dq, void* dk, void* dv, void* ws,
                                  int* sp) {
    const int Z = p->B * p->Hq, Zk = p->B * p->Hkv, d = p->d, N = p->N;
    const int64_t nd = (int64_t)N * d;
    BwdParams b{};
    b.q = Tensor4{const_cast<void*>(q), nd, d, nd * Z, Z, N, 1};
    b.o = Tensor4{const_cast<void*>(o), nd, d, nd * Z, Z, N, 1};
    b.dout = Tensor4{const_cast<void*>(dout), nd, d, nd * Z, Z, N, 1};
    b.k = Tensor4{const_cast<void*>(k), nd, d, nd * Zk, Zk, N, 1};
    b.v = Tensor4{const_cast<void*>(v), nd, d, nd * Zk, Zk, N, 1};
    b.lse = lse;
    b.l_s_head = N;
    b.l_s_tok = 1;
    b.l_s_outer = (int64_t)Z * N;
    b.ws = static_cast<float*>(ws);
    b.n_z = Z;
    b.dq = dq; b.dk = dk; b.dv = dv;
    b.d = d;
    b.g = p->Hq / p->Hkv;
    b.causal = p->causal ? 1 : 0;
    b.ring_i0 = 0; b.ring_t = 0; b.ring_p = 1; b.bsz = 1; b.n_outer = 1;
    b.scale = eff_scale(p);
    b.status = sp;
    return b;
}

// The one-pass backward: workspace rows with the dQ accumulator zeroed, dK/dV/dQ-partials, dQ rounded.
static cudaError_t one_pass_bwd(BwdParams b, const usp_problem* p, void* ws, const char* const names[3],
                                cudaStream_t s) {
    b.dq_acc = reinterpret_cast<float*>(static_cast<char*>(ws) + bwd_rows_bytes(p));
    cudaError_t e = traced(names[0], s, [&] { return launch_bwd_pre(b, s); });
    if (e == cudaSuccess) e = traced(names[1], s, [&] { return launch_bwd_dkdvq(b, s); });
    if (e == cudaSuccess) e = traced(names[2], s, [&] { return launch_bwd_dq_store(b, s); });
    return e;
}

usp_status usp_attn_bwd(const usp_problem* p, const void* q, const void* k, const void* v, const void* o,
                        const float* lse, const void* dout, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                        usp_stream stream) {
    usp_status st = attn_bwd_check(p, q, k, v, o, lse, dout, dq, dk, dv);
    if (st != USP_OK || empty(p)) return st;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return USP_ERR_MISALIGNED;
    if (ws_bytes < usp_attn_bwd_workspace_size(p)) return USP_ERR_WORKSPACE;
    int* sp = status_ptr();
    if (!sp) return USP_ERR_CUDA;
    const BwdParams b = head_sharded_bwd(p, q, k, v, o, lse, dout, dq, dk, dv, ws, sp);
    static const char* const names[3] = {"attn_bwd_pre", "attn_bwd_dkdvq", "attn_bwd_dq_store"};
    return cuda_status(one_pass_bwd(b, p, ws, names, static_cast<cudaStream_t>(stream)));
}

usp_status usp_attn_bwd_deterministic(const usp_problem* p, const void* q, const void* k, const void* v,
                                      const void* o, const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                      void* ws, size_t ws_bytes, usp_stream stream) {
    usp_status st = attn_bwd_check(p, q, k, v, o, lse, dout, dq, dk, dv);
    if (st != USP_OK || empty(p)) return st;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return USP_ERR_MISALIGNED;
    if (ws_bytes < usp_attn_bwd_deterministic_workspace_size(p)) return USP_ERR_WORKSPACE;
    int* sp = status_ptr();
    if (!sp) return USP_ERR_CUDA;
    const BwdParams b = head_sharded_bwd(p, q, k, v, o, lse, dout, dq, dk, dv, ws, sp);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = traced("attn_bwd_pre", s, [&] { return launch_bwd_pre(b, s); });
    if (e == cudaSuccess) e = traced("attn_bwd_dkdv", s, [&] { return launch_bwd_dkdv(b, s); });
    if (e == cudaSuccess) e = traced("attn_bwd_dq", s, [&] { return launch_bwd_dq(b, s); });
    return cuda_status(e);
}

usp_status usp_ring_merge(int64_t rows, int d, const float* o_a, const float* lse_a, const float* o_b,
                          const float* lse_b, float* o, float* lse, usp_stream stream) {
    if (rows < 0 || d < 1 || d % 4 != 0) return USP_ERR_INVALID_ARG;
    if (rows == 0) return USP_OK;
    const void* ptrs[] = {o_a, lse_a, o_b, lse_b, o, lse};
    for (const void* ptr : ptrs)
        if (!aligned16(ptr)) return USP_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return cuda_status(
        traced("ring_merge", s, [&] { return launch_lse_merge(rows, d, o_a, lse_a, o_b, lse_b, o, lse, s); }));
}

// The ring schedule over n_groups ring members, for a forward whose tensors and decode are set
// (ring_p = n_groups; outer index = member * per_member + the index within the member).  Step t
// attends member i's queries to member (i - t) mod n_groups's keys -- under the causal mask only
// members i >= t, the rest see none of those keys -- and merges each partial into the running
// float32 output (rows in member-major order, rows_per_member each) by log-sum-exp.  The final
// output is rounded to bf16 once.
static cudaError_t ring_fwd_schedule(FwdParams f, int n_groups, int per_member, size_t rows, size_t rows_per_member,
                                     float* acc_o, float* part_o, float* part_l, float* lse, void* o,
                                     const char* name, cudaStream_t s) {
    const int d = f.d;
    for (int t = 0; t < n_groups; ++t) {
        f.ring_t = t;
        f.ring_i0 = f.causal ? t : 0;
        f.n_outer = (f.causal ? n_groups - t : n_groups) * per_member;
        f.o_f32 = t == 0 ? acc_o : part_o;
        f.lse = t == 0 ? lse : part_l;
        cudaError_t e = traced(name, s, [&] { return launch_attn_fwd_bf16(f, s); });
        if (e != cudaSuccess) return e;
        if (t > 0) {
            const size_t r0 = (size_t)f.ring_i0 * rows_per_member;
            e = traced("ring_merge", s, [&] {
                return launch_lse_merge((int64_t)(rows - r0), d, acc_o + r0 * d, lse + r0, part_o + r0 * d,
                                        part_l + r0, acc_o + r0 * d, lse + r0, s);
            });
            if (e != cudaSuccess) return e;
        }
    }
    return traced("ring_to_bf16", s, [&] { return launch_f32_to_bf16(acc_o, o, (int64_t)(rows * d), s); });
}

// The ring backward over n_groups members (b's tensors, workspace rows and float32 accumulators
// set; the pre pass already run): at step t member i adds its partial gradients for the block
// pair (i, (i - t) mod n_groups) -- dK, dV travel with the KV block, dQ stays with the queries,
// masked only on the diagonal (t = 0).  Every block receives its first contribution at t = 0, so
// later steps add.  The accumulators are rounded to bf16 once.
// Every step runs the one-pass kernel: its dQ partials go into the float32 dQ accumulator b.dq_acc
// (zeroed by the pre pass, rounded to bf16 into dq at the end), its dK and dV into the float32 accumulators
// b.dk_f32 and b.dv_f32 (written at t = 0, added to after).
static cudaError_t ring_bwd_schedule(BwdParams b, int n_groups, int per_member, bool causal, size_t k_elems,
                                     void* dq, void* dk, void* dv, const char* name_step, cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    for (int t = 0; e == cudaSuccess && t < n_groups; ++t) {
        b.ring_t = t;
        b.ring_i0 = causal ? t : 0;
        b.n_outer = (causal ? n_groups - t : n_groups) * per_member;
        b.causal = (causal && t == 0) ? 1 : 0;
        b.accumulate = t > 0 ? 1 : 0;
        e = traced(name_step, s, [&] { return launch_bwd_dkdvq(b, s); });
    }
    b.dq = dq;
    if (e == cudaSuccess) e = traced("ring_bwd_dq_store", s, [&] { return launch_bwd_dq_store(b, s); });
    if (e == cudaSuccess) e = traced("ring_to_bf16", s, [&] { return launch_f32_to_bf16(b.dk_f32, dk, (int64_t)k_elems, s); });
    if (e == cudaSuccess) e = traced("ring_to_bf16", s, [&] { return launch_f32_to_bf16(b.dv_f32, dv, (int64_t)k_elems, s); });
    return e;
}

// Ring workspace: float32 running output [rows][d], float32 partial output
// [rows][d] and partial LSE [rows], rows = P*B*(N/P)*Hq in sequence-sharded
// order.  The caller's lse buffer holds the running LSE.
static size_t ring_part(size_t bytes) { return (bytes + 255) & ~(size_t)255; }

size_t usp_ring_workspace_size(const usp_problem* p) {
    if (check_problem(p, false) != USP_OK) return 0;
    const size_t rows = (size_t)p->B * p->N * p->Hq;
    return 2 * ring_part(rows * p->d * sizeof(float)) + ring_part(rows * sizeof(float));
}

usp_status usp_ring_attn_fwd(const usp_problem* p, const void* q, const void* k, const void* v, void* o, float* lse,
                             void* ws, size_t ws_bytes, usp_stream stream) {
    usp_status st = check_problem(p, false);
    if (st != USP_OK) return st;
    if (p->d != 64 && p->d != 128) return USP_ERR_UNSUPPORTED;
    if (p->dtype != USP_BF16) return USP_ERR_UNSUPPORTED;
    if ((int64_t)p->B * p->P > 65535) return USP_ERR_UNSUPPORTED;
    if (empty(p)) return USP_OK;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return USP_ERR_MISALIGNED;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return USP_ERR_MISALIGNED;
    if (ws_bytes < usp_ring_workspace_size(p)) return USP_ERR_WORKSPACE;
    int* sp = status_ptr();
    if (!sp) return USP_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    const int P = p->P, B = p->B, Hq = p->Hq, Hkv = p->Hkv, d = p->d;
    const int Np = p->N / P;
    const size_t rows = (size_t)B * p->N * Hq;
    float* acc_o = static_cast<float*>(ws);
    float* part_o = reinterpret_cast<float*>(static_cast<char*>(ws) + ring_part(rows * d * sizeof(float)));
    float* part_l = reinterpret_cast<float*>(static_cast<char*>(ws) + 2 * ring_part(rows * d * sizeof(float)));
    const size_t rows_per_rank = (size_t)B * Np * Hq;

    FwdParams f{};
    f.q = Tensor4{const_cast<void*>(q), d, (int64_t)Hq * d, (int64_t)Np * Hq * d, Hq, Np, P * B};
    f.k = Tensor4{const_cast<void*>(k), d, (int64_t)Hkv * d, (int64_t)Np * Hkv * d, Hkv, Np, P * B};
    f.v = Tensor4{const_cast<void*>(v), d, (int64_t)Hkv * d, (int64_t)Np * Hkv * d, Hkv, Np, P * B};
    f.d = d;
    f.g = Hq / Hkv;
    f.n_heads = Hq;
    f.q_len = Np;
    f.kv_len = Np;
    f.ring_p = P;
    f.bsz = B;
    f.np = Np;
    f.causal = p->causal ? 1 : 0;
    f.scale = eff_scale(p);
    f.o_bf16 = nullptr;
    f.o_s_head = d;
    f.o_s_tok = (int64_t)Hq * d;
    f.o_s_outer = (int64_t)Np * Hq * d;
    f.l_s_head = 1;
    f.l_s_tok = Hq;
    f.l_s_outer = (int64_t)Np * Hq;
    f.status = sp;

    // rank i attends block i - t only when that block is not in its future
    return cuda_status(
        ring_fwd_schedule(f, P, B, rows, rows_per_rank, acc_o, part_o, part_l, lse, o, "ring_attn_partial", s));
}

// Ring backward workspace: the backward rows (40 bytes per padded query row
// of every rank and head: D, lse*log2(e), -lse/scale and -D as bf16 splits),
// the float32 dQ accumulator (d values per padded row, in 128-row tiles), then
// float32 accumulators for dK and dV in sequence-sharded order.
static size_t ring_bwd_rows(const usp_problem* p) {
    const size_t npad = ((size_t)(p->N / p->P) + 127) / 128 * 128;
    return (size_t)p->P * p->B * p->Hq * npad;
}

size_t usp_ring_bwd_workspace_size(const usp_problem* p) {
    if (check_problem(p, false) != USP_OK) return 0;
    const size_t k_elems = (size_t)p->B * p->N * p->Hkv * p->d;
    return ring_part(ring_bwd_rows(p) * 40) + ring_part(ring_bwd_rows(p) * p->d * 4) + 2 * ring_part(k_elems * 4);
}

usp_status usp_ring_attn_bwd(const usp_problem* p, const void* q, const void* k, const void* v, const void* o,
                             const float* lse, const void* dout, void* dq, void* dk, void* dv, void* ws,
                             size_t ws_bytes, usp_stream stream) {
    usp_status st = check_problem(p, false);
    if (st != USP_OK) return st;
    if (p->d != 64 && p->d != 128) return USP_ERR_UNSUPPORTED;
    if (p->dtype != USP_BF16) return USP_ERR_UNSUPPORTED;
    if ((int64_t)p->B * p->P > 65535) return USP_ERR_UNSUPPORTED;
    if (empty(p)) return USP_OK;
    const void* ptrs[] = {q, k, v, o, lse, dout, dq, dk, dv};
    for (const void* ptr : ptrs)
        if (!aligned16(ptr)) return USP_ERR_MISALIGNED;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return USP_ERR_MISALIGNED;
    if (ws_bytes < usp_ring_bwd_workspace_size(p)) return USP_ERR_WORKSPACE;
    int* sp = status_ptr();
    if (!sp) return USP_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    const int P = p->P, B = p->B, Hq = p->Hq, Hkv = p->Hkv, d = p->d;
    const int Np = p->N / P;
    const size_t k_elems = (size_t)B * p->N * Hkv * d;
    char* w = static_cast<char*>(ws);
    float* acc_dq = reinterpret_cast<float*>(w + ring_part(ring_bwd_rows(p) * 40));
    float* acc_dk = reinterpret_cast<float*>(reinterpret_cast<char*>(acc_dq) + ring_part(ring_bwd_rows(p) * d * 4));
    float* acc_dv = reinterpret_cast<float*>(reinterpret_cast<char*>(acc_dk) + ring_part(k_elems * 4));

    BwdParams b{};
    const int64_t qs_tok = (int64_t)Hq * d, ks_tok = (int64_t)Hkv * d;
    b.q = Tensor4{const_cast<void*>(q), d, qs_tok, (int64_t)Np * qs_tok, Hq, Np, P * B};
    b.o = Tensor4{const_cast<void*>(o), d, qs_tok, (int64_t)Np * qs_tok, Hq, Np, P * B};
    b.dout = Tensor4{const_cast<void*>(dout), d, qs_tok, (int64_t)Np * qs_tok, Hq, Np, P * B};
    b.k = Tensor4{const_cast<void*>(k), d, ks_tok, (int64_t)Np * ks_tok, Hkv, Np, P * B};
    b.v = Tensor4{const_cast<void*>(v), d, ks_tok, (int64_t)Np * ks_tok, Hkv, Np, P * B};
    b.lse = lse;  // [P][B][N/P][Hq], the merged LSE of usp_ring_attn_fwd
    b.l_s_head = 1;
    b.l_s_tok = Hq;
    b.l_s_outer = (int64_t)Np * Hq;
    b.ws = reinterpret_cast<float*>(w);
    b.n_z = P * B * Hq;
    b.dq_acc = acc_dq;
    b.dk_f32 = acc_dk;
    b.dv_f32 = acc_dv;
    b.d = d;
    b.g = Hq / Hkv;
    b.ring_p = P;
    b.bsz = B;
    b.scale = eff_scale(p);
    b.status = sp;

    // D and the lse rows of every rank (they use the final O and the merged LSE)
    cudaError_t e = traced("ring_bwd_pre", s, [&] { return launch_bwd_pre(b, s); });
    if (e == cudaSuccess) e = ring_bwd_schedule(b, P, B, p->causal != 0, k_elems, dq, dk, dv, "ring_bwd_dkdvq", s);
    return cuda_status(e);
}

// ---- all-gather-KV context parallelism
// Workspace: the gathered K and V (bf16, [B][N][Hkv][d]); the backward adds
// its 40-byte rows per padded query row of every rank and head and float32
// dK, dV accumulators in the gathered layout.
static size_t gathered_bytes(const usp_problem* p) { return (size_t)p->B * p->N * p->Hkv * p->d * 2; }

size_t usp_allgather_workspace_size(const usp_problem* p) {
    if (check_problem(p, false) != USP_OK) return 0;
    return 2 * ring_part(gathered_bytes(p));
}

size_t usp_allgather_bwd_workspace_size(const usp_problem* p) {
    if (check_problem(p, false) != USP_OK) return 0;
    return 2 * ring_part(gathered_bytes(p)) + ring_part(ring_bwd_rows(p) * 40) + ring_part(ring_bwd_rows(p) * p->d * 4) +
           2 * ring_part(gathered_bytes(p) * 2);
}

static usp_status allgather_checks(const usp_problem* p, std::initializer_list<const void*> ptrs, const void* ws) {
    usp_status st = check_problem(p, false);
    if (st != USP_OK) return st;
    if (p->d != 64 && p->d != 128) return USP_ERR_UNSUPPORTED;
    if (p->dtype != USP_BF16) return USP_ERR_UNSUPPORTED;
    if ((int64_t)p->B * p->P > 65535) return USP_ERR_UNSUPPORTED;
    if (empty(p)) return USP_OK;
    for (const void* ptr : ptrs)
        if (!aligned16(ptr)) return USP_ERR_MISALIGNED;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return USP_ERR_MISALIGNED;
    return USP_OK;
}

// Every rank's K and V shard into one sequence per batch: one copy per (rank, batch) chunk.
static cudaError_t gather_kv(const usp_problem* p, const void* k, const void* v, void* kg, void* vg, cudaStream_t s) {
    const int P = p->P, B = p->B, Np = p->N / P;
    const size_t row = (size_t)p->Hkv * p->d * 2, chunk = (size_t)Np * row;
    return traced("allgather_kv", s, [&] {
        for (int i = 0; i < P; ++i)
            for (int b = 0; b < B; ++b) {
                const size_t src = ((size_t)i * B + b) * chunk, dst = ((size_t)b * p->N + (size_t)i * Np) * row;
                cudaError_t e = cudaMemcpyAsync(static_cast<char*>(kg) + dst, static_cast<const char*>(k) + src, chunk,
                                                cudaMemcpyDeviceToDevice, s);
                if (e == cudaSuccess)
                    e = cudaMemcpyAsync(static_cast<char*>(vg) + dst, static_cast<const char*>(v) + src, chunk,
                                        cudaMemcpyDeviceToDevice, s);
                if (e != cudaSuccess) return e;
            }
        return cudaSuccess;
    });
}

usp_status usp_allgather_attn_fwd(const usp_problem* p, const void* q, const void* k, const void* v, void* o,
                                  float* lse, void* ws, size_t ws_bytes, usp_stream stream) {
    usp_status st = allgather_checks(p, {q, k, v, o, lse}, ws);
    if (st != USP_OK || empty(p)) return st;
    if (ws_bytes < usp_allgather_workspace_size(p)) return USP_ERR_WORKSPACE;
    int* sp = status_ptr();
    if (!sp) return USP_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int P = p->P, B = p->B, Hq = p->Hq, Hkv = p->Hkv, d = p->d, N = p->N, Np = N / P;
    void* kg = ws;
    void* vg = static_cast<char*>(ws) + ring_part(gathered_bytes(p));
    if (gather_kv(p, k, v, kg, vg, s) != cudaSuccess) return USP_ERR_CUDA;

    FwdParams f{};
    f.q = Tensor4{const_cast<void*>(q), d, (int64_t)Hq * d, (int64_t)Np * Hq * d, Hq, Np, P * B};
    f.k = Tensor4{kg, d, (int64_t)Hkv * d, (int64_t)N * Hkv * d, Hkv, N, B};
    f.v = Tensor4{vg, d, (int64_t)Hkv * d, (int64_t)N * Hkv * d, Hkv, N, B};
    f.d = d;
    f.g = Hq / Hkv;
    f.n_heads = Hq;
    f.n_outer = P * B;
    f.q_len = Np;
    f.kv_len = N;
    f.ring_i0 = 0;
    f.ring_t = 0;
    f.ring_p = P;
    f.bsz = B;
    f.np = Np;
    f.kv_gathered = 1;
    f.causal = p->causal ? 1 : 0;
    f.scale = eff_scale(p);
    f.o_bf16 = o;
    f.o_s_head = d;
    f.o_s_tok = (int64_t)Hq * d;
    f.o_s_outer = (int64_t)Np * Hq * d;
    f.lse = lse;
    f.l_s_head = 1;
    f.l_s_tok = Hq;
    f.l_s_outer = (int64_t)Np * Hq;
    f.status = sp;
    return cuda_status(traced("allgather_attn_fwd", s, [&] { return launch_attn_fwd_bf16(f, s); }));
}

usp_status usp_allgather_attn_bwd(const usp_problem* p, const void* q, const void* k, const void* v, const void* o,
                                  const float* lse, const void* dout, void* dq, void* dk, void* dv, void* ws,
                                  size_t ws_bytes, usp_stream stream) {
    usp_status st = allgather_checks(p, {q, k, v, o, lse, dout, dq, dk, dv}, ws);
    if (st != USP_OK || empty(p)) return st;
    if (ws_bytes < usp_allgather_bwd_workspace_size(p)) return USP_ERR_WORKSPACE;
    int* sp = status_ptr();
    if (!sp) return USP_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int P = p->P, B = p->B, Hq = p->Hq, Hkv = p->Hkv, d = p->d, N = p->N, Np = N / P;
    char* w = static_cast<char*>(ws);
    void* kg = w;
    void* vg = w + ring_part(gathered_bytes(p));
    float* rows = reinterpret_cast<float*>(w + 2 * ring_part(gathered_bytes(p)));
    float* acc_dq = reinterpret_cast<float*>(reinterpret_cast<char*>(rows) + ring_part(ring_bwd_rows(p) * 40));
    float* acc_dk = reinterpret_cast<float*>(reinterpret_cast<char*>(acc_dq) + ring_part(ring_bwd_rows(p) * d * 4));
    float* acc_dv = reinterpret_cast<float*>(reinterpret_cast<char*>(acc_dk) + ring_part(gathered_bytes(p) * 2));
    if (gather_kv(p, k, v, kg, vg, s) != cudaSuccess) return USP_ERR_CUDA;

    BwdParams b{};
    const int64_t qs_tok = (int64_t)Hq * d, ks_tok = (int64_t)Hkv * d;
    b.q = Tensor4{const_cast<void*>(q), d, qs_tok, (int64_t)Np * qs_tok, Hq, Np, P * B};
    b.o = Tensor4{const_cast<void*>(o), d, qs_tok, (int64_t)Np * qs_tok, Hq, Np, P * B};
    b.dout = Tensor4{const_cast<void*>(dout), d, qs_tok, (int64_t)Np * qs_tok, Hq, Np, P * B};
    b.k = Tensor4{kg, d, ks_tok, (int64_t)N * ks_tok, Hkv, N, B};
    b.v = Tensor4{vg, d, ks_tok, (int64_t)N * ks_tok, Hkv, N, B};
    b.lse = lse;
    b.l_s_head = 1;
    b.l_s_tok = Hq;
    b.l_s_outer = (int64_t)Np * Hq;
    b.ws = rows;
    b.n_z = P * B * Hq;
    b.dq = dq;
    b.dq_acc = acc_dq;
    b.dk_f32 = acc_dk;
    b.dv_f32 = acc_dv;
    b.d = d;
    b.g = Hq / Hkv;
    b.causal = p->causal ? 1 : 0;
    b.ring_t = 0;
    b.ring_p = P;
    b.bsz = B;
    b.kv_gathered = 1;
    b.scale = eff_scale(p);
    b.status = sp;

    cudaError_t e = traced("allgather_bwd_pre", s, [&] { return launch_bwd_pre(b, s); });
    // dK, dV: rank i's partial over the gathered keys, summed over the ranks in float32 (the
    // reduce part of a reduce-scatter), one launch per rank in rank order; each launch also adds
    // rank i's dQ partials (dQ_i is complete after rank i's launch)
    for (int i = 0; e == cudaSuccess && i < P; ++i) {
        b.ring_i0 = i;
        b.n_outer = B;
        b.accumulate = i > 0 ? 1 : 0;
        e = traced("allgather_bwd_dkdvq", s, [&] { return launch_bwd_dkdvq(b, s); });
    }
    b.ring_i0 = 0;
    b.n_outer = P * B;
    if (e == cudaSuccess) e = traced("allgather_bwd_dq_store", s, [&] { return launch_bwd_dq_store(b, s); });
    // the scatter part: rank j keeps the rows of its own shard, rounded to bf16
    const int64_t chunk = (int64_t)Np * Hkv * d;
    for (int j = 0; e == cudaSuccess && j < P; ++j)
        for (int bb = 0; e == cudaSuccess && bb < B; ++bb) {
            const int64_t src = ((int64_t)bb * N + (int64_t)j * Np) * Hkv * d, dst = ((int64_t)j * B + bb) * chunk;
            e = traced("allgather_scatter", s, [&] {
                cudaError_t e2 = launch_f32_to_bf16(acc_dk + src, static_cast<uint16_t*>(dk) + dst, chunk, s);
                return e2 == cudaSuccess ? launch_f32_to_bf16(acc_dv + src, static_cast<uint16_t*>(dv) + dst, chunk, s)
                                         : e2;
            });
        }
    return cuda_status(e);
}

// ---- zigzag (load-balanced) ring attention
// The sequence is cut into 2P chunks of c = N/(2P) tokens; rank r holds chunks
// r and 2P-1-r as the two halves of its shard ([P][B][2][c][H][d]).
static size_t zz_rows(const usp_problem* p) {
    const size_t c = (size_t)p->N / (2 * (size_t)p->P);
    return 2 * (size_t)p->P * p->B * p->Hq * ((c + 127) / 128 * 128);
}

static usp_status zz_check(const usp_problem* p) {
    usp_status st = check_problem(p, false);
    if (st != USP_OK) return st;
    if (p->N % (2 * p->P) != 0) return USP_ERR_INVALID_ARG;
    return USP_OK;
}

static usp_status zz_copy(const usp_problem* p, int Hx, const void* src, void* dst, bool to_zigzag,
                          cudaStream_t s) {
    usp_status st = zz_check(p);
    if (st != USP_OK) return st;
    if (Hx < 1) return USP_ERR_INVALID_ARG;
    if (empty(p)) return USP_OK;
    if (!src || !dst) return USP_ERR_INVALID_ARG;
    const int P = p->P, B = p->B;
    const size_t c = (size_t)p->N / (2 * P);
    const size_t esz = p->dtype == USP_BF16 ? 2 : 4, chunk = c * Hx * p->d * esz;
    const char* a = static_cast<const char*>(src);
    char* z = static_cast<char*>(dst);
    if (a < z + 2 * (size_t)P * B * chunk && z < a + 2 * (size_t)P * B * chunk) return USP_ERR_INVALID_ARG;
    return cuda_status(traced("zigzag_copy", s, [&] {
        for (int g = 0; g < 2 * P; ++g)
            for (int b = 0; b < B; ++b) {
                // chunk g: contiguous shard g/2, half g%2; zigzag rank (g < P ? g : 2P-1-g), half (g >= P)
                const size_t off_c = (((size_t)(g / 2) * B + b) * 2 + g % 2) * chunk;
                const size_t zr = g < P ? g : 2 * P - 1 - g;
                const size_t off_z = ((zr * B + b) * 2 + (g >= P ? 1 : 0)) * chunk;
                cudaError_t e = to_zigzag ? cudaMemcpyAsync(z + off_z, a + off_c, chunk, cudaMemcpyDeviceToDevice, s)
                                          : cudaMemcpyAsync(z + off_c, a + off_z, chunk, cudaMemcpyDeviceToDevice, s);
                if (e != cudaSuccess) return e;
            }
        return cudaSuccess;
    }));
}

usp_status usp_zigzag_shard(const usp_problem* p, int Hx, const void* src, void* dst, usp_stream stream) {
    return zz_copy(p, Hx, src, dst, true, static_cast<cudaStream_t>(stream));
}

usp_status usp_zigzag_unshard(const usp_problem* p, int Hx, const void* src, void* dst, usp_stream stream) {
    return zz_copy(p, Hx, src, dst, false, static_cast<cudaStream_t>(stream));
}

size_t usp_zigzag_workspace_size(const usp_problem* p) {
    if (zz_check(p) != USP_OK) return 0;
    return usp_ring_workspace_size(p);
}

size_t usp_zigzag_bwd_workspace_size(const usp_problem* p) {
    if (zz_check(p) != USP_OK) return 0;
    const size_t k_elems = (size_t)p->B * p->N * p->Hkv * p->d;
    return ring_part(zz_rows(p) * 40) + ring_part(zz_rows(p) * p->d * 4) + 2 * ring_part(k_elems * 4);
}

static usp_status zz_common_checks(const usp_problem* p, std::initializer_list<const void*> ptrs, const void* ws) {
    usp_status st = zz_check(p);
    if (st != USP_OK) return st;
    if (p->d != 64 && p->d != 128) return USP_ERR_UNSUPPORTED;
    if (p->dtype != USP_BF16) return USP_ERR_UNSUPPORTED;
    if ((int64_t)p->B * p->P * 2 > 65535) return USP_ERR_UNSUPPORTED;
    if (empty(p)) return USP_OK;
    for (const void* ptr : ptrs)
        if (!aligned16(ptr)) return USP_ERR_MISALIGNED;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return USP_ERR_MISALIGNED;
    return USP_OK;
}

usp_status usp_zigzag_attn_fwd(const usp_problem* p, const void* q, const void* k, const void* v, void* o, float* lse,
                               void* ws, size_t ws_bytes, usp_stream stream) {
    usp_status st = zz_common_checks(p, {q, k, v, o, lse}, ws);
    if (st != USP_OK || empty(p)) return st;
    if (ws_bytes < usp_zigzag_workspace_size(p)) return USP_ERR_WORKSPACE;
    int* sp = status_ptr();
    if (!sp) return USP_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int P = p->P, B = p->B, Hq = p->Hq, Hkv = p->Hkv, d = p->d;
    const int c = p->N / (2 * P);
    const size_t rows = (size_t)B * p->N * Hq;
    float* acc_o = static_cast<float*>(ws);
    float* part_o = reinterpret_cast<float*>(static_cast<char*>(ws) + ring_part(rows * d * sizeof(float)));
    float* part_l = reinterpret_cast<float*>(static_cast<char*>(ws) + 2 * ring_part(rows * d * sizeof(float)));

    FwdParams f{};
    f.q = Tensor4{const_cast<void*>(q), d, (int64_t)Hq * d, (int64_t)c * Hq * d, Hq, c, 2 * P * B};
    f.k = Tensor4{const_cast<void*>(k), d, (int64_t)Hkv * d, (int64_t)c * Hkv * d, Hkv, c, 2 * P * B};
    f.v = Tensor4{const_cast<void*>(v), d, (int64_t)Hkv * d, (int64_t)c * Hkv * d, Hkv, c, 2 * P * B};
    f.d = d;
    f.g = Hq / Hkv;
    f.n_heads = Hq;
    f.n_outer = 2 * P * B;
    f.q_len = c;
    f.kv_len = c;
    f.ring_i0 = 0;
    f.ring_p = P;
    f.bsz = B;
    f.np = c;
    f.zigzag = 1;
    f.causal = p->causal ? 1 : 0;
    f.scale = eff_scale(p);
    f.o_s_head = d;
    f.o_s_tok = (int64_t)Hq * d;
    f.o_s_outer = (int64_t)c * Hq * d;
    f.l_s_head = 1;
    f.l_s_tok = Hq;
    f.l_s_outer = (int64_t)c * Hq;
    f.status = sp;
    // step t, KV half kh: every rank attends both of its query chunks to chunk kh of the KV block it
    // holds; pairs wholly in the future come out empty (LSE -inf) and merge as the identity
    for (int t = 0; t < P; ++t)
        for (int kh = 0; kh < 2; ++kh) {
            const bool first = t == 0 && kh == 0;
            f.ring_t = t;
            f.zz_kh = kh;
            f.o_f32 = first ? acc_o : part_o;
            f.lse = first ? lse : part_l;
            cudaError_t e = traced("zigzag_attn_partial", s, [&] { return launch_attn_fwd_bf16(f, s); });
            if (e == cudaSuccess && !first)
                e = traced("ring_merge", s, [&] {
                    return launch_lse_merge((int64_t)rows, d, acc_o, lse, part_o, part_l, acc_o, lse, s);
                });
            if (e != cudaSuccess) return USP_ERR_CUDA;
        }
    return cuda_status(traced("ring_to_bf16", s, [&] { return launch_f32_to_bf16(acc_o, o, (int64_t)(rows * d), s); }));
}

usp_status usp_zigzag_attn_bwd(const usp_problem* p, const void* q, const void* k, const void* v, const void* o,
                               const float* lse, const void* dout, void* dq, void* dk, void* dv, void* ws,
                               size_t ws_bytes, usp_stream stream) {
    usp_status st = zz_common_checks(p, {q, k, v, o, lse, dout, dq, dk, dv}, ws);
    if (st != USP_OK || empty(p)) return st;
    if (ws_bytes < usp_zigzag_bwd_workspace_size(p)) return USP_ERR_WORKSPACE;
    int* sp = status_ptr();
    if (!sp) return USP_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int P = p->P, B = p->B, Hq = p->Hq, Hkv = p->Hkv, d = p->d;
    const int c = p->N / (2 * P);
    const size_t k_elems = (size_t)B * p->N * Hkv * d;
    char* w = static_cast<char*>(ws);
    float* acc_dq = reinterpret_cast<float*>(w + ring_part(zz_rows(p) * 40));
    float* acc_dk = reinterpret_cast<float*>(reinterpret_cast<char*>(acc_dq) + ring_part(zz_rows(p) * d * 4));
    float* acc_dv = reinterpret_cast<float*>(reinterpret_cast<char*>(acc_dk) + ring_part(k_elems * 4));

    BwdParams b{};
    const int64_t qs_tok = (int64_t)Hq * d, ks_tok = (int64_t)Hkv * d;
    b.q = Tensor4{const_cast<void*>(q), d, qs_tok, (int64_t)c * qs_tok, Hq, c, 2 * P * B};
    b.o = Tensor4{const_cast<void*>(o), d, qs_tok, (int64_t)c * qs_tok, Hq, c, 2 * P * B};
    b.dout = Tensor4{const_cast<void*>(dout), d, qs_tok, (int64_t)c * qs_tok, Hq, c, 2 * P * B};
    b.k = Tensor4{const_cast<void*>(k), d, ks_tok, (int64_t)c * ks_tok, Hkv, c, 2 * P * B};
    b.v = Tensor4{const_cast<void*>(v), d, ks_tok, (int64_t)c * ks_tok, Hkv, c, 2 * P * B};
    b.lse = lse;
    b.l_s_head = 1;
    b.l_s_tok = Hq;
    b.l_s_outer = (int64_t)c * Hq;
    b.ws = reinterpret_cast<float*>(w);
    b.n_z = 2 * P * B * Hq;
    b.dq_acc = acc_dq;
    b.dk_f32 = acc_dk;
    b.dv_f32 = acc_dv;
    b.d = d;
    b.g = Hq / Hkv;
    b.causal = p->causal ? 1 : 0;
    b.ring_i0 = 0;
    b.ring_p = P;
    b.bsz = B;
    b.zigzag = 1;
    b.scale = eff_scale(p);
    b.status = sp;

    cudaError_t e = traced("zigzag_bwd_pre", s, [&] { return launch_bwd_pre(b, s); });
    for (int t = 0; e == cudaSuccess && t < P; ++t)
        for (int kh = 0; e == cudaSuccess && kh < 2; ++kh) {
            b.ring_t = t;
            b.zz_kh = kh;
            // KV chunk kh against one query half at a time (each CTA owns its key rows): dK, dV of the
            // chunk (first written at t = 0 by query half 0) and the half's dQ partials
            for (int qh = 0; e == cudaSuccess && qh < 2; ++qh) {
                b.zz_qh = qh;
                b.n_outer = P * B;
                b.accumulate = (t == 0 && qh == 0) ? 0 : 1;
                e = traced("zigzag_bwd_dkdvq", s, [&] { return launch_bwd_dkdvq(b, s); });
            }
        }
    b.dq = dq;
    if (e == cudaSuccess) e = traced("zigzag_bwd_dq_store", s, [&] { return launch_bwd_dq_store(b, s); });
    if (e == cudaSuccess) e = traced("ring_to_bf16", s, [&] { return launch_f32_to_bf16(acc_dk, dk, (int64_t)k_elems, s); });
    if (e == cudaSuccess) e = traced("ring_to_bf16", s, [&] { return launch_f32_to_bf16(acc_dv, dv, (int64_t)k_elems, s); });
    return cuda_status(e);
}

// ---- Ulysses attention with the all-to-all fused into the attention kernels
// Q, K, V, O, dO, dQ, dK, dV stay in the sequence-sharded layout [P][B][N/P][H][d]
// and the LSE in [P][B][N/P][Hq]: the kernels read and write every rank's shard in
// place (split_pos), so no remap runs.  Per query head the work is the head-
// sharded path's, tile for tile: the results are the remapped path's, bit for bit.
static usp_status fused_checks(const usp_problem* p, std::initializer_list<const void*> ptrs) {
    usp_status st = check_problem(p);
    if (st != USP_OK) return st;
    if (p->d != 64 && p->d != 128) return USP_ERR_UNSUPPORTED;
    if (p->dtype != USP_BF16) return USP_ERR_UNSUPPORTED;
    if ((p->N / p->P) % 128 != 0) return USP_ERR_UNSUPPORTED;  // shards of whole 128-row tiles
    if ((int64_t)p->B * p->P > 65535) return USP_ERR_UNSUPPORTED;
    if (empty(p)) return USP_OK;
    for (const void* ptr : ptrs)
        if (!aligned16(ptr)) return USP_ERR_MISALIGNED;
    return USP_OK;
}

// sequence-sharded view of one operand family with H heads
static Tensor4 seq_view(const void* ptr, const usp_problem* p, int H) {
    const int64_t Np = p->N / p->P, tok = (int64_t)H * p->d;
    return Tensor4{const_cast<void*>(ptr), p->d, tok, Np * tok, H, (int)Np, p->P * p->B};
}

usp_status usp_fused_attn_fwd(const usp_problem* p, const void* q, const void* k, const void* v, void* o, float* lse,
                              usp_stream stream) {
    usp_status st = fused_checks(p, {q, k, v, o, lse});
    if (st != USP_OK || empty(p)) return st;
    int* sp = status_ptr();
    if (!sp) return USP_ERR_CUDA;
    const int B = p->B, Hq = p->Hq, d = p->d, Np = p->N / p->P;
    FwdParams f{};
    f.q = seq_view(q, p, Hq);
    f.k = seq_view(k, p, p->Hkv);
    f.v = seq_view(v, p, p->Hkv);
    f.d = d;
    f.g = Hq / p->Hkv;
    f.n_heads = Hq;
    f.n_outer = B;  // one outer index per batch, global positions 0 .. N-1
    f.q_len = p->N;
    f.kv_len = p->N;
    f.ring_p = 1;
    f.bsz = B;
    f.split_np = Np;
    f.split_b = B;
    f.causal = p->causal ? 1 : 0;
    f.scale = eff_scale(p);
    f.o_bf16 = o;
    f.o_s_head = d;
    f.o_s_tok = (int64_t)Hq * d;
    f.o_s_outer = (int64_t)Np * Hq * d;
    f.lse = lse;
    f.l_s_head = 1;
    f.l_s_tok = Hq;
    f.l_s_outer = (int64_t)Np * Hq;
    f.status = sp;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return cuda_status(traced("fused_attn_fwd", s, [&] { return launch_attn_fwd_bf16(f, s); }));
}

size_t usp_fused_attn_bwd_workspace_size(const usp_problem* p) {
    if (check_problem(p) != USP_OK) return 0;
    return usp_attn_bwd_workspace_size(p);  // the same rows: (batch, head, position)
}

usp_status usp_fused_attn_bwd(const usp_problem* p, const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dout, void* dq, void* dk, void* dv, void* ws,
                              size_t ws_bytes, usp_stream stream) {
    usp_status st = fused_checks(p, {q, k, v, o, lse, dout, dq, dk, dv});
    if (st != USP_OK || empty(p)) return st;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return USP_ERR_MISALIGNED;
    if (ws_bytes < usp_fused_attn_bwd_workspace_size(p)) return USP_ERR_WORKSPACE;
    int* sp = status_ptr();
    if (!sp) return USP_ERR_CUDA;
    const int B = p->B, Hq = p->Hq, Np = p->N / p->P;
    BwdParams b{};
    b.q = seq_view(q, p, Hq);
    b.o = seq_view(o, p, Hq);
    b.dout = seq_view(dout, p, Hq);
    b.k = seq_view(k, p, p->Hkv);
    b.v = seq_view(v, p, p->Hkv);
    b.lse = lse;
    b.l_s_head = 1;
    b.l_s_tok = Hq;
    b.l_s_outer = (int64_t)Np * Hq;
    b.ws = static_cast<float*>(ws);
    b.n_z = B * Hq;
    b.dq = dq;
    b.dk = dk;
    b.dv = dv;
    b.d = p->d;
    b.g = Hq / p->Hkv;
    b.causal = p->causal ? 1 : 0;
    b.ring_p = 1;
    b.bsz = B;
    b.n_outer = B;
    b.split_np = Np;
    b.split_b = B;
    b.scale = eff_scale(p);
    b.status = sp;
    static const char* const names[3] = {"fused_bwd_pre", "fused_bwd_dkdvq", "fused_bwd_dq_store"};
    return cuda_status(one_pass_bwd(b, p, ws, names, static_cast<cudaStream_t>(stream)));
}

// ---- 2-D (hybrid) sequence parallelism: Ulysses inside groups, ring across them
// P = Pu * Pr ranks.  Ring group g (0 .. Pr-1) is the Pu consecutive ranks g*Pu ..
// g*Pu + Pu - 1, holding the contiguous token chunk g of Nc = N/Pr tokens.  The
// all-to-all inside a group leaves rank g*Pu + u with heads u*H/Pu .. (u+1)*H/Pu - 1
// of chunk g: the hybrid layout [P][B][H/Pu][Nc][d] (LSE [P][B][Hq/Pu][Nc]).  The
// ring then runs over the Pr groups, each query head meeting its KV head's chunks.
static usp_status hybrid_check(const usp_problem* p, int Pu) {
    usp_status st = check_problem(p, false);
    if (st != USP_OK) return st;
    if (Pu < 1 || p->P % Pu != 0 || p->Hq % Pu != 0 || p->Hkv % Pu != 0) return USP_ERR_INVALID_ARG;
    return USP_OK;
}

static usp_status hybrid_a2a(int dir, const usp_problem* p, int Pu, int Hx, const void* src, void* dst,
                             usp_stream stream) {
    usp_status st = hybrid_check(p, Pu);
    if (st != USP_OK) return st;
    if (Hx != p->Hq && Hx != p->Hkv) return USP_ERR_INVALID_ARG;
    const int row_bytes = p->d * elem_size(p->dtype);
    if (row_bytes != 64 && row_bytes != 128 && row_bytes != 256 && row_bytes != 512) return USP_ERR_UNSUPPORTED;
    if (empty(p)) return USP_OK;
    if (!aligned16(src) || !aligned16(dst)) return USP_ERR_MISALIGNED;
    const size_t bytes = (size_t)p->B * Hx * (size_t)p->N * row_bytes;
    const char* sb = static_cast<const char*>(src);
    char* tb = static_cast<char*>(dst);
    if (sb < tb + bytes && tb < sb + bytes) return USP_ERR_INVALID_ARG;  // overlap
    // each group's Pu shards are one contiguous block on both sides: a Ulysses remap of Nc tokens
    const int Pr = p->P / Pu, Nc = p->N / Pr;
    const size_t blk = bytes / Pr;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (int g = 0; g < Pr; ++g) {
        cudaError_t e = traced(dir == 0 ? "hybrid_seq2head" : "hybrid_head2seq", s, [&] {
            return launch_remap(dir, sb + g * blk, tb + g * blk, p->B, Hx, Nc, Pu, row_bytes, s);
        });
        if (e != cudaSuccess) return USP_ERR_CUDA;
    }
    return USP_OK;
}

usp_status usp_hybrid_seq2head(const usp_problem* p, int Pu, int Hx, const void* src, void* dst, usp_stream stream) {
    return hybrid_a2a(0, p, Pu, Hx, src, dst, stream);
}

usp_status usp_hybrid_head2seq(const usp_problem* p, int Pu, int Hx, const void* src, void* dst, usp_stream stream) {
    return hybrid_a2a(1, p, Pu, Hx, src, dst, stream);
}

static usp_status hybrid_attn_checks(const usp_problem* p, int Pu, std::initializer_list<const void*> ptrs,
                                     const void* ws) {
    usp_status st = hybrid_check(p, Pu);
    if (st != USP_OK) return st;
    if (p->d != 64 && p->d != 128) return USP_ERR_UNSUPPORTED;
    if (p->dtype != USP_BF16) return USP_ERR_UNSUPPORTED;
    if ((int64_t)p->B * p->P > 65535) return USP_ERR_UNSUPPORTED;
    if (empty(p)) return USP_OK;
    for (const void* ptr : ptrs)
        if (!aligned16(ptr)) return USP_ERR_MISALIGNED;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return USP_ERR_MISALIGNED;
    return USP_OK;
}

// hybrid-layout view of one operand family with H heads (H/Pu per rank)
static Tensor4 hybrid_view(const void* ptr, const usp_problem* p, int Pu, int H) {
    const int64_t Nc = p->N / (p->P / Pu), Hl = H / Pu;
    return Tensor4{const_cast<void*>(ptr), Nc * p->d, p->d, Hl * Nc * p->d, (int)Hl, (int)Nc, p->P * p->B};
}

// Forward workspace: float32 running and partial outputs and the partial LSE,
// one row per (rank, batch, local head, token), in the hybrid layout.
size_t usp_hybrid_workspace_size(const usp_problem* p, int Pu) {
    if (hybrid_check(p, Pu) != USP_OK) return 0;
    const size_t rows = (size_t)p->B * p->N * p->Hq;
    return 2 * ring_part(rows * p->d * sizeof(float)) + ring_part(rows * sizeof(float));
}

usp_status usp_hybrid_attn_fwd(const usp_problem* p, int Pu, const void* q, const void* k, const void* v, void* o,
                               float* lse, void* ws, size_t ws_bytes, usp_stream stream) {
    usp_status st = hybrid_attn_checks(p, Pu, {q, k, v, o, lse}, ws);
    if (st != USP_OK || empty(p)) return st;
    if (ws_bytes < usp_hybrid_workspace_size(p, Pu)) return USP_ERR_WORKSPACE;
    int* sp = status_ptr();
    if (!sp) return USP_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int Pr = p->P / Pu, B = p->B, d = p->d, Nc = p->N / Pr, Hl = p->Hq / Pu;
    const size_t rows = (size_t)B * p->N * p->Hq;
    const size_t rows_per_group = (size_t)Pu * B * Hl * Nc;
    float* acc_o = static_cast<float*>(ws);
    float* part_o = reinterpret_cast<float*>(static_cast<char*>(ws) + ring_part(rows * d * sizeof(float)));
    float* part_l = reinterpret_cast<float*>(static_cast<char*>(ws) + 2 * ring_part(rows * d * sizeof(float)));

    // the ring decode over groups: query group i, its rank-and-batch index u*B + b as the "batch"
    // (bsz = Pu*B), so that outer index i*Pu*B + u*B + b is rank i*Pu + u, batch b
    FwdParams f{};
    f.q = hybrid_view(q, p, Pu, p->Hq);
    f.k = hybrid_view(k, p, Pu, p->Hkv);
    f.v = hybrid_view(v, p, Pu, p->Hkv);
    f.d = d;
    f.g = p->Hq / p->Hkv;
    f.n_heads = Hl;
    f.q_len = Nc;
    f.kv_len = Nc;
    f.ring_p = Pr;
    f.bsz = Pu * B;
    f.np = Nc;
    f.causal = p->causal ? 1 : 0;
    f.scale = eff_scale(p);
    f.o_s_head = (int64_t)Nc * d;
    f.o_s_tok = d;
    f.o_s_outer = (int64_t)Hl * Nc * d;
    f.l_s_head = Nc;
    f.l_s_tok = 1;
    f.l_s_outer = (int64_t)Hl * Nc;
    f.status = sp;
    return cuda_status(ring_fwd_schedule(f, Pr, Pu * B, rows, rows_per_group, acc_o, part_o, part_l, lse, o,
                                         "hybrid_attn_partial", s));
}

// Backward workspace: 40 bytes per padded query row of every (rank, batch, local head), then
// float32 accumulators for dQ, dK and dV in the hybrid layout.
static size_t hybrid_bwd_rows(const usp_problem* p, int Pu) {
    const size_t nc = (size_t)p->N / (p->P / Pu), npad = (nc + 127) / 128 * 128;
    return (size_t)p->P * p->B * (p->Hq / Pu) * npad;
}

size_t usp_hybrid_bwd_workspace_size(const usp_problem* p, int Pu) {
    if (hybrid_check(p, Pu) != USP_OK) return 0;
    const size_t k_elems = (size_t)p->B * p->N * p->Hkv * p->d;
    return ring_part(hybrid_bwd_rows(p, Pu) * 40) + ring_part(hybrid_bwd_rows(p, Pu) * p->d * 4) +
           2 * ring_part(k_elems * 4);
}

usp_status usp_hybrid_attn_bwd(const usp_problem* p, int Pu, const void* q, const void* k, const void* v,
                               const void* o, const float* lse, const void* dout, void* dq, void* dk, void* dv,
                               void* ws, size_t ws_bytes, usp_stream stream) {
    usp_status st = hybrid_attn_checks(p, Pu, {q, k, v, o, lse, dout, dq, dk, dv}, ws);
    if (st != USP_OK || empty(p)) return st;
    if (ws_bytes < usp_hybrid_bwd_workspace_size(p, Pu)) return USP_ERR_WORKSPACE;
    int* sp = status_ptr();
    if (!sp) return USP_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int Pr = p->P / Pu, B = p->B, d = p->d, Nc = p->N / Pr, Hl = p->Hq / Pu;
    const size_t k_elems = (size_t)B * p->N * p->Hkv * d;
    char* w = static_cast<char*>(ws);
    float* acc_dq = reinterpret_cast<float*>(w + ring_part(hybrid_bwd_rows(p, Pu) * 40));
    float* acc_dk = reinterpret_cast<float*>(reinterpret_cast<char*>(acc_dq) + ring_part(hybrid_bwd_rows(p, Pu) * d * 4));
    float* acc_dv = reinterpret_cast<float*>(reinterpret_cast<char*>(acc_dk) + ring_part(k_elems * 4));

    BwdParams b{};
    b.q = hybrid_view(q, p, Pu, p->Hq);
    b.o = hybrid_view(o, p, Pu, p->Hq);
    b.dout = hybrid_view(dout, p, Pu, p->Hq);
    b.k = hybrid_view(k, p, Pu, p->Hkv);
    b.v = hybrid_view(v, p, Pu, p->Hkv);
    b.lse = lse;  // [P][B][Hq/Pu][Nc], the merged LSE of usp_hybrid_attn_fwd
    b.l_s_head = Nc;
    b.l_s_tok = 1;
    b.l_s_outer = (int64_t)Hl * Nc;
    b.ws = reinterpret_cast<float*>(w);
    b.n_z = p->P * B * Hl;
    b.dq_acc = acc_dq;
    b.dk_f32 = acc_dk;
    b.dv_f32 = acc_dv;
    b.d = d;
    b.g = p->Hq / p->Hkv;
    b.ring_p = Pr;
    b.bsz = Pu * B;
    b.scale = eff_scale(p);
    b.status = sp;

    // as the ring backward, over groups: dK, dV travel with the KV chunk, dQ stays
    cudaError_t e = traced("hybrid_bwd_pre", s, [&] { return launch_bwd_pre(b, s); });
    if (e == cudaSuccess) e = ring_bwd_schedule(b, Pr, Pu * B, p->causal != 0, k_elems, dq, dk, dv, "hybrid_bwd_dkdvq", s);
    return cuda_status(e);
}

usp_status usp_trace_enable(int on) {
    std::lock_guard<std::mutex> lock(g_trace_mu);
    g_trace_on = on != 0;
    return USP_OK;
}

usp_status usp_trace_reset(void) {
    std::lock_guard<std::mutex> lock(g_trace_mu);
    for (auto& t : g_trace_pending) {
        cudaEventSynchronize(t.b);
        g_trace_pool.push_back(t.a);
        g_trace_pool.push_back(t.b);
    }
    g_trace_pending.clear();
    g_trace_acc.clear();
    return USP_OK;
}

int usp_trace_report(usp_trace_entry* out, int max_entries) {
    std::lock_guard<std::mutex> lock(g_trace_mu);
    bool failed = false;
    for (auto& t : g_trace_pending) {
        float ms = 0.f;
        if (cudaEventSynchronize(t.b) != cudaSuccess || cudaEventElapsedTime(&ms, t.a, t.b) != cudaSuccess)
            failed = true;
        TraceAcc& acc = g_trace_acc[t.name];
        acc.launches += 1;
        acc.ms += ms;
        g_trace_pool.push_back(t.a);
        g_trace_pool.push_back(t.b);
    }
    g_trace_pending.clear();
    if (failed) return -1;
    int n = 0;
    for (const auto& kv : g_trace_acc) {
        if (out && n < max_entries) {
            std::memset(out[n].name, 0, sizeof(out[n].name));
            std::strncpy(out[n].name, kv.first.c_str(), sizeof(out[n].name) - 1);
            out[n].launches = kv.second.launches;
            out[n].total_ms = kv.second.ms;
        }
        ++n;
    }
    return n;
}

}  // extern "C"

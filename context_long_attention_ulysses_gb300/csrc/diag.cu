// Failure-detection check without a fault.  Every wait in the library's
// kernels is bounded: after kWaitLimitNs it records its site in the device
// status word and the kernel returns, so that the host learns of a stalled
// pipeline from usp_device_status() and the context stays usable.  This probe
// runs that path on purpose: one CTA waits on a barrier phase that nothing
// completes, gives up after the limit and returns normally.  A second entry
// sets the status word directly, so that every CTA of the kernels launched
// after it gives up at its first wait that is not already satisfied: the
// abort path of real kernels, with their loads and MMAs in flight, which
// they drain before freeing TMEM and exiting.
#include "kernels.h"
#include "ptx.cuh"

namespace usp {

namespace {

constexpr int kProbeSite = 99;  // the site code the probe records (0x54000000 | 99)
constexpr int kRaiseSite = 98;  // the site code usp_diag_raise_status records

__global__ void __launch_bounds__(32) wait_timeout_probe_kernel(int* status) {
    __shared__ alignas(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
    }
    __syncthreads();
    // nothing arrives on the barrier, so its phase 0 never completes and the wait gives up
    if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, &abort_flag, kProbeSite, status);
    __syncthreads();
}

// Records a give-up in the status word, as a timed-out wait does.
__global__ void __launch_bounds__(32) raise_status_kernel(int* status) {
    if (threadIdx.x == 0) atomicCAS(status, 0, 0x54000000 | kRaiseSite);
}

}  // namespace

cudaError_t launch_wait_timeout_probe(int* status, cudaStream_t stream) {
    wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(status);
    return cudaGetLastError();
}

cudaError_t launch_raise_status(int* status, cudaStream_t stream) {
    raise_status_kernel<<<1, 32, 0, stream>>>(status);
    return cudaGetLastError();
}

}  // namespace usp

// Probe of the bounded-wait path every kernel's barrier waits take (the
// sm_121a hardening commit on the FastVideo kernel page: failures come back as
// error codes, never as a hung or trapped GPU).  One warp waits on an mbarrier
// phase; unless asked to, nothing arrives on it, so the wait runs out after
// its limit, raises the abort flag and sets the timeout bit of the device
// status word, and the kernel returns normally.
#include "vsa_internal.h"
#include "vsa_ptx.cuh"
#include "vsa_wait.cuh"

namespace vsa {
namespace {

__global__ void __launch_bounds__(32, 1) wait_probe_kernel(int32_t arrive, uint64_t limit_ns, int32_t *status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncwarp();
    if (arrive && threadIdx.x == 0) mbar_arrive(b);  // completes phase 0
    __syncwarp();
    wait_warp(b, 0u, &abort_flag, status, limit_ns);
}

}  // namespace

cudaError_t launch_wait_probe(int32_t arrive, uint64_t limit_ns, int32_t *status, cudaStream_t stream) {
    wait_probe_kernel<<<1, 32, 0, stream>>>(arrive, limit_ns, status);
    return cudaGetLastError();
}

}  // namespace vsa

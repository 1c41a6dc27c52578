// vsa_block_sparse_fwd_noalloc: the block-sparse forward for callers that
// cannot allocate device memory.
//
// Some callers have no way to obtain a workspace: code running where
// cudaMalloc is unavailable or forbidden (inside a host callback, in a
// process whose allocator is owned by someone else, in a plug-in that may not
// touch the device heap), or code that must not allocate between steps so
// its memory footprint stays fixed.  This entry point takes the same inputs
// and outputs as vsa_block_sparse_fwd but uses a fixed scratch area that the
// library owns: a file-scope device array of VSA_NOALLOC_SCRATCH_BYTES bytes.
// Every GPU that loads the library holds that array until the process exits.
//
// The array holds the work order and the work counter of the attention
// kernel.  The ordering kernel rewrites the order and resets the counter to
// zero at the start of every call, so no state carries over between calls
// even though the array keeps the last call's contents.  All calls on a
// device share the one array: calls that can overlap on the GPU (different
// streams without ordering between them) race and give wrong results.
#include <mutex>

#include <cuda_runtime.h>

#include "vsa.h"
#include "vsa_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[VSA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Per device: the scratch array's device address and the context it was
// looked up in.  The address belongs to that context: after cudaDeviceReset
// the module is loaded again in a new context and the array moves, so a
// changed context ID means a fresh lookup.
struct ScratchEntry {
    std::mutex lock;
    unsigned long long ctx = 0;
    void *addr = nullptr;
};
ScratchEntry g_scratch[kMaxDevices];

// Device address of the scratch array on the current device, looked up once
// per device and context (the array's name is only a host-side handle and must
// not be passed to a kernel directly).
vsa_status scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return VSA_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return VSA_ERR_ARCH;
    ScratchEntry &e = g_scratch[dev];
    std::lock_guard<std::mutex> g(e.lock);
    if (e.addr == nullptr || e.ctx != vsa::current_context_id()) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            cudaGetLastError();
            return VSA_ERR_CUDA;
        }
        if (major != 10 || minor != 3) return VSA_ERR_ARCH;
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            e.addr = nullptr;
            return VSA_ERR_CUDA;
        }
        e.addr = p;
        e.ctx = vsa::current_context_id();  // the lookup made the device's context current
    }
    *out = e.addr;
    return VSA_OK;
}

}  // namespace

extern "C" vsa_status vsa_block_sparse_fwd_noalloc(const void *q, const void *k, const void *v,
                                                   const int32_t *q2k_idx, const int32_t *q2k_num,
                                                   const int32_t *block_sizes, void *out, float *lse,
                                                   const vsa_dims *dims, vsa_stream_t stream) {
    const size_t need = vsa_block_sparse_workspace_size_min(dims);
    if (need == 0)  // invalid dims: report the same error the main entry point gives
        return vsa_block_sparse_fwd(q, k, v, q2k_idx, q2k_num, block_sizes, out, lse, dims, nullptr, 0, stream);
    if (need > (size_t)VSA_NOALLOC_SCRATCH_BYTES) return VSA_ERR_LIMITS;
    void *scratch = nullptr;
    vsa_status st = scratch_address(&scratch);
    if (st != VSA_OK) return st;
    return vsa_block_sparse_fwd(q, k, v, q2k_idx, q2k_num, block_sizes, out, lse, dims, scratch,
                                (size_t)VSA_NOALLOC_SCRATCH_BYTES, stream);
}

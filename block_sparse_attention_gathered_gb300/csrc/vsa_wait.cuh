// Pieces shared by the attention kernels: tcgen05 descriptors and bounded
// barrier waits.
#pragma once

#include "vsa_internal.h"
#include "vsa_ptx.cuh"

namespace vsa {
namespace {

using namespace ptx;

constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kSleepHintNs = 20000;  // upper bound of one sleeping try_wait

// Instruction descriptor, tcgen05.mma kind::f16: bf16 A and B, fp32 D,
// A K-major, B K-major or MN-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle (rows of 128 bytes,
// 8-row / 1024-byte swizzle atoms; buffers are 1024-byte aligned).  The start
// address sits in the low 14 bits (address >> 4), so a byte offset b is added
// to a descriptor as b >> 4.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Bounded wait on an mbarrier phase.  Returns false when the CTA is aborting
// (another role gave up) or when this wait itself ran past the limit; in the
// latter case it raises the CTA's abort flag and sets the timeout bit of the
// device status word.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                         int32_t *status, uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = 0;
    for (uint32_t it = 1;; ++it) {
        // sleep in the barrier instead of spinning: spinning warps take issue
        // slots from the softmax warps that share their SM sub-partition
        if (mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
        if ((it & 7u) == 0) {
            if (*abort_flag) return false;
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > limit_ns) {
                *abort_flag = 1;
                atomicOr(status, kFlagTimeout);
                return false;
            }
        }
    }
}

// Same bound, but polling without sleeping: for a single thread whose wait
// sits on the critical path (the MMA issuer waiting for P), where the wake-up
// delay of a sleeping wait costs more than the issue slots polling takes.
__device__ __forceinline__ bool wait_bar_spin(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                              int32_t *status) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 255u) {
            if (*abort_flag) return false;
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                atomicOr(status, kFlagTimeout);
                return false;
            }
        }
    }
}

// Warp-uniform form: every lane of the warp gets the same answer, so the
// .sync.aligned tcgen05 instructions that follow are never reached by part of
// a warp.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          int32_t *status, uint64_t limit_ns = kWaitLimitNs) {
    return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag, status, limit_ns));
}

// Wait used only while draining after an abort: ignores the abort flag, gives
// up after the limit (the copies it waits for complete on their own).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) return;
    }
}

}  // namespace
}  // namespace vsa

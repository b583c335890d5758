// Bounded mbarrier waits for the warp-specialised tensor-core kernels.
//
// Every wait gives up after kTimeoutNs of %globaltimer: it then raises the CTA's
// abort flag (seen by the other roles' waits) and records the timeout bit in the
// device error word, so a kernel whose producer or peer stopped returns instead of
// spinning forever.
#pragma once
#include <cstdint>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {
namespace tc {

constexpr uint64_t kTimeoutNs = 2000000000ull;

// Wait for the phase of `bar` with the given parity; false on timeout or when
// another role has already aborted.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                         uint32_t *err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kTimeoutNs) {
            *abort_flag = 1;
            record_error(err, kErrTimeout);
            return false;
        }
    }
}

// wait_bar for a barrier completed by a release arrival from the other CTA of the
// cluster (acquire at cluster scope).
__device__ __forceinline__ bool wait_bar_cluster(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                                 uint32_t *err) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kTimeoutNs) {
            *abort_flag = 1;
            record_error(err, kErrTimeout);
            return false;
        }
    }
}

// Wait without honouring the abort flag (used to drain work already in flight).
__device__ __forceinline__ void drain_bar(uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > kTimeoutNs) break;
}

}  // namespace tc
}  // namespace moe

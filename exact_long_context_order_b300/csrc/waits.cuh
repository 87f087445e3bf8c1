// Bounded mbarrier waits shared by the tensor-core kernels.  A wait gives up
// when the CTA's abort flag is set or after `limit` SM clock cycles; then it
// sets the flag, records kStatusTimeout in the device status word and returns
// false, so the kernel can drain its in-flight copies and MMAs and exit
// instead of hanging.
#pragma once
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace ra {

__device__ __forceinline__ bool wait_bar(uint32_t b, uint32_t parity, volatile int* abort_flag,
                                         unsigned int* status, long long limit) {
    if (mbar_try_wait(b, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(b, parity)) return true;
        if ((it & 255u) == 0) {
            if (*abort_flag) return false;
            if (clock64() - t0 > limit) {
                *abort_flag = 1;
                atomicOr(status, kStatusTimeout);
                return false;
            }
        }
    }
}

// Short bounded wait used only while draining after an abort.
__device__ __forceinline__ void drain_wait(uint32_t b, uint32_t parity, long long limit) {
    const long long t0 = clock64();
    while (!mbar_try_wait(b, parity)) {
        if (clock64() - t0 > limit) return;
    }
}

}  // namespace ra

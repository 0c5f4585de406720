// l2hint.cuh -- L2 warm-up hint shared by the GEMV and dequant kernels.
#pragma once

#include <stdint.h>

namespace qmm {

// Warm L2 with the 16-byte units inside [a0, a1) (both ends rounded down to
// 16 bytes, so nothing outside the range is touched), 64 KB per request.  A
// cache hint: harmless even while a kernel still running writes the range.
__device__ __forceinline__ void prefetch_l2_range(uintptr_t a0, uintptr_t a1) {
    a0 &= ~uintptr_t(15);
    a1 &= ~uintptr_t(15);
    for (uintptr_t a = a0; a < a1; a += 65536) {
        const uintptr_t len = (a1 - a) < 65536 ? (a1 - a) : 65536;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(static_cast<uint64_t>(a)),
                     "r"(static_cast<uint32_t>(len))
                     : "memory");
    }
}

}  // namespace qmm

// Device helpers shared by the tensor-core kernels.
#pragma once

#include <cstdint>

#include "sm103_ptx.cuh"

namespace fa {
namespace tc {

using namespace ptx;

// A bounded wait that also returns early once another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                              volatile int *abort_flag)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t spin = 1;; ++spin) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((spin & 63u) == 0u) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > limit_ns) return false;
        }
    }
}

// The same wait made by a whole warp: every lane waits, and the warp leaves
// converged with one verdict (true only if every lane saw the phase).
__device__ __forceinline__ bool wait_or_abort_w(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                                volatile int *abort_flag)
{
    const bool done = wait_or_abort(bar, parity, limit_ns, abort_flag);
    return __all_sync(0xffffffffu, done);
}

// Maximum of 128 scores: eight independent chains of three-input maxima,
// then a short combine (depth 11 instead of a 127-long dependency chain).
__device__ __forceinline__ float row_max_128(const float (&s)[128])
{
    float a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = max3f(s[16 * i], s[16 * i + 1], s[16 * i + 2]);
#pragma unroll
    for (int k = 3; k < 15; k += 2)
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] = max3f(a[i], s[16 * i + k], s[16 * i + k + 1]);
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = fmaxf(a[i], s[16 * i + 15]);
    return max3f(max3f(a[0], a[1], a[2]), max3f(a[3], a[4], a[5]), fmaxf(a[6], a[7]));
}

}  // namespace tc
}  // namespace fa

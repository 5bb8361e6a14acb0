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
// converged with one outcome (true only if every lane saw the phase).
__device__ __forceinline__ bool wait_or_abort_w(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                                volatile int *abort_flag)
{
    const bool done = wait_or_abort(bar, parity, limit_ns, abort_flag);
    return __all_sync(0xffffffffu, done);
}

// wait_or_abort with cluster-scope acquire, for barriers other CTAs of the
// cluster arrive on; polls without suspending.
__device__ __forceinline__ bool wait_or_abort_cluster(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                                      volatile int *abort_flag)
{
    if (mbar_test_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t spin = 1;; ++spin) {
        if (mbar_test_wait_cluster(bar, parity)) return true;
        if ((spin & 63u) == 0u) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > limit_ns) return false;
        }
    }
}

// Maximum of NV scores (NV a multiple of 8): eight independent chains of
// three-input maxima, then a short combine (depth about NV / 16 + 3 instead
// of an NV-long dependency chain).
template <int NV>
__device__ __forceinline__ float row_max(const float (&s)[NV])
{
    static_assert(NV % 8 == 0 && NV >= 16, "row_max: NV must be a multiple of 8, at least 16");
    constexpr int C = NV / 8;
    float a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = s[i * C];
#pragma unroll
    for (int k = 1; k + 1 < C; k += 2)
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] = max3f(a[i], s[i * C + k], s[i * C + k + 1]);
    if constexpr (C % 2 == 0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] = fmaxf(a[i], s[i * C + C - 1]);
    }
    return max3f(max3f(a[0], a[1], a[2]), max3f(a[3], a[4], a[5]), fmaxf(a[6], a[7]));
}

__device__ __forceinline__ float row_max_128(const float (&s)[128]) { return row_max<128>(s); }

}  // namespace tc
}  // namespace fa

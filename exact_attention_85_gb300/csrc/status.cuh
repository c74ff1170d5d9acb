// status.cuh -- the per-device status word written by bounded waits.
#pragma once

#include <cstdint>

namespace fa {

// Bit 31 marks a timeout; the low bits keep the site code of the first wait
// that ran out (a small integer naming the barrier, for diagnosis).
constexpr unsigned int kStatusTimeout = 0x80000000u;

// Bit 30 marks device-side arguments found invalid by a kernel (packed
// sequence offsets that are not a non-decreasing prefix sum within bounds);
// the kernel then skips the affected work instead of reading out of range.
constexpr unsigned int kStatusBadArgs = 0x40000000u;

__device__ __forceinline__ void record_timeout(unsigned int *status, uint32_t site) {
    if (status) atomicCAS(status, 0u, kStatusTimeout | (site & 0xFFFFu));
}

__device__ __forceinline__ void record_bad_args(unsigned int *status) {
    if (status) atomicOr(status, kStatusBadArgs);
}

}  // namespace fa

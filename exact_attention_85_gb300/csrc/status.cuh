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

// Bit 29 marks a kernel that found its dynamic shared-memory window too far
// from a 1024-byte boundary for its 128-byte-swizzled operand tiles; the
// kernel then does nothing (a launch-configuration failure, not a timeout).
constexpr unsigned int kStatusBadLaunch = 0x20000000u;

// The first timeout also records its site; other bits already set (bad
// arguments, bad launch) do not stop a timeout from being recorded.
__device__ __forceinline__ void record_timeout(unsigned int *status, uint32_t site) {
    if (!status) return;
    const unsigned int old = atomicOr(status, kStatusTimeout);
    if (!(old & kStatusTimeout)) atomicOr(status, site & 0xFFFFu);
}

__device__ __forceinline__ void record_bad_args(unsigned int *status) {
    if (status) atomicOr(status, kStatusBadArgs);
}

__device__ __forceinline__ void record_bad_launch(unsigned int *status) {
    if (status) atomicOr(status, kStatusBadLaunch);
}

}  // namespace fa

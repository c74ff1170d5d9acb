// status.cuh -- the per-device status words written by kernels.
//
// Word 0 records timeouts of bounded waits; word 1 collects the other
// conditions.  Keeping them apart lets a timeout be recorded with one
// compare-and-swap on a word nothing else writes, which keeps the wait loops
// (inlined in every kernel) as small as they can be.
#pragma once

#include <cstdint>

namespace fa {

// Word 0: bit 31 marks a timeout; the low bits keep the site code of the
// first wait that ran out (a small integer naming the barrier, for
// diagnosis).
constexpr unsigned int kStatusTimeout = 0x80000000u;

// Word 1, bit 30: device-side arguments found invalid by a kernel (packed
// sequence offsets that are not a non-decreasing prefix sum within bounds);
// the kernel then skips the affected work instead of reading out of range.
constexpr unsigned int kStatusBadArgs = 0x40000000u;

// Word 1, bit 29: a kernel found its dynamic shared-memory window too far
// from a 1024-byte boundary for its 128-byte-swizzled operand tiles; the
// kernel then does nothing (a launch-configuration failure, not a timeout).
constexpr unsigned int kStatusBadLaunch = 0x20000000u;

// `status` is the address of word 0 (word 1 follows it).
__device__ __forceinline__ void record_timeout(unsigned int *status, uint32_t site) {
    if (status) atomicCAS(status, 0u, kStatusTimeout | (site & 0xFFFFu));
}

__device__ __forceinline__ void record_bad_args(unsigned int *status) {
    if (status) atomicOr(status + 1, kStatusBadArgs);
}

__device__ __forceinline__ void record_bad_launch(unsigned int *status) {
    if (status) atomicOr(status + 1, kStatusBadLaunch);
}

}  // namespace fa

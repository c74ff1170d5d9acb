// status.cuh -- the per-device status word written by bounded waits.
#pragma once

#include <cstdint>

namespace fa {

// Bit 31 marks a timeout; the low bits keep the site code of the first wait
// that ran out (a small integer naming the barrier, for diagnosis).
constexpr unsigned int kStatusTimeout = 0x80000000u;

__device__ __forceinline__ void record_timeout(unsigned int *status, uint32_t site) {
    if (status) atomicCAS(status, 0u, kStatusTimeout | (site & 0xFFFFu));
}

}  // namespace fa

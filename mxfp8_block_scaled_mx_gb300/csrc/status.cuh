// status.cuh -- the device status word: kernels record faults they detect
// (a pipeline wait that timed out, invalid group offsets) by OR-ing a bit
// into a 32-bit word in device memory; mx_device_status() reads and clears it.
#pragma once

#include <cstdint>

namespace mx {

enum : uint32_t {
  MX_DEV_TIMEOUT = 1u,      // a bounded mbarrier wait gave up
  MX_DEV_BAD_OFFSETS = 2u,  // group offsets not 0 = o_0 <= ... <= o_G = total
};

__device__ __forceinline__ void record_device_status(uint32_t* status, uint32_t code) {
  atomicOr(status, code);
}

}  // namespace mx

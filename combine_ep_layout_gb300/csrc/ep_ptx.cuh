// ep_ptx.cuh -- small inline-PTX helpers shared by the kernels.
#pragma once

#include <cstdint>

namespace epg {

// Bit mask of the lanes below the calling lane.
__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

}  // namespace epg

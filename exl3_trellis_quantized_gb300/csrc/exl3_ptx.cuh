// exl3_ptx.cuh -- small address helpers shared by the EXL3 kernels.
#pragma once

#include <stdint.h>

namespace exl3 {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

}  // namespace exl3

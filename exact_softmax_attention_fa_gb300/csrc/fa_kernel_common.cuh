// Small device helpers shared by the attention kernels: the timeout record
// and fp32 global reductions.
#pragma once

#include <cstdint>

#include "fa.h"

namespace fa {

// Record the first timed-out wait of the launch in the device status word
// ([0] code, [1] role, [2] block, [3] thread) and raise the CTA's abort flag.
__device__ __forceinline__ void record_timeout(uint32_t* status, int* abort_flag, uint32_t where) {
  if (atomicCAS(status, 0u, static_cast<uint32_t>(FA_ERR_TIMEOUT)) == 0u) {
    status[1] = where;
    status[2] = blockIdx.x;
    status[3] = threadIdx.x;
  }
  *reinterpret_cast<volatile int*>(abort_flag) = 1;
}

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

__device__ __forceinline__ void red_add_f32(float* addr, float a) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(a) : "memory");
}

__device__ __forceinline__ float4 ldg_f4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }

}  // namespace fa

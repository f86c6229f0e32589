// Small device helpers shared by the attention kernels: the timeout record
// and fp32 global reductions.
#pragma once

#include <cstdint>

#include "fa.h"
#include "sm103_ptx.cuh"

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

// Waits after an abort for work this CTA has already issued (TMA copies, MMAs
// committed to a barrier). Such work always completes, so these waits do not
// use the caller's wait limit, which may be a few milliseconds; they are still
// bounded, at the larger of that limit and one second.
constexpr uint64_t kDrainLimitNs = 1000000000ull;
__device__ __forceinline__ uint64_t drain_limit(uint64_t lim) { return lim > kDrainLimitNs ? lim : kDrainLimitNs; }

// Wait for the latest phase of a barrier whose arrival (a TMA copy's bytes,
// an MMA commit) was issued earlier; the abort flag is not consulted. (A
// variant that slept between polls, inlined or called, raised the kernels'
// register pressure and spills on their per-tile paths: the d = 256
// backward ran 13 % slower.)
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t lim) {
  const int zero = 0;
  mbar_wait(bar, parity, &zero, drain_limit(lim));
}

// MMA issuer leaving early: every tcgen05 MMA it issued must complete before
// the CTA frees its tensor memory and shared memory. `bar` is a barrier of
// count 1 used for nothing else (one phase per kernel).
__device__ __forceinline__ void drain_mmas(uint64_t* bar, uint64_t lim) {
  umma_commit(bar);
  drain_wait(bar, 0, lim);
}

// Test hook (fa_debug_skip_arrival in fa.h), in two forms that cost nothing
// on the kernels' per-tile paths: a load role leaves out one of its copies
// (debug_skip_here, checked once per item), and an MMA or softmax role's
// barrier is initialised in block 0 to expect one more arrival than the role
// makes (debug_extra), so the first wait on it gives up.
__device__ __forceinline__ bool debug_skip_here(uint32_t debug_skip, uint32_t role, bool first) {
  return debug_skip == role && first && blockIdx.x == 0;
}
__device__ __forceinline__ uint32_t debug_extra(uint32_t debug_skip, uint32_t role) {
  return debug_skip == role && blockIdx.x == 0 ? 1u : 0u;
}

__device__ __forceinline__ void red_add_f32(float* addr, float a) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(a) : "memory");
}

__device__ __forceinline__ float4 ldg_f4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }

// ---------------------------------------------------------------------------
// Work-item queue of a persistent kernel. CTA b starts on item b; afterwards
// its producer thread claims item G + atomicAdd(ctr[0], 1) and publishes it
// through kItemSlots smem slots (item_ring, item_full, item_empty of the
// kernel's shared struct) to the CTA's consumer threads. An item >= the item
// count ends every role's loop. ctr[1] counts CTAs done claiming; the last
// one resets both words for the next launch.
// ---------------------------------------------------------------------------
constexpr int kItemSlots = 4;

template <class Shared>
__device__ __forceinline__ bool publish_item(Shared& sh, int u, int item, uint64_t lim) {
  const int s = u % kItemSlots;
  if (u >= kItemSlots && !mbar_wait(&sh.item_empty[s], ((u / kItemSlots) - 1) & 1, &sh.abort_flag, lim))
    return false;
  *reinterpret_cast<volatile int*>(&sh.item_ring[s]) = item;
  mbar_arrive(&sh.item_full[s]);
  return true;
}

// The u-th item of this CTA, or -1 if the wait timed out.
template <class Shared>
__device__ __forceinline__ int take_item(Shared& sh, int u, uint64_t lim) {
  const int s = u % kItemSlots;
  if (!mbar_wait(&sh.item_full[s], (u / kItemSlots) & 1, &sh.abort_flag, lim)) return -1;
  const int item = *reinterpret_cast<volatile int*>(&sh.item_ring[s]);
  mbar_arrive(&sh.item_empty[s]);
  return item;
}

__device__ __forceinline__ int claim_item(uint32_t* ctr) {
  return static_cast<int>(gridDim.x) + static_cast<int>(atomicAdd(ctr, 1u));
}

__device__ __forceinline__ void finish_claiming(uint32_t* ctr) {
  if (atomicAdd(ctr + 1, 1u) == gridDim.x - 1) {
    atomicExch(ctr, 0u);
    atomicExch(ctr + 1, 0u);
  }
}

}  // namespace fa

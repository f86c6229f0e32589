// Internal interfaces between the C-ABI layer (fa_api.cu) and the kernel
// translation units. Host-side only; no torch types anywhere.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa.h"

namespace fa {

// Device status word layout (4 x uint32): [0] first error code, [1] where
// (role id), [2] blockIdx.x, [3] threadIdx.x.
enum : uint32_t {
  WHERE_FWD_LOAD = 1,
  WHERE_FWD_MMA = 2,
  WHERE_FWD_SOFTMAX = 3,
  WHERE_BWD_LOAD = 11,
  WHERE_BWD_MMA = 12,
  WHERE_BWD_SOFTMAX = 13,
  WHERE_BWD_DQ = 14,
  WHERE_PROBE = 99,
};

// Tiles of the [B*H][N][d] bf16 tensors, as seen by TMA: 128 rows x 64
// columns per box, 128-byte swizzle.
struct FwdLaunch {
  CUtensorMap tmQ, tmK, tmV, tmO;
  float* lse;
  uint32_t* status;
  int Nq, Nk, BH, d, causal;
  int causal_off;    // Nk - Nq: query i sees key j iff j <= i + causal_off (bottom-right alignment)
  int splits;        // key ranges per query tile; > 1: partial results go to o_part / lse_part
  int kv_per_split;  // 128-key tiles per range
  float* o_part;     // splits > 1: fp32 O of each range [splits][BH][Nq][d], normalised by its own l
  float* lse_part;   // splits > 1: [splits][BH][Nq], natural log; the combine kernel merges them
  __nv_bfloat16* o;  // [BH][Nq][d]: written by the combine kernel (splits > 1)
  int group;         // query heads per K/V head: query head bh reads K/V head bh / group
  int pack;          // query heads sharing one 128-row tile (1, or the group when query blocks are short)
  int rph;           // query positions per head in a tile: 128 / pack
  float scale_log2;  // scale * log2(e): scores are exponentiated in base 2
  uint64_t wait_limit_ns;
  int num_sms;
  uint32_t debug_skip;  // test hook: role (WHERE_*) whose first arrival block 0 leaves out; 0 = none
};

struct BwdLaunch {
  CUtensorMap tmQ, tmK, tmV, tmdO, tmdK, tmdV;
  CUtensorMap tmdQacc;  // fp32 [BH][Npad][d] accumulator, 128 rows x 32 columns per box
  const __nv_bfloat16* o;
  const __nv_bfloat16* dO;
  const float* lse;
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;  // [BH][N][d]
  __nv_bfloat16* dv;  // [BH][N][d]
  float* D;       // [BH][Npad]
  float* lse2;    // [BH][Npad], base-2 logsumexp (+inf on padding rows)
  float* dq_acc;  // [BH][Npad][d]
  uint32_t* sched;  // [4]: main kernel's next work item and CTAs done claiming; the same for the dQ kernel
  int deterministic; // 1: dQ from the separate dQ kernel (no atomics); the main kernel skips it
  uint32_t* status;
  int N, Npad, BH, d, causal;
  int BHkv, group;   // K/V heads (B * H_kv) and query heads per K/V head
  int chunks;        // work items per (K/V head, key tile): the group split into chunks of group/chunks heads
  float* kv_part;    // chunks > 1: fp32 partial dK [chunks][BHkv][N][d], then partial dV likewise
  float scale;       // softmax scale (dK, dQ carry it)
  float scale_log2;  // scale * log2(e)
  uint64_t wait_limit_ns;
  int num_sms;
  uint32_t debug_skip;  // test hook: role (WHERE_*) whose first arrival block 0 leaves out; 0 = none
  // 1: the dQ kernel is launched to overlap the kernel before it in the
  // stream, which must be the dK/dV pass of the same call (it reads nothing
  // that pass writes); it still completes only after that pass has.
  int overlap_prev;
};

// Checks of the sizes, flag and scale common to every entry point; *empty is
// set when the problem has no rows (fa_api.cu).
fa_status_t check_common(int B, int H, int N, int d, int causal, float scale, bool* empty);


// Launchers (defined in the kernel translation units). Return cudaSuccess or
// the launch error.
cudaError_t launch_fwd(const FwdLaunch& a, cudaStream_t stream);
cudaError_t launch_fwd_combine(const FwdLaunch& a, cudaStream_t stream);  // splits > 1: merge the partials
cudaError_t launch_fwd_packed(const FwdLaunch& a, cudaStream_t stream);   // fa_fwd_pack.cu: pack > 1
cudaError_t launch_bwd_pre(const BwdLaunch& a, cudaStream_t stream);   // D, base-2 L, zero dQ accumulator
cudaError_t launch_bwd_main(const BwdLaunch& a, cudaStream_t stream);  // dK, dV; dQ into the accumulator
cudaError_t launch_bwd_post(const BwdLaunch& a, cudaStream_t stream);  // dQ = bf16(accumulator)
cudaError_t launch_bwd_main_d256(const BwdLaunch& a, cudaStream_t stream);  // fa_bwd256.cu
cudaError_t launch_bwd_dq(const BwdLaunch& a, cudaStream_t stream);  // fa_bwd_dq.cu: dq without atomics
cudaError_t launch_bwd_dq256(const BwdLaunch& a, cudaStream_t stream);  // fa_bwd_dq256.cu: the same at d = 256
cudaError_t launch_timeout_probe(uint32_t* status, uint64_t limit_ns, cudaStream_t stream);

}  // namespace fa

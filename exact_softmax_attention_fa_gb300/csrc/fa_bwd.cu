// Backward pass of exact softmax attention for sm_103a.
//
// Method (web pages on FlashAttention-2):
//   "FlashAttention 2: ..." reading note (papers.chlience.com) 5.3 and the
//   paper-graph-ui summary, "The Backward Pass": precompute
//   D_i = sum_k dO_ik O_ik; then, with key blocks OUTER (dK_j, dV_j stay on
//   chip) and query blocks inner: S = Q_i K_j^T, P = exp(S - L_i),
//   dV_j += P^T dO_i, dP = dO_i V_j^T, dS = P o (dP - D_i),
//   dQ_i += dS K_j (accumulated across key blocks with atomic adds, reading
//   note 5.4), dK_j += dS^T Q_i.
//
// GB300 mapping (our design):
//   Three kernels on the caller's stream (the deterministic backward runs
//   the first, the second without dQ, and the dQ kernel of fa_bwd_dq.cu):
//   1. bwd_pre_kernel (HBM-bound): D from the stored bf16 O and dO, the
//      base-2 logsumexp L*log2(e), and zeroes the fp32 dQ accumulator. Every
//      head is padded to a multiple of 128 rows; padding rows get D = 0 and
//      L = +inf so their probabilities are exactly 0.
//   2. fa_bwd_kernel: persistent, one CTA per SM taking work items
//      (head, 128-key tile j) from a global counter (causal: longest first).
//      Everything is computed transposed, with keys on the 128 TMEM lanes:
//        S^T = K_j Q_i^T and dP^T = V_j dO_i^T   (SS MMAs into TMEM)
//        two softmax warpgroups, each owning 64 of the tile's queries; thread
//          r = key r: P^T = 2^(S^T scale log2e - L log2e) and
//          dS^T = P^T o (dP^T - D) * scale; P^T (bf16) goes back to TMEM,
//          dS^T (bf16) to a 128-byte-swizzled smem tile
//        dV += P^T dO_i      (A = P^T from TMEM, B = dO_i MN-major)
//        dK += dS^T Q_i      (A = dS^T smem, K-major; B = Q_i MN-major)
//        dQ_i (d = 64) = dS K_j, or dQ_i^T (d = 128) = K_j^T dS^T, from the
//          same smem tile read MN-major, into TMEM; the softmax warpgroups
//          drain it into the fp32 accumulator with reductions (d = 128:
//          scalar reductions that cover whole 128-byte lines; d = 64: TMA
//          reduce-adds of a swizzled smem staging tile).
//      Two 128-column TMEM regions with fixed roles: region 0 holds S^T(i)
//      and then P^T(i), region 1 dP^T(i) and then dQ_i; S^T(i+1) reuses
//      region 0 once dV(i) is done and dP^T(i+1) reuses region 1 once dQ_i
//      was drained. dK, dV (fp32, TMEM) are written once per item, straight
//      from TMEM to global memory (or, when a group's query heads are split
//      into chunks, as fp32 partials that bwd_kv_sum_kernel adds in chunk
//      order), while the MMA warp starts the next item.
//      The DQ = false instantiation skips the dQ product and drain: the
//      deterministic backward (fa_bwd at d = 128) forms dQ in fa_bwd_dq.cu.
//   3. bwd_post_kernel (HBM-bound): dQ = bf16(accumulator).
//
// TMEM columns (512 allocated): dK [0, d), dV [d, 2d), region 0 [256, 384),
// region 1 [384, 512).
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "fa_internal.h"
#include "fa_kernel_common.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

// Warps: 0-3 and 4-7 softmax + dQ drain (query columns 0-63 / 64-127),
// 8 TMA loads, 9 MMA issue.
constexpr int kThreads = 320;
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr float kLog2e = 1.44269504088896340736f;

template <int HD>
struct BwdCfg {
  static constexpr int CHUNKS = HD / 64;
  static constexpr int TILE_BYTES = 128 * HD * 2;
  static constexpr int CHUNK_BYTES = 128 * 128;
  static constexpr int QST = HD == 64 ? 3 : 2;  // Q_i / dO_i pipeline stages
  static constexpr int DS_BYTES = 128 * 128 * 2;
  static constexpr uint32_t DK_COL = 0;
  static constexpr uint32_t DV_COL = HD;
  static constexpr uint32_t REG_A = 256;  // S^T, then P^T (bf16)
  static constexpr uint32_t REG_B = 384;  // dP^T, then dQ_i (d = 128: dQ_i^T)
  static constexpr bool DQ_T = HD == 128;
  // d = 64: dQ_i is staged in smem (fp32, two 128 x 32 swizzled chunks, one
  // per warpgroup) and added to the accumulator by TMA reduce-adds.
  static constexpr bool DQ_TMA = HD == 64;
  static constexpr int DQS_BYTES = DQ_TMA ? 128 * 64 * 4 : 0;
  static constexpr int LD_BYTES = 2 * 128 * 4;  // per warpgroup: 64 base-2 L + 64 scaled D
  // smem: K_j, V_j, QST x (Q_i, dO_i), dS^T, L/D staging
  static constexpr int SMEM_BYTES = (2 + 2 * QST) * TILE_BYTES + DS_BYTES + LD_BYTES + DQS_BYTES + 1024;
};

struct BwdShared {
  uint64_t kv_full;
  uint64_t qdo_full[4], qdo_empty[4];
  uint64_t s_full, dp_full, pa_ready, ds_ready, pv_done, dq_full, dq_free, acc_done;
  uint64_t acc_free;  // dK, dV of the previous item read out of TMEM
  uint64_t mma_drain;  // the MMA thread's last commit: all its MMAs done before the CTA exits
  // Work-item queue filled by the load thread (item >= BH*T ends the loop).
  uint64_t item_full[4], item_empty[4];
  int item_ring[4];
  uint32_t tmem_base;
  int abort_flag;
};

// Work item: key tile j of K/V head bh and chunk c of the g query heads that
// share it (query head bh*g + t reads K/V head bh; a group is split into
// `chunks` chunks of gs = g / chunks heads). Its query stream is, for each
// query head of the chunk, query tiles i0..T-1 (causal: i0 = j); dK_j and dV_j
// accumulate over all of them. Causal items are numbered most-work-first (key
// tile j meets T - j query tiles per head); non-causal items of one chunk are
// adjacent (Q/dO reuse in L2).
template <bool CAUSAL>
struct BwdWork {
  int bh, c, j, i0, T, nq, gs, q0;
  __device__ BwdWork(int item, int BHkv, int N, int g, int chunks) {
    T = (N + 127) / 128;
    int unit;  // bh * chunks + c
    if (CAUSAL) {
      unit = item % (BHkv * chunks);
      j = item / (BHkv * chunks);
    } else {
      unit = item / T;
      j = item % T;
    }
    bh = unit / chunks;
    c = unit - bh * chunks;
    gs = g / chunks;
    q0 = bh * g + c * gs;
    i0 = CAUSAL ? j : 0;
    nq = T - i0;
  }
  __device__ int n_iter() const { return gs * nq; }
  // (query head, query tile) of a step of the query stream, advanced in order
  // (no per-step division on the softmax warps' path)
  struct Pos {
    int bh, i;
  };
  __device__ Pos first() const { return Pos{q0, i0}; }
  __device__ void advance(Pos& p) const {
    if (++p.i == T) {
      p.i = i0;
      ++p.bh;
    }
  }
};

// Dynamic schedule (fa_kernel_common.cuh): items are claimed from sched[0..1]
// of the workspace, so CTAs that run ahead take more items and causal items
// come heaviest first. Consumers of the item queue: the MMA thread and the
// 256 softmax threads.
constexpr int kItemConsumers = 1 + 256;

// Grouped K/V heads split over several work items: dK, dV = bf16 of the sum
// of the chunks' fp32 partials, added in chunk order (bitwise reproducible).
// Thread v handles 8 consecutive elements of dK (v < n8) or dV.
__global__ void __launch_bounds__(256) bwd_kv_sum_kernel(const float* __restrict__ part,
                                                         __nv_bfloat16* __restrict__ dk,
                                                         __nv_bfloat16* __restrict__ dv, int chunks, long long n8) {
  const long long v = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (v >= 2 * n8) return;
  const bool is_v = v >= n8;
  const long long e = (is_v ? v - n8 : v) * 8;  // element offset in [BHkv][N][d]
  const size_t len = static_cast<size_t>(n8) * 8;
  const float* src = part + (is_v ? static_cast<size_t>(chunks) * len : 0) + e;
  float4 a = ldg_f4(src), b = ldg_f4(src + 4);
  for (int c = 1; c < chunks; ++c) {
    const float4 a2 = ldg_f4(src + c * len), b2 = ldg_f4(src + c * len + 4);
    a.x += a2.x; a.y += a2.y; a.z += a2.z; a.w += a2.w;
    b.x += b2.x; b.y += b2.y; b.z += b2.z; b.w += b2.w;
  }
  uint4 out;
  out.x = pack_bf16x2(a.x, a.y);
  out.y = pack_bf16x2(a.z, a.w);
  out.z = pack_bf16x2(b.x, b.y);
  out.w = pack_bf16x2(b.z, b.w);
  *reinterpret_cast<uint4*>((is_v ? dv : dk) + e) = out;
}

// ---------------------------------------------------------------------------
// 1. preprocess
// ---------------------------------------------------------------------------
// One group of d/8 lanes per padded row: D = sum(dO * O) in fp32 from bf16,
// lse2 = L * log2(e) (+inf on padding rows), dq_acc row = 0.
template <int HD>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                      const __nv_bfloat16* __restrict__ dO,
                                                      const float* __restrict__ lse, float* __restrict__ D,
                                                      float* __restrict__ lse2, float* __restrict__ dq_acc,
                                                      uint32_t* __restrict__ sched, int N, int Npad,
                                                      long long total_rows) {
  if (blockIdx.x == 0 && threadIdx.x < 4) sched[threadIdx.x] = 0u;
  constexpr int LPR = HD / 8;  // lanes per row, 16 bytes of O and dO each
  constexpr int RPW = 32 / LPR;
  const long long row = (static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32) * RPW +
                        (threadIdx.x % 32) / LPR;
  const int sub = threadIdx.x % LPR;
  float acc = 0.f;
  const bool in_range = row < total_rows;
  long long bh = 0;
  int n = 0;
  if (in_range) {
    bh = row / Npad;
    n = static_cast<int>(row - bh * Npad);
    if (n < N) {
      const size_t off = (static_cast<size_t>(bh) * N + n) * HD + sub * 8;
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(o + off));
      const uint4 b = __ldg(reinterpret_cast<const uint4*>(dO + off));
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 fa = __bfloat1622float2(a2[k]);
        const float2 fb = __bfloat1622float2(b2[k]);
        acc = fmaf(fa.x, fb.x, acc);
        acc = fmaf(fa.y, fb.y, acc);
      }
    }
    if (dq_acc) {  // null when dQ is formed without the accumulator
      float4* z = reinterpret_cast<float4*>(dq_acc + static_cast<size_t>(row) * HD + sub * 8);
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
#pragma unroll
  for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (in_range && sub == 0) {
    D[row] = acc;
    lse2[row] = n < N ? lse[static_cast<size_t>(bh) * N + n] * kLog2e : INFINITY;
  }
}

// ---------------------------------------------------------------------------
// 3. postprocess: dq = bf16(dq_acc) on the real rows
// ---------------------------------------------------------------------------
template <int HD>
__global__ void __launch_bounds__(256) bwd_post_kernel(const float* __restrict__ dq_acc,
                                                       __nv_bfloat16* __restrict__ dq, int N, int Npad,
                                                       long long total_vec) {
  const long long v = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;  // 8 elements each
  if (v >= total_vec) return;
  constexpr int VPR = HD / 8;
  const long long row = v / VPR;  // row of [BH][N]
  const int sub = static_cast<int>(v - row * VPR);
  const long long bh = row / N;
  const int n = static_cast<int>(row - bh * N);
  const float* src = dq_acc + (static_cast<size_t>(bh) * Npad + n) * HD + sub * 8;
  const float4 a = ldg_f4(src), b = ldg_f4(src + 4);
  uint4 out;
  out.x = pack_bf16x2(a.x, a.y);
  out.y = pack_bf16x2(a.z, a.w);
  out.z = pack_bf16x2(b.x, b.y);
  out.w = pack_bf16x2(b.z, b.w);
  *reinterpret_cast<uint4*>(dq + static_cast<size_t>(row) * HD + sub * 8) = out;
}

// ---------------------------------------------------------------------------
// 2. main kernel roles
// ---------------------------------------------------------------------------
// TMA producer (one thread). Per item: the first Q_i/dO_i tile, then K_j and
// V_j once every MMA of the previous item has completed (they read the old
// K_j/V_j), then the remaining Q_i/dO_i tiles through the ring (global tile
// counter g).
template <int HD, bool CAUSAL>
__device__ void bwd_load_role(const BwdLaunch& p, BwdShared& sh, uint8_t* sK, uint8_t* sV, uint8_t* sQ,
                              uint8_t* sdO) {
  using C = BwdCfg<HD>;
  tma_prefetch_desc(&p.tmQ);
  tma_prefetch_desc(&p.tmK);
  tma_prefetch_desc(&p.tmV);
  tma_prefetch_desc(&p.tmdO);
  tma_prefetch_desc(&p.tmdQacc);
  const int T = (p.N + 127) / 128;
  const int total = p.BHkv * p.chunks * T;
  const uint64_t lim = p.wait_limit_ns;
  int g = 0, items = 0, issued = 0, kv_issued = 0;
  bool aborted = false;
  auto load_qdo = [&](int gg, int i, int bh) -> bool {
    const int s = gg % C::QST;
    if (gg >= C::QST && !mbar_wait(&sh.qdo_empty[s], ((gg / C::QST) - 1) & 1, &sh.abort_flag, lim)) return false;
    mbar_arrive_expect_tx(&sh.qdo_full[s], 2 * C::TILE_BYTES);
#pragma unroll
    for (int c = 0; c < C::CHUNKS; ++c) {
      tma_load_3d(sQ + s * C::TILE_BYTES + c * C::CHUNK_BYTES, &p.tmQ, &sh.qdo_full[s], c * 64, i * 128, bh);
      tma_load_3d(sdO + s * C::TILE_BYTES + c * C::CHUNK_BYTES, &p.tmdO, &sh.qdo_full[s], c * 64, i * 128, bh);
    }
    ++issued;
    return true;
  };
  int item = blockIdx.x;  // the grid never exceeds the item count
  while (!aborted) {
    if (!publish_item(sh, items, item, lim)) {
      aborted = true;
      break;
    }
    if (item >= total) break;
    const BwdWork<CAUSAL> wk(item, p.BHkv, p.N, p.group, p.chunks);
    const int n_iter = wk.n_iter();
    typename BwdWork<CAUSAL>::Pos pos = wk.first();
    if (!load_qdo(g, pos.i, pos.bh)) {
      aborted = true;
      break;
    }
    if (items > 0 && !mbar_wait(&sh.acc_done, (items - 1) & 1, &sh.abort_flag, lim)) {
      aborted = true;
      break;
    }
    if (!debug_skip_here(p.debug_skip, WHERE_BWD_LOAD, items == 0)) {  // test hook
      mbar_arrive_expect_tx(&sh.kv_full, 2 * C::TILE_BYTES);
#pragma unroll
      for (int c = 0; c < C::CHUNKS; ++c) {
        tma_load_3d(sK + c * C::CHUNK_BYTES, &p.tmK, &sh.kv_full, c * 64, wk.j * 128, wk.bh);
        tma_load_3d(sV + c * C::CHUNK_BYTES, &p.tmV, &sh.kv_full, c * 64, wk.j * 128, wk.bh);
      }
      ++kv_issued;
    }
    for (int n = 1; n < n_iter; ++n) {
      wk.advance(pos);
      if (!load_qdo(g + n, pos.i, pos.bh)) {
        aborted = true;
        break;
      }
    }
    g += n_iter;
    ++items;
    if (!aborted) item = claim_item(p.sched);
  }
  finish_claiming(p.sched);
  if (aborted) record_timeout(p.status, &sh.abort_flag, WHERE_BWD_LOAD);
  // The copies already issued land before the CTA can exit (after an abort
  // no consumer may wait for them).
  for (int n = max(0, issued - C::QST); n < issued; ++n)
    drain_wait(&sh.qdo_full[n % C::QST], (n / C::QST) & 1, lim);
  if (kv_issued > 0) drain_wait(&sh.kv_full, (kv_issued - 1) & 1, lim);
}

// One thread issues every MMA. Per query tile n of an item (global index g;
// region A: S^T then P^T; region B: dP^T then dQ_n):
//   dV += P^T dO_n        after phase A(n)          (overlaps phase B(n))
//   S^T(n+1) -> A         after dV(n) released P^T (overlaps phase B(n))
//   dK += dS^T Q_n        after phase B(n)          (overlaps phase A(n+1))
//   dQ_n -> B             after phase B(n)          (overlaps phase A(n+1))
//   dP^T(n+1) -> B        after the dQ_n drain
// An item's first dV/dK (which overwrite the accumulators) wait until the
// previous item's epilogue has read dK/dV out of TMEM.
template <int HD, bool CAUSAL, bool DQ>
__device__ void bwd_mma_role(const BwdLaunch& p, BwdShared& sh, uint8_t* sK, uint8_t* sV, uint8_t* sQ,
                             uint8_t* sdO, uint8_t* sDS, uint32_t tmem) {
  using C = BwdCfg<HD>;
  constexpr uint32_t kIdescSq = make_idesc_bf16_f32(128, 128, false, false);  // S^T, dP^T
  constexpr uint32_t kIdescAcc = make_idesc_bf16_f32(128, HD, false, true);   // dV, dK
  constexpr uint32_t kIdescDq = make_idesc_bf16_f32(128, C::DQ_T ? 128 : HD, true, true);  // dQ (or dQ^T)
  const uint32_t k_addr = smem_u32(sK), v_addr = smem_u32(sV), q_addr = smem_u32(sQ), do_addr = smem_u32(sdO),
                 ds_addr = smem_u32(sDS);
  const uint64_t lim = p.wait_limit_ns;
  const int T = (p.N + 127) / 128;
  const int total = p.BHkv * p.chunks * T;

  // D[tmem] = A (128 x HD, K-major) * B (128 x HD, K-major)^T
  auto issue_sq = [&](uint32_t d_col, uint32_t a_addr, uint32_t b_addr) {
    const uint64_t ad = make_smem_desc_sw128(a_addr, 16, 1024), bd = make_smem_desc_sw128(b_addr, 16, 1024);
#pragma unroll
    for (int ks = 0; ks < HD / 16; ++ks) {
      const uint32_t off = (ks >> 2) * C::CHUNK_BYTES + (ks & 3) * 32;
      umma_ss(tmem + d_col, desc_add(ad, off), desc_add(bd, off), kIdescSq, ks > 0 ? 1u : 0u);
    }
  };
  auto fail = [&]() {
    record_timeout(p.status, &sh.abort_flag, WHERE_BWD_MMA);
    drain_mmas(&sh.mma_drain, lim);
  };

  int g = 0, items = 0;
  while (true) {
    const int item = take_item(sh, items, lim);
    if (item < 0) return fail();
    if (item >= total) break;
    const BwdWork<CAUSAL> wk(item, p.BHkv, p.N, p.group, p.chunks);
    const int n_iter = wk.n_iter();
    const int s0 = g % C::QST;
    if (!mbar_wait(&sh.kv_full, items & 1, &sh.abort_flag, lim) ||
        !mbar_wait(&sh.qdo_full[s0], (g / C::QST) & 1, &sh.abort_flag, lim))
      return fail();
    // Region A held the previous item's last P^T, region B its last dQ.
    if (g > 0 && !mbar_wait(&sh.pv_done, (g - 1) & 1, &sh.abort_flag, lim)) return fail();
    tc_fence_after_sync();
    issue_sq(C::REG_A, k_addr, q_addr + s0 * C::TILE_BYTES);  // S^T(first)
    umma_commit(&sh.s_full);
    if (DQ && g > 0 && !mbar_wait(&sh.dq_free, (g - 1) & 1, &sh.abort_flag, lim)) return fail();
    tc_fence_after_sync();
    issue_sq(C::REG_B, v_addr, do_addr + s0 * C::TILE_BYTES);  // dP^T(first)
    umma_commit(&sh.dp_full);

    for (int n = 0; n < n_iter; ++n, ++g) {
      const int s = g % C::QST;
      const bool has_next = n + 1 < n_iter;
      const int s1 = (g + 1) % C::QST;
      const uint32_t qa = q_addr + s * C::TILE_BYTES, doa = do_addr + s * C::TILE_BYTES;
      if (!mbar_wait(&sh.pa_ready, g & 1, &sh.abort_flag, lim)) return fail();
      if (n == 0 && items > 0 && !mbar_wait(&sh.acc_free, (items - 1) & 1, &sh.abort_flag, lim)) return fail();
      tc_fence_after_sync();
      // dV += P^T dO_n; P^T (bf16) sits in columns [0,32) and [64,96) of region A
      const uint64_t dod = make_smem_desc_sw128(doa, C::CHUNK_BYTES, 1024);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma_ts(tmem + C::DV_COL, tmem + C::REG_A + (ks >> 2) * 64 + (ks & 3) * 8, desc_add(dod, ks * 2048), kIdescAcc,
                (n > 0 || ks > 0) ? 1u : 0u);
      umma_commit(&sh.pv_done);
      if (has_next) {
        // S^T(n+1) overwrites P^T(n): wait until dV(n) has read it.
        if (!mbar_wait(&sh.qdo_full[s1], ((g + 1) / C::QST) & 1, &sh.abort_flag, lim)) return fail();
        if (!mbar_wait(&sh.pv_done, g & 1, &sh.abort_flag, lim)) return fail();
        tc_fence_after_sync();
        issue_sq(C::REG_A, k_addr, q_addr + s1 * C::TILE_BYTES);
        umma_commit(&sh.s_full);
      }
      if (!mbar_wait(&sh.ds_ready, g & 1, &sh.abort_flag, lim)) return fail();
      tc_fence_after_sync();
      // dK += dS^T Q_n
      const uint64_t dsk = make_smem_desc_sw128(ds_addr, 16, 1024), qmn = make_smem_desc_sw128(qa, C::CHUNK_BYTES, 1024);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma_ss(tmem + C::DK_COL, desc_add(dsk, (ks >> 2) * C::CHUNK_BYTES + (ks & 3) * 32), desc_add(qmn, ks * 2048),
                kIdescAcc, (n > 0 || ks > 0) ? 1u : 0u);
      if constexpr (DQ) {
        // dQ_n into region B. d = 128: dQ_n^T = K_j^T dS^T (head-dim columns on
        // the lanes, queries along the columns), so the drain's reductions
        // cover whole 128-byte lines. d = 64: dQ_n = dS K_j (queries on lanes).
        const uint64_t dsm = make_smem_desc_sw128(ds_addr, C::CHUNK_BYTES, 1024);
        const uint64_t kmn = make_smem_desc_sw128(k_addr, C::CHUNK_BYTES, 1024);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t ds_mn = desc_add(dsm, ks * 2048);
          const uint64_t k_mn = desc_add(kmn, ks * 2048);
          if constexpr (C::DQ_T)
            umma_ss(tmem + C::REG_B, k_mn, ds_mn, kIdescDq, ks > 0 ? 1u : 0u);
          else
            umma_ss(tmem + C::REG_B, ds_mn, k_mn, kIdescDq, ks > 0 ? 1u : 0u);
        }
        umma_commit(&sh.dq_full);
      }
      umma_commit(&sh.qdo_empty[s]);
      if (has_next) {
        if (DQ && !mbar_wait(&sh.dq_free, g & 1, &sh.abort_flag, lim)) return fail();
        tc_fence_after_sync();
        issue_sq(C::REG_B, v_addr, do_addr + s1 * C::TILE_BYTES);  // dP^T(n+1) over the drained dQ_n
        umma_commit(&sh.dp_full);
      }
    }
    umma_commit(&sh.acc_done);
    ++items;
  }
  // Normally the epilogues have waited for the last products; if a softmax
  // warpgroup gave up, nothing has.
  drain_mmas(&sh.mma_drain, lim);
}

// Warpgroup w (w = 0, 1) owns query columns [64w, 64w + 64) of every tile:
// thread r owns key r (TMEM lane r) in phases A and B, and head-dim column r
// (d = 128) or query r (d = 64) in the dQ drain. Per tile n the order is
// B(n), A(n+1), drain(n): phase A(n+1) overlaps the dK(n) and dQ_n MMAs and
// the drain's reductions overlap dP^T(n+1) and dV(n+1). After an item's last
// tile, warpgroup 0 writes dK_j and warpgroup 1 dV_j straight from TMEM to
// global memory while the MMA warp already starts the next item.
template <int HD, bool CAUSAL, bool DQ>
__device__ void bwd_softmax_role(const BwdLaunch& p, BwdShared& sh, uint8_t* sDS, float* sLD, uint8_t* sDQ,
                                 uint32_t tmem, int w) {
  using C = BwdCfg<HD>;
  const int r = threadIdx.x & 127;
  const uint32_t lane_base = static_cast<uint32_t>((threadIdx.x >> 5) & 3) << 21;
  const float c2 = p.scale_log2;
  const float sc = p.scale;
  const uint64_t lim = p.wait_limit_ns;
  const uint32_t ds_chunk = smem_u32(sDS) + w * C::CHUNK_BYTES;  // queries 64w .. 64w+63
  float* ld_l2 = sLD + w * 128;  // 64 base-2 logsumexps, then 64 scaled D values
  float* ld_d = ld_l2 + 64;
  const uint32_t bar_id = 1 + w;
  const uint32_t tA = tmem + lane_base + C::REG_A + 64 * w;
  const uint32_t tB = tmem + lane_base + C::REG_B + 64 * w;
  const int T = (p.N + 127) / 128;
  const int total = p.BHkv * p.chunks * T;
  bool alive = true;
  constexpr bool kPrefetchStats = !DQ && HD == 128;
  // P^T of the current tile as the bf16 pairs written to TMEM, kept from
  // phase A to phase B: dS uses the same rounded P as the dV MMA.
  uint32_t pk[32];

  // L2 / D of query tile i of head bh for this warpgroup's 64 columns:
  // thread r < 64 loads L2[r], thread r >= 64 loads D[r - 64] * scale.
  auto fetch_ld = [&](int bh, int i) -> float {
    const size_t row = static_cast<size_t>(bh) * p.Npad + i * 128 + 64 * w;
    return r < 64 ? __ldg(p.lse2 + row + r) : __ldg(p.D + row + (r - 64)) * sc;
  };
  auto wait_all = [&](uint64_t* bar, int parity, int where) {
    alive = alive && __all_sync(0xffffffffu, mbar_wait(bar, parity, &sh.abort_flag, lim));
    if (!alive) record_timeout(p.status, &sh.abort_flag, where);
    tc_fence_after_sync();
  };

  // ---- phase A of query tile i (global tile g): P^T = 2^(S^T * scale *
  // log2e - L2), written back to TMEM as bf16. After a timed-out wait a warp
  // stops working but still passes every named barrier, so the warpgroup's
  // barrier counts stay matched.
  auto phase_a = [&](const BwdWork<CAUSAL>& wk, int i, int g) {
    // The 64 base-2 logsumexps of this warpgroup's queries, read from smem
    // while S^T is still being computed (read in the loop they sit on the
    // phase's critical path: measured ~800 of ~1600 cycles at d = 128). Only
    // where the registers allow it (d = 128 without dQ); elsewhere they are
    // read in the loop.
    float4 lv[kPrefetchStats ? 16 : 1];
    if constexpr (kPrefetchStats) {
#pragma unroll
      for (int c = 0; c < 16; ++c) lv[c] = *reinterpret_cast<const float4*>(ld_l2 + 4 * c);
    }
    wait_all(&sh.s_full, g & 1, WHERE_BWD_SOFTMAX);
    if (!alive) return;
    float pv[64];
    {
      uint32_t a[32], b[32];
      tmem_ld32(tA, a);
      tmem_ld32(tA + 32, b);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        pv[c] = __uint_as_float(a[c]);
        pv[32 + c] = __uint_as_float(b[c]);
      }
    }
    // Only the key-tail tile and the causal diagonal tile need masking:
    // query (64w + c) sees key r only if 64w + c >= r.
    const bool key_valid = wk.j * 128 + r < p.N;
    const bool masked = !key_valid || (CAUSAL && i == wk.j);
    const int c_lo = !key_valid ? 64 : ((CAUSAL && i == wk.j) ? r - 64 * w : 0);
    // Three passes over the row (exponent arguments, exponentials, bf16
    // pairs) give the scheduler long runs of independent instructions.
#pragma unroll
    for (int c4 = 0; c4 < 64; c4 += 4) {
      const float4 l = kPrefetchStats ? lv[kPrefetchStats ? c4 / 4 : 0] : *reinterpret_cast<const float4*>(ld_l2 + c4);
      const float2 x01 = ffma2_bcast_mul(pv[c4], pv[c4 + 1], c2, -l.x, -l.y);
      const float2 x23 = ffma2_bcast_mul(pv[c4 + 2], pv[c4 + 3], c2, -l.z, -l.w);
      pv[c4] = x01.x;
      pv[c4 + 1] = x01.y;
      pv[c4 + 2] = x23.x;
      pv[c4 + 3] = x23.y;
    }
#pragma unroll
    for (int c = 0; c < 64; ++c) pv[c] = ex2_approx(pv[c]);
    if (masked) {
#pragma unroll
      for (int c = 0; c < 64; ++c)
        if (c < c_lo) pv[c] = 0.f;
    }
#pragma unroll
    for (int c = 0; c < 32; ++c) pk[c] = pack_bf16x2(pv[2 * c], pv[2 * c + 1]);
    tmem_st32(tA, pk);  // columns [64w, 64w + 32): already read
    tmem_st_wait();
    tc_fence_before_sync();
    mbar_arrive(&sh.pa_ready);
  };

  // ---- phase B: dS^T = P^T o (dP^T - D) * scale -> smem (bf16, swizzled)
  auto phase_b = [&](int g) {
    // the scaled D values, read from smem while dP^T is still being computed
    // (as the logsumexps in phase A)
    float4 dvv[kPrefetchStats ? 16 : 1];
    if constexpr (kPrefetchStats) {
#pragma unroll
      for (int c = 0; c < 16; ++c) dvv[c] = *reinterpret_cast<const float4*>(ld_d + 4 * c);
    }
    wait_all(&sh.dp_full, g & 1, WHERE_BWD_SOFTMAX);
    if (!alive) return;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t dpv[32];
      tmem_ld32(tB + 32 * h, dpv);
      tmem_ld_wait();
      uint32_t dk[16];
#pragma unroll
      for (int c4 = 0; c4 < 32; c4 += 4) {
        const float4 dd = kPrefetchStats ? dvv[kPrefetchStats ? (32 * h + c4) / 4 : 0]
                                         : *reinterpret_cast<const float4*>(ld_d + 32 * h + c4);
        const float dv4[4] = {dd.x, dd.y, dd.z, dd.w};
        const float2 p01 = unpack_bf16x2(pk[16 * h + c4 / 2]);
        const float2 p23 = unpack_bf16x2(pk[16 * h + c4 / 2 + 1]);
        const float2 g01 =
            ffma2_bcast_mul(__uint_as_float(dpv[c4]), __uint_as_float(dpv[c4 + 1]), sc, -dv4[0], -dv4[1]);
        const float2 g23 =
            ffma2_bcast_mul(__uint_as_float(dpv[c4 + 2]), __uint_as_float(dpv[c4 + 3]), sc, -dv4[2], -dv4[3]);
        const float2 ds01 = fmul2(p01, g01);
        const float2 ds23 = fmul2(p23, g23);
        dk[c4 / 2] = pack_bf16x2(ds01.x, ds01.y);
        dk[c4 / 2 + 1] = pack_bf16x2(ds23.x, ds23.y);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        st_shared_v4(ds_chunk + sw128_offset(r, 4 * h + u), dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    mbar_arrive(&sh.ds_ready);
  };

  // ---- dQ drain of query tile i (global tile g) out of region B
  auto drain = [&](int bh, int i, int g) {
    wait_all(&sh.dq_full, g & 1, WHERE_BWD_DQ);
    if constexpr (C::DQ_T) {
      // lane r = head-dim column r, this warpgroup's 64 queries along the
      // columns: for a fixed query the warp's 32 lanes add into 32
      // consecutive floats, one full 128-byte line per reduction. (Staging
      // the tile for TMA reduce-adds through the dS^T tile measured slower:
      // the staging reads land on the softmax warps' path.)
      if (!alive) return;
      float* dst = p.dq_acc + (static_cast<size_t>(bh) * p.Npad + i * 128 + 64 * w) * HD + r;
      uint32_t v[64];
      tmem_ld32(tB, *reinterpret_cast<uint32_t(*)[32]>(v));
      tmem_ld32(tB + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
      tmem_ld_wait();
      tc_fence_before_sync();
      mbar_arrive(&sh.dq_free);
#pragma unroll
      for (int c = 0; c < 64; ++c) red_add_f32(dst + static_cast<size_t>(c) * HD, __uint_as_float(v[c]));
    } else {
      // lane r = query r, head-dim columns [32w, 32w + 32): stage the row in
      // this warpgroup's swizzled smem chunk, then one thread reduce-adds the
      // 128 x 32 chunk into the accumulator through TMA.
      uint32_t v[32];
      if (alive) {
        tmem_ld32(tmem + lane_base + C::REG_B + 32 * w, v);
        tmem_ld_wait();
        tc_fence_before_sync();
        mbar_arrive(&sh.dq_free);
      }
      if (r == 0) tma_store_wait_read_all();  // the previous reduce has read the chunk
      named_barrier_sync(bar_id, 128);
      uint8_t* chunk = sDQ + w * 128 * 128;
      if (alive) {
#pragma unroll
        for (int u = 0; u < 8; ++u)
          st_shared_v4(smem_u32(chunk) + sw128_offset(r, u), v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
        fence_proxy_async_smem();
      }
      named_barrier_sync(bar_id, 128);
      if (alive && r == 0) {
        tma_reduce_add_3d(&p.tmdQacc, chunk, 32 * w, i * 128, bh);
        tma_store_commit();
      }
    }
  };

  // ---- item epilogue: w = 0 writes dK_j, w = 1 writes dV_j; thread r
  // writes key row r, rows past N are skipped. One chunk per group: fp32 TMEM
  // -> bf16 -> dk / dv. Several: the chunk's fp32 partial sum goes to the
  // workspace, and the post kernel adds the chunks in a fixed order.
  auto epilogue = [&](const BwdWork<CAUSAL>& wk, int items) {
    wait_all(&sh.acc_done, items & 1, WHERE_BWD_SOFTMAX);
    if (!alive) return;
    const int key = wk.j * 128 + r;
    const uint32_t t = tmem + lane_base + (w == 0 ? C::DK_COL : C::DV_COL);
    const size_t row = static_cast<size_t>(wk.bh) * p.N + key;
    if (p.chunks == 1) {
      __nv_bfloat16* dst = (w == 0 ? p.dk : p.dv) + row * HD;
#pragma unroll 1
      for (int c = 0; c < HD; c += 32) {
        uint32_t v[32];
        tmem_ld32(t + c, v);
        tmem_ld_wait();
        if (c + 32 == HD) {  // both accumulators read: the next item may overwrite them
          tc_fence_before_sync();
          mbar_arrive(&sh.acc_free);
        }
        if (key < p.N) {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            *reinterpret_cast<uint4*>(dst + c + 8 * u) =
                make_uint4(pack_bf16x2(__uint_as_float(v[8 * u + 0]), __uint_as_float(v[8 * u + 1])),
                           pack_bf16x2(__uint_as_float(v[8 * u + 2]), __uint_as_float(v[8 * u + 3])),
                           pack_bf16x2(__uint_as_float(v[8 * u + 4]), __uint_as_float(v[8 * u + 5])),
                           pack_bf16x2(__uint_as_float(v[8 * u + 6]), __uint_as_float(v[8 * u + 7])));
        }
      }
    } else {
      const size_t part_len = static_cast<size_t>(p.chunks) * p.BHkv * p.N * HD;
      float* part = p.kv_part + (w == 0 ? 0 : part_len) + (static_cast<size_t>(wk.c) * p.BHkv * p.N + row) * HD;
#pragma unroll 1
      for (int c = 0; c < HD; c += 32) {
        uint32_t v[32];
        tmem_ld32(t + c, v);
        tmem_ld_wait();
        if (c + 32 == HD) {
          tc_fence_before_sync();
          mbar_arrive(&sh.acc_free);
        }
        if (key < p.N) {
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<uint4*>(part + c + 4 * u) = make_uint4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
        }
      }
    }
  };


  // The next work item, agreed on by the whole warpgroup: a warp whose wait
  // timed out makes every warp of the group leave the loop at the same point.
  auto next_item = [&](int u) -> int {
    const int it = alive ? take_item(sh, u, lim) : -1;
    if (!named_barrier_and(bar_id, 128, it >= 0)) {
      if (alive) record_timeout(p.status, &sh.abort_flag, WHERE_BWD_SOFTMAX);
      alive = false;
      return total;
    }
    return it;
  };

  int g = 0, items = 0;
  int item = next_item(0);
  float ld = 0.f;
  if (item < total) {
    const BwdWork<CAUSAL> wk0(item, p.BHkv, p.N, p.group, p.chunks);
    ld = fetch_ld(wk0.q0, wk0.i0);
  }
  while (item < total) {
    const BwdWork<CAUSAL> wk(item, p.BHkv, p.N, p.group, p.chunks);
    const int n_iter = wk.n_iter();
    if (items > 0) named_barrier_sync(bar_id, 128);  // the previous item's L2 / D reads are done
    sLD[w * 128 + r] = ld;
    named_barrier_sync(bar_id, 128);
    typename BwdWork<CAUSAL>::Pos cur = wk.first();
    phase_a(wk, cur.i, g);
    for (int n = 0; n < n_iter; ++n) {
      const bool has_next = n + 1 < n_iter;
      typename BwdWork<CAUSAL>::Pos nxt = cur;
      wk.advance(nxt);
      const float next_ld = has_next ? fetch_ld(nxt.bh, nxt.i) : 0.f;  // lands during phase B
      phase_b(g + n);
      if (has_next) {
        named_barrier_sync(bar_id, 128);  // every thread is done reading this tile's L2 / D
        sLD[w * 128 + r] = next_ld;
        named_barrier_sync(bar_id, 128);
        phase_a(wk, nxt.i, g + n + 1);
      }
      if constexpr (DQ) drain(cur.bh, cur.i, g + n);
      cur = nxt;
    }
    const int item_next = next_item(items + 1);
    if (item_next < total) {
      const BwdWork<CAUSAL> wk1(item_next, p.BHkv, p.N, p.group, p.chunks);
      ld = fetch_ld(wk1.q0, wk1.i0);  // lands during the epilogue
    }
    epilogue(wk, items);
    g += n_iter;
    ++items;
    item = item_next;
  }
  if (DQ && !C::DQ_T && r == 0) tma_store_wait_all();  // reduce-adds complete before the CTA can exit
}

template <int HD, bool CAUSAL, bool DQ>
__global__ void __launch_bounds__(kThreads, 1) fa_bwd_kernel(const __grid_constant__ BwdLaunch p) {
  using C = BwdCfg<HD>;
  extern __shared__ uint8_t smem_dyn[];
  __shared__ BwdShared sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = sK + C::TILE_BYTES;
  uint8_t* sQ = sV + C::TILE_BYTES;
  uint8_t* sdO = sQ + C::QST * C::TILE_BYTES;
  uint8_t* sDS = sdO + C::QST * C::TILE_BYTES;
  float* sLD = reinterpret_cast<float*>(sDS + C::DS_BYTES);
  uint8_t* sDQ = sDS + C::DS_BYTES + C::LD_BYTES;  // 1024-aligned: DS and LD sizes are multiples of 1024
  const int warp = threadIdx.x >> 5;
  // Without dQ this pass writes nothing the dQ kernel reads, so a dQ kernel
  // queued behind it may take SMs as soon as this grid's CTAs leave them.
  if constexpr (!DQ) griddep_launch_dependents();
  const int wg = warp >> 2;

  if (threadIdx.x == 0) {
    mbar_init(&sh.kv_full, 1);
    for (int s = 0; s < 4; ++s) {
      mbar_init(&sh.qdo_full[s], 1);
      mbar_init(&sh.qdo_empty[s], 1);
    }
    // test hook: the S, P or dQ barrier waits for one arrival too many
    mbar_init(&sh.s_full, 1 + debug_extra(p.debug_skip, WHERE_BWD_MMA));
    mbar_init(&sh.dp_full, 1);
    mbar_init(&sh.pa_ready, 256 + debug_extra(p.debug_skip, WHERE_BWD_SOFTMAX));
    mbar_init(&sh.ds_ready, 256);
    mbar_init(&sh.pv_done, 1);
    mbar_init(&sh.dq_full, 1);
    mbar_init(&sh.dq_free, 256 + debug_extra(p.debug_skip, WHERE_BWD_DQ));
    mbar_init(&sh.acc_done, 1);
    mbar_init(&sh.acc_free, 256);
    mbar_init(&sh.mma_drain, 1);
    for (int s = 0; s < kItemSlots; ++s) {
      mbar_init(&sh.item_full[s], 1);
      mbar_init(&sh.item_empty[s], kItemConsumers);
    }
    sh.abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&sh.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sh.tmem_base;

  if (warp == kLoadWarp) {
    if (lane_id() == 0) bwd_load_role<HD, CAUSAL>(p, sh, sK, sV, sQ, sdO);
  } else if (warp == kMmaWarp) {
    if (lane_id() == 0) bwd_mma_role<HD, CAUSAL, DQ>(p, sh, sK, sV, sQ, sdO, sDS, tmem);
  } else {
    bwd_softmax_role<HD, CAUSAL, DQ>(p, sh, sDS, sLD, sDQ, tmem, wg);
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

template <int HD>
cudaError_t launch_pre_t(const BwdLaunch& a, cudaStream_t stream) {
  const long long rows = static_cast<long long>(a.BH) * a.Npad;
  constexpr int RPB = 8 * (32 / (HD / 8));  // rows per 256-thread block
  const long long blocks = (rows + RPB - 1) / RPB;
  bwd_pre_kernel<HD><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a.o, a.dO, a.lse, a.D, a.lse2,
                                                                        a.deterministic ? nullptr : a.dq_acc, a.sched,
                                                                        a.N, a.Npad, rows);
  return cudaGetLastError();
}

template <int HD, bool CAUSAL, bool DQ>
cudaError_t launch_main_t(const BwdLaunch& a, cudaStream_t stream) {
  using C = BwdCfg<HD>;
  auto kern = fa_bwd_kernel<HD, CAUSAL, DQ>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int T = (a.N + 127) / 128;
  const long long items = static_cast<long long>(a.BH) * T;
  // Persistent: one CTA per SM (the smem footprint allows no more).
  const long long grid = items < a.num_sms ? items : a.num_sms;
  kern<<<static_cast<unsigned>(grid), kThreads, C::SMEM_BYTES, stream>>>(a);
  return cudaGetLastError();
}

template <int HD>
cudaError_t launch_post_t(const BwdLaunch& a, cudaStream_t stream) {
  const long long vec = static_cast<long long>(a.BH) * a.N * (HD / 8);
  if (!a.deterministic)  // the dQ kernel has written dq itself
    bwd_post_kernel<HD><<<static_cast<unsigned>((vec + 255) / 256), 256, 0, stream>>>(a.dq_acc, a.dq, a.N, a.Npad,
                                                                                     vec);
  if (a.chunks > 1) {
    const long long n8 = static_cast<long long>(a.BHkv) * a.N * HD / 8;
    bwd_kv_sum_kernel<<<static_cast<unsigned>((2 * n8 + 255) / 256), 256, 0, stream>>>(a.kv_part, a.dk, a.dv,
                                                                                     a.chunks, n8);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_pre(const BwdLaunch& a, cudaStream_t stream) {
  switch (a.d) {
    case 64: return launch_pre_t<64>(a, stream);
    case 128: return launch_pre_t<128>(a, stream);
    case 256: return launch_pre_t<256>(a, stream);
    default: return cudaErrorNotSupported;
  }
}

cudaError_t launch_bwd_main(const BwdLaunch& a, cudaStream_t stream) {
  switch (a.d) {
    case 64:
      if (a.deterministic)
        return a.causal ? launch_main_t<64, true, false>(a, stream) : launch_main_t<64, false, false>(a, stream);
      return a.causal ? launch_main_t<64, true, true>(a, stream) : launch_main_t<64, false, true>(a, stream);
    case 128:
      if (a.deterministic)
        return a.causal ? launch_main_t<128, true, false>(a, stream) : launch_main_t<128, false, false>(a, stream);
      return a.causal ? launch_main_t<128, true, true>(a, stream) : launch_main_t<128, false, true>(a, stream);
    case 256: return launch_bwd_main_d256(a, stream);
    default: return cudaErrorNotSupported;
  }
}

cudaError_t launch_bwd_post(const BwdLaunch& a, cudaStream_t stream) {
  switch (a.d) {
    case 64: return launch_post_t<64>(a, stream);
    case 128: return launch_post_t<128>(a, stream);
    case 256: return launch_post_t<256>(a, stream);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace fa

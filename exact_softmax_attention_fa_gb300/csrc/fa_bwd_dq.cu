// dQ of the backward pass without atomics, for sm_103a.
//
// Method (web pages on FlashAttention-2): the reading note (papers.chlience.com)
// 5.3-5.4 and the paper-graph-ui summary, "The Backward Pass", accumulate
// dQ_i += dS_ij K_j across key blocks with atomic adds, so dQ is not bitwise
// reproducible. This kernel is the deterministic alternative: one work item
// owns query tile i of one head and loops over the key tiles itself, so dQ_i
// is summed on chip in a fixed order:
//   S = Q_i K_j^T, P = 2^(S scale log2e - L_i log2e), dP = dO_i V_j^T,
//   dS = P o (dP - D_i) * scale, dQ_i += dS K_j,
// with L and D from the preprocess kernel. The backward main kernel then runs
// without its dQ products and reductions, and computes only dK and dV.
//
// GB300 mapping: persistent, one CTA (320 threads) per SM taking items from a
// counter in the workspace (causal: the query tiles that see the most keys
// first). Warp 8 streams Q_i, dO_i once per item and K_j, V_j through two
// rings (K deeper: K_j is read by S(j) and, late, by the dQ product);
// warp 9 issues the MMAs (S and dP into TMEM, dQ accumulated in TMEM);
// warpgroups 0 and 1 own key columns [64w, 64w + 64) of every tile, thread r
// = query row r = TMEM lane r, so the row statistics L_r and D_r are
// per-thread scalars. P (bf16, the rounding the dV product of the main kernel
// uses) stays in registers; dS (bf16) is written back into the columns of
// its own tile's S buffer, already read, and is the TMEM A operand of
// dQ += dS K_j, with K_j as the MN-major B operand.
//
// TMEM columns (512 allocated): S buffers [0, 128) and [128, 256), dP
// [256, 384), dQ [384, 384 + d).
#include <cuda_bf16.h>

#include <algorithm>

#include "fa_internal.h"
#include "fa_kernel_common.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kThreads = 320;
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kItemConsumers = 1 + 256;  // the MMA thread and the softmax threads

template <int HD>
struct DqCfg {
  static constexpr int CHUNKS = HD / 64;
  static constexpr int TILE_BYTES = 128 * HD * 2;
  static constexpr int CHUNK_BYTES = 128 * 128;
  // K_j is read by S(j) early and by the dQ product late; V_j only by dP(j).
  // A deeper K ring lets S(j+1) start while K_j is still in use. d = 128:
  // 4 K stages and 1 V stage (the smem of 3 + 2 measured 1 % slower).
  static constexpr int KST = 4;                 // K_j ring stages
  static constexpr int VST = HD == 64 ? 2 : 1;  // V_j ring stages
  // S is double-buffered (tile t in buffer t & 1), so S(t+1) is computed
  // while the softmax still works on tile t.
  static constexpr uint32_t S_COL = 0, DP_COL = 256, DQ_COL = 384;
  __host__ __device__ static constexpr uint32_t s_col(int b) { return S_COL + 128u * uint32_t(b); }
  // smem: Q_i, dO_i, KST x K_j, VST x V_j (dS lives in TMEM)
  static constexpr int SMEM_BYTES = (2 + KST + VST) * TILE_BYTES + 1024;
};

struct DqShared {
  uint64_t q_full, q_free;
  uint64_t k_full[4], k_empty[4], v_full[2], v_empty[2];
  uint64_t s_full[2];  // per S buffer
  // ds_ready[t & 1]: dS(t) is in TMEM. Two barriers, because the softmax can
  // finish tile t+1 (it needs only dP(t+1), issued before the MMA thread
  // waits for dS(t)) before that wait starts: on one barrier the wait would
  // then see two completed phases and take the pending third for its own.
  // Tile t+2 needs dP(t+2), issued after the wait, so one barrier per tile
  // parity can be at most one phase ahead of its waiter.
  uint64_t dp_full, dp_free, ds_ready[2], dq_done, acc_done, acc_free;
  uint64_t mma_drain;  // the MMA thread's last commit: all its MMAs done before the CTA exits
  uint64_t item_full[kItemSlots], item_empty[kItemSlots];
  int item_ring[kItemSlots];
  uint32_t tmem_base;
  int abort_flag;
};

// Work item: query tile i of query head bh; key tiles 0 .. nkv-1 (causal:
// the tiles up to the diagonal). Causal items are numbered most-work-first;
// non-causal items of one head are adjacent (K/V reuse in L2).
template <bool CAUSAL>
struct DqWork {
  int bh, i, nkv;
  __device__ DqWork(int item, int BH, int N) {
    const int T = (N + 127) / 128;
    if (CAUSAL) {
      i = T - 1 - item / BH;
      bh = item % BH;
      nkv = i + 1;
    } else {
      bh = item / T;
      i = item % T;
      nkv = T;
    }
  }
};

// TMA producer (one thread): Q_i and dO_i once per item, after the previous
// item's last S and dP products have read them; K_j, V_j through the ring.
template <int HD, bool CAUSAL>
__device__ void dq_load_role(const BwdLaunch& p, DqShared& sh, uint8_t* sQ, uint8_t* sdO, uint8_t* sK,
                             uint8_t* sV) {
  using C = DqCfg<HD>;
  tma_prefetch_desc(&p.tmQ);
  tma_prefetch_desc(&p.tmdO);
  tma_prefetch_desc(&p.tmK);
  tma_prefetch_desc(&p.tmV);
  const int T = (p.N + 127) / 128;
  const int total = p.BH * T;
  const uint64_t lim = p.wait_limit_ns;
  int u = 0, kv = 0, q_issued = 0;  // kv: K/V tiles loaded
  bool k_extra = false;              // K of tile kv issued, its V not (abort in between)
  bool aborted = false;
  auto load_kv = [&](int j, int kvh) -> bool {
    const int ks = kv % C::KST, vs = kv % C::VST;
    if (kv >= C::KST && !mbar_wait(&sh.k_empty[ks], ((kv / C::KST) - 1) & 1, &sh.abort_flag, lim)) return false;
    mbar_arrive_expect_tx(&sh.k_full[ks], C::TILE_BYTES);
#pragma unroll
    for (int c = 0; c < C::CHUNKS; ++c)
      tma_load_3d(sK + ks * C::TILE_BYTES + c * C::CHUNK_BYTES, &p.tmK, &sh.k_full[ks], c * 64, j * 128, kvh);
    k_extra = true;
    if (kv >= C::VST && !mbar_wait(&sh.v_empty[vs], ((kv / C::VST) - 1) & 1, &sh.abort_flag, lim)) return false;
    mbar_arrive_expect_tx(&sh.v_full[vs], C::TILE_BYTES);
#pragma unroll
    for (int c = 0; c < C::CHUNKS; ++c)
      tma_load_3d(sV + vs * C::TILE_BYTES + c * C::CHUNK_BYTES, &p.tmV, &sh.v_full[vs], c * 64, j * 128, kvh);
    ++kv;
    k_extra = false;
    return true;
  };
  int item = blockIdx.x;  // the grid never exceeds the item count
  while (!aborted) {
    if (!publish_item(sh, u, item, lim)) {
      aborted = true;
      break;
    }
    if (item >= total) break;
    const DqWork<CAUSAL> wk(item, p.BH, p.N);
    const int kvh = wk.bh / p.group;  // grouped K/V heads
    // The first K/V tile loads while the previous item still reads Q_i, dO_i.
    if (!load_kv(0, kvh) || (u > 0 && !mbar_wait(&sh.q_free, (u - 1) & 1, &sh.abort_flag, lim))) {
      aborted = true;
      break;
    }
    if (!debug_skip_here(p.debug_skip, WHERE_BWD_LOAD, u == 0)) {  // test hook
      mbar_arrive_expect_tx(&sh.q_full, 2 * C::TILE_BYTES);
#pragma unroll
      for (int c = 0; c < C::CHUNKS; ++c) {
        tma_load_3d(sQ + c * C::CHUNK_BYTES, &p.tmQ, &sh.q_full, c * 64, wk.i * 128, wk.bh);
        tma_load_3d(sdO + c * C::CHUNK_BYTES, &p.tmdO, &sh.q_full, c * 64, wk.i * 128, wk.bh);
      }
      ++q_issued;
    }
    for (int j = 1; j < wk.nkv && !aborted; ++j) aborted = !load_kv(j, kvh);
    ++u;
    if (!aborted) item = claim_item(p.sched + 2);
  }
  finish_claiming(p.sched + 2);
  if (aborted) record_timeout(p.status, &sh.abort_flag, WHERE_BWD_LOAD);
  // The copies already issued land before the CTA can exit (after an abort
  // no consumer may wait for them). An aborted load_kv may have issued K_j
  // without V_j: kv counts only tiles whose K and V were both issued. Each
  // slot waits for the latest phase issued into it only (an older phase of a
  // slot can no longer be told apart once a newer one has completed).
  const int k_last = k_extra ? kv : kv - 1;
  for (int n = std::max(0, k_last - C::KST + 1); n <= k_last; ++n)
    drain_wait(&sh.k_full[n % C::KST], (n / C::KST) & 1, lim);
  for (int n = std::max(0, kv - C::VST); n < kv; ++n) drain_wait(&sh.v_full[n % C::VST], (n / C::VST) & 1, lim);
  if (q_issued > 0) drain_wait(&sh.q_full, (q_issued - 1) & 1, lim);
}

// One thread issues every MMA. Per key tile j (global tile t):
//   S(t+1)   into the other S buffer once K_{j+1} is in and the dQ product
//            of tile t-1 (whose dS sat there) is done (overlaps A(t), B(t))
//   dP(t+1)  once phase B(t) has read dP(t)        (overlaps the rest of B(t))
//   dQ += dS(t) K_j   once phase B(t) wrote dS(t)  (overlaps phase A(t+1))
template <int HD, bool CAUSAL>
__device__ void dq_mma_role(const BwdLaunch& p, DqShared& sh, uint8_t* sQ, uint8_t* sdO, uint8_t* sK, uint8_t* sV,
                            uint32_t tmem) {
  using C = DqCfg<HD>;
  constexpr uint32_t kIdescSq = make_idesc_bf16_f32(128, 128, false, false);  // S, dP: A, B K-major
  constexpr uint32_t kIdescDq = make_idesc_bf16_f32(128, HD, false, true);    // A = dS (TMEM), B = K_j MN-major
  const uint32_t q_addr = smem_u32(sQ), do_addr = smem_u32(sdO), k_addr = smem_u32(sK), v_addr = smem_u32(sV);
  const uint64_t lim = p.wait_limit_ns;
  const int T = (p.N + 127) / 128;
  const int total = p.BH * T;

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

  // S(t) into buffer t & 1, which tile t - 2 used.
  // done_tile: the latest dQ product issued (tile t - 2 inside an item, t - 1
  // at an item's start); its completion implies that of every earlier one,
  // including the product of tile t - 2 whose dS sat in buffer t & 1.
  auto issue_s = [&](int t, int kvi, int done_tile) -> bool {  // kvi: the tile's index in the K/V stream
    const int stage = kvi % C::KST;
    if (!mbar_wait(&sh.k_full[stage], (kvi / C::KST) & 1, &sh.abort_flag, lim)) return false;
    if (t >= 2 && !mbar_wait(&sh.dq_done, done_tile & 1, &sh.abort_flag, lim)) return false;
    tc_fence_after_sync();
    issue_sq(C::s_col(t & 1), q_addr, k_addr + stage * C::TILE_BYTES);
    umma_commit(&sh.s_full[t & 1]);
    return true;
  };
  // dP(t) over dP(t - 1): wait until phase B(t - 1) loaded it.
  auto issue_dp = [&](int t, int kvi) -> bool {
    const int stage = kvi % C::VST;
    if (!mbar_wait(&sh.v_full[stage], (kvi / C::VST) & 1, &sh.abort_flag, lim)) return false;
    if (t >= 1 && !mbar_wait(&sh.dp_free, (t - 1) & 1, &sh.abort_flag, lim)) return false;
    tc_fence_after_sync();
    issue_sq(C::DP_COL, do_addr, v_addr + stage * C::TILE_BYTES);
    umma_commit(&sh.dp_full);
    umma_commit(&sh.v_empty[stage]);  // V_j is read by dP(j) only
    return true;
  };

  int u = 0, kv = 0, t = 0;
  while (true) {
    const int item = take_item(sh, u, lim);
    if (item < 0) return fail();
    if (item >= total) break;
    const DqWork<CAUSAL> wk(item, p.BH, p.N);
    if (!mbar_wait(&sh.q_full, u & 1, &sh.abort_flag, lim) || !issue_s(t, kv, t - 1) || !issue_dp(t, kv))
      return fail();
    if (wk.nkv == 1) umma_commit(&sh.q_free);
    // Per tile t: S(t+1) as soon as its K tile is in, dP(t+1) once phase B(t)
    // has read dP(t), dQ += dS(t) K once phase B(t) has written dS(t).
    for (int j = 0; j < wk.nkv; ++j, ++kv, ++t) {
      const int s = kv % C::KST;
      if (j + 1 < wk.nkv) {
        if (!issue_s(t + 1, kv + 1, t - 1) || !issue_dp(t + 1, kv + 1)) return fail();
        if (j + 2 == wk.nkv) umma_commit(&sh.q_free);  // the item's last S and dP are issued
      }
      if (!mbar_wait(&sh.ds_ready[t & 1], (t >> 1) & 1, &sh.abort_flag, lim)) return fail();
      // the first dQ product of an item overwrites the accumulator: the
      // previous item's epilogue must have read it
      if (j == 0 && u > 0 && !mbar_wait(&sh.acc_free, (u - 1) & 1, &sh.abort_flag, lim)) return fail();
      tc_fence_after_sync();
      // dS (bf16 pairs) sits in columns [0, 32) and [64, 96) of S buffer t & 1:
      // keys 16 ks .. 16 ks + 15 are 8 columns at 64 (ks / 4) + 8 (ks % 4)
      const uint64_t kd = make_smem_desc_sw128(k_addr + s * C::TILE_BYTES, C::CHUNK_BYTES, 1024);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma_ts(tmem + C::DQ_COL, tmem + C::s_col(t & 1) + (ks >> 2) * 64 + (ks & 3) * 8, desc_add(kd, ks * 2048),
                kIdescDq, (j > 0 || ks > 0) ? 1u : 0u);
      umma_commit(&sh.dq_done);
      umma_commit(&sh.k_empty[s]);
    }
    umma_commit(&sh.acc_done);
    ++u;
  }
  // Normally the epilogues have waited for the last products; if a softmax
  // warpgroup gave up, nothing has.
  drain_mmas(&sh.mma_drain, lim);
}

// Warpgroup w owns key columns [64w, 64w + 64) of every tile; thread r owns
// query row r. Phase A: P = 2^(S scale log2e - L2_r) (bf16-rounded, kept in
// registers). Phase B: dS = P o (dP scale - D_r scale) into the dS tile. At
// the end of an item warpgroup w writes dQ columns [w d/2, (w+1) d/2).
template <int HD, bool CAUSAL>
__device__ void dq_softmax_role(const BwdLaunch& p, DqShared& sh, uint32_t tmem, int w) {
  using C = DqCfg<HD>;
  const int r = threadIdx.x & 127;
  const uint32_t lane_base = static_cast<uint32_t>((threadIdx.x >> 5) & 3) << 21;
  const float c2 = p.scale_log2;
  const float sc = p.scale;
  const uint64_t lim = p.wait_limit_ns;
  const uint32_t tS0 = tmem + lane_base + C::S_COL + 64 * w;  // + 128 for buffer 1
  const uint32_t tDP = tmem + lane_base + C::DP_COL + 64 * w;
  const uint32_t bar_id = 1 + w;
  const int T = (p.N + 127) / 128;
  const int total = p.BH * T;
  bool alive = true;
  uint32_t pk[32];  // P of the current tile, bf16 pairs

  auto wait_all = [&](uint64_t* bar, int parity, int where) {
    alive = alive && __all_sync(0xffffffffu, mbar_wait(bar, parity, &sh.abort_flag, lim));
    if (!alive) record_timeout(p.status, &sh.abort_flag, where);
    tc_fence_after_sync();
  };
  // The next work item, agreed on by the whole warpgroup (see the main kernel).
  auto next_item = [&](int u) -> int {
    const int it = alive ? take_item(sh, u, lim) : -1;
    if (!named_barrier_and(bar_id, 128, it >= 0)) {
      if (alive) record_timeout(p.status, &sh.abort_flag, WHERE_BWD_SOFTMAX);
      alive = false;
      return total;
    }
    return it;
  };

  int u = 0, t = 0;
  int item = next_item(0);
  while (item < total) {
    const DqWork<CAUSAL> wk(item, p.BH, p.N);
    const int row = wk.i * 128 + r;
    const size_t srow = static_cast<size_t>(wk.bh) * p.Npad + row;
    const float l2 = __ldg(p.lse2 + srow);  // +inf on padding rows: their P is 0
    const float dsc = __ldg(p.D + srow) * sc;
    for (int j = 0; j < wk.nkv; ++j, ++t) {
      // ---- phase A
      wait_all(&sh.s_full[t & 1], (t >> 1) & 1, WHERE_BWD_SOFTMAX);
      if (alive) {
        float pv[64];
        {
          const uint32_t tS = tS0 + 128u * uint32_t(t & 1);
          uint32_t a[32], b[32];
          tmem_ld32(tS, a);
          tmem_ld32(tS + 32, b);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            pv[c] = __uint_as_float(a[c]);
            pv[32 + c] = __uint_as_float(b[c]);
          }
        }

        // key 128j + 64w + c is seen if it is < N and (causal) <= the query row
        const int kbase = j * 128 + 64 * w;
        int c_hi = std::min(64, p.N - kbase);
        if (CAUSAL && j == wk.i) c_hi = std::min(c_hi, r - 64 * w + 1);
        const bool masked = c_hi < 64;
#pragma unroll
        for (int c4 = 0; c4 < 64; c4 += 4) {
          const float2 x01 = ffma2_bcast(pv[c4], pv[c4 + 1], c2, -l2);
          const float2 x23 = ffma2_bcast(pv[c4 + 2], pv[c4 + 3], c2, -l2);
          pv[c4] = ex2_approx(x01.x);
          pv[c4 + 1] = ex2_approx(x01.y);
          pv[c4 + 2] = ex2_approx(x23.x);
          pv[c4 + 3] = ex2_approx(x23.y);
          if (masked) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              if (c4 + q >= c_hi) pv[c4 + q] = 0.f;
          }
          pk[c4 / 2] = pack_bf16x2(pv[c4], pv[c4 + 1]);
          pk[c4 / 2 + 1] = pack_bf16x2(pv[c4 + 2], pv[c4 + 3]);
        }
      }
      // ---- phase B: dS into the first 32 columns of this warpgroup's half of
      // S buffer t & 1 (phase A has read them)
      wait_all(&sh.dp_full, t & 1, WHERE_BWD_SOFTMAX);
      if (alive) {
        uint32_t ds[32];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t dpv[32];
          tmem_ld32(tDP + 32 * h, dpv);
          tmem_ld_wait();
          if (h == 1) {
            tc_fence_before_sync();
            mbar_arrive(&sh.dp_free);
          }
#pragma unroll
          for (int c4 = 0; c4 < 32; c4 += 4) {
            const float2 p01 = unpack_bf16x2(pk[16 * h + c4 / 2]);
            const float2 p23 = unpack_bf16x2(pk[16 * h + c4 / 2 + 1]);
            const float2 g01 = ffma2_bcast(__uint_as_float(dpv[c4]), __uint_as_float(dpv[c4 + 1]), sc, -dsc);
            const float2 g23 = ffma2_bcast(__uint_as_float(dpv[c4 + 2]), __uint_as_float(dpv[c4 + 3]), sc, -dsc);
            const float2 d01 = fmul2(p01, g01);
            const float2 d23 = fmul2(p23, g23);
            ds[16 * h + c4 / 2] = pack_bf16x2(d01.x, d01.y);
            ds[16 * h + c4 / 2 + 1] = pack_bf16x2(d23.x, d23.y);
          }
        }
        tmem_st32(tS0 + 128u * uint32_t(t & 1), ds);
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(&sh.ds_ready[t & 1]);
      }
    }
    const int item_next = next_item(u + 1);
    // ---- epilogue: dQ (fp32, TMEM) -> bf16 -> dq; rows past N are skipped
    wait_all(&sh.acc_done, u & 1, WHERE_BWD_SOFTMAX);
    if (alive) {
      const uint32_t tq = tmem + lane_base + C::DQ_COL + w * (HD / 2);
      __nv_bfloat16* dst = p.dq + (static_cast<size_t>(wk.bh) * p.N + row) * HD + w * (HD / 2);
#pragma unroll
      for (int c = 0; c < HD / 2; c += 32) {
        uint32_t v[32];
        tmem_ld32(tq + c, v);
        tmem_ld_wait();
        if (c + 32 == HD / 2) {  // the next item may overwrite the accumulator
          tc_fence_before_sync();
          mbar_arrive(&sh.acc_free);
        }
        if (row < p.N) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4*>(dst + c + 8 * q) =
                make_uint4(pack_bf16x2(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1])),
                           pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                           pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                           pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
        }
      }
    }
    ++u;
    item = item_next;
  }
}

template <int HD, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1) fa_bwd_dq_kernel(const __grid_constant__ BwdLaunch p) {
  using C = DqCfg<HD>;
  extern __shared__ uint8_t smem_dyn[];
  __shared__ DqShared sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sdO = sQ + C::TILE_BYTES;
  uint8_t* sK = sdO + C::TILE_BYTES;
  uint8_t* sV = sK + C::KST * C::TILE_BYTES;
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    mbar_init(&sh.q_full, 1);
    mbar_init(&sh.q_free, 1);
    for (int s = 0; s < 4; ++s) {
      mbar_init(&sh.k_full[s], 1);
      mbar_init(&sh.k_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sh.v_full[s], 1);
      mbar_init(&sh.v_empty[s], 1);
    }
    // test hook: buffer 0's S or dS barrier waits for one arrival too many
    for (int b = 0; b < 2; ++b) mbar_init(&sh.s_full[b], 1 + (b == 0 ? debug_extra(p.debug_skip, WHERE_BWD_MMA) : 0u));
    mbar_init(&sh.dp_full, 1);
    mbar_init(&sh.dp_free, 256);
    for (int b = 0; b < 2; ++b)
      mbar_init(&sh.ds_ready[b], 256 + (b == 0 ? debug_extra(p.debug_skip, WHERE_BWD_SOFTMAX) : 0u));
    mbar_init(&sh.dq_done, 1);
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
    if (lane_id() == 0) dq_load_role<HD, CAUSAL>(p, sh, sQ, sdO, sK, sV);
  } else if (warp == kMmaWarp) {
    if (lane_id() == 0) dq_mma_role<HD, CAUSAL>(p, sh, sQ, sdO, sK, sV, tmem);
  } else {
    dq_softmax_role<HD, CAUSAL>(p, sh, tmem, warp >> 2);
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
  // Launched to overlap the dK/dV pass (overlap_prev), this grid must not
  // complete before that pass has: work queued after it may read dK and dV.
  if (threadIdx.x == 0) griddep_wait();
}

template <int HD, bool CAUSAL>
cudaError_t launch_t(const BwdLaunch& a, cudaStream_t stream) {
  using C = DqCfg<HD>;
  auto kern = fa_bwd_dq_kernel<HD, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const long long items = static_cast<long long>(a.BH) * ((a.N + 127) / 128);
  const long long grid = items < a.num_sms ? items : a.num_sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.overlap_prev ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

cudaError_t launch_bwd_dq(const BwdLaunch& a, cudaStream_t stream) {
  switch (a.d) {
    case 64: return a.causal ? launch_t<64, true>(a, stream) : launch_t<64, false>(a, stream);
    case 128: return a.causal ? launch_t<128, true>(a, stream) : launch_t<128, false>(a, stream);
    case 256: return launch_bwd_dq256(a, stream);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace fa

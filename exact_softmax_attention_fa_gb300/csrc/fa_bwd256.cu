// Backward main kernel for head dimension 256 on sm_103a.
//
// Same method as fa_bwd.cu (reading note 5.3; paper-graph-ui summary, "The
// Backward Pass": key blocks outer, recompute S and P = exp(S - L), dV += P^T
// dO, dP = dO V^T, dS = P o (dP - D), dK += dS^T Q, dQ += dS K), with a split
// of its own because at d = 256 the fp32 dK and dV of one 128-key tile alone
// would fill all 512 TMEM columns, and the bf16 K, V, Q and dO tiles of 128
// rows alone would need 256 KB of shared memory:
//   - A work item is (K/V head, 128-key tile j, half h of the head
//     dimension); it accumulates columns [128h, 128h + 128) of dK_j and dV_j
//     and, in the atomic instantiation, adds columns [128h, 128h + 128) of
//     every dQ_i. The two items of a key tile both compute S^T and dP^T over
//     the full head dimension.
//   - Persistent: one CTA per SM claims items from a counter in the
//     workspace (causal: the key tiles that see the most query tiles first).
//   - K_j and V_j (64 KB each) stay in shared memory for the item. Query
//     tiles have 64 rows and stream through four rings of half tiles
//     (64 rows x 128 columns, 16 KB): Q_i and dO_i each split into the item's
//     half h and the other half. The other halves are read only by S^T(i)
//     and dP^T(i) and are released right after them; the h halves are also
//     the B operands of dK += dS^T Q_i[:, h] and dV += P^T dO_i[:, h]. Q's h
//     ring has two slots: S^T(i+1) is issued before dK(i) has released
//     Q_i's half.
//   - Everything is computed transposed, keys on the TMEM lanes: S^T = K_j
//     Q_i^T and dP^T = V_j dO_i^T (SS MMAs, 128 keys x 64 queries); two
//     softmax warpgroups, each owning 32 of the tile's queries, form
//     P^T = 2^(S^T scale log2e - L log2e) (bf16, back into TMEM, the A
//     operand of dV) and dS^T = P^T o (dP^T - D) scale (bf16, into a
//     swizzled smem tile, the A operand of dK and the B operand of
//     dQ_i^T = K_j[:, h]^T dS^T, head-dim columns on the lanes, so each warp's
//     fp32 reductions into the dQ accumulator cover whole 128-byte lines).
//   - MMA order per query tile n: dV(n) after phase A(n); S^T(n+1) once dV(n)
//     has read P^T(n); dK(n), dQ(n) after phase B(n); dP^T(n+1). The softmax
//     warpgroups run B(n), A(n+1), drain(n): phase A(n+1) overlaps dK(n) and
//     dQ(n), and the drain's reductions overlap dP^T(n+1) and dV(n+1).
//   - dK_j and dV_j are written once per item straight from TMEM while the
//     MMA thread starts the next item.
//   - The DQ = false instantiation skips the dQ product and drain: the
//     deterministic backward forms dQ in fa_bwd_dq256.cu.
// TMEM columns (512 allocated): dK half [0, 128), dV half [128, 256),
// S^T then P^T [256, 320), dP^T [320, 384), dQ^T half in two buffers
// [384, 448) and [448, 512) (tile n in buffer n & 1).
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "fa_internal.h"
#include "fa_kernel_common.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kThreads = 320;
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kItemConsumers = 1 + 256;  // the MMA thread and the softmax threads

struct Cfg256 {
  static constexpr int HD = 256;
  static constexpr int BQ = 64;                    // query rows per tile
  static constexpr int KV_CHUNK = 128 * 128;       // [128 keys][64 d] bf16
  static constexpr int KV_BYTES = 4 * KV_CHUNK;    // 64 KB
  static constexpr int Q_CHUNK = BQ * 128;         // [64 rows][64 d] bf16, 8 KB
  static constexpr int HALF_BYTES = 2 * Q_CHUNK;   // [64 rows][128 d], 16 KB
  static constexpr int QH_SLOTS = 2;               // Q_i[:, h] ring
  static constexpr int DS_BYTES = 128 * BQ * 2;    // [128 keys][64 queries] bf16
  static constexpr int LD_BYTES = 2 * 64 * 4;      // per warpgroup: 32 base-2 L + 32 scaled D
  static constexpr uint32_t DK_COL = 0, DV_COL = 128, REG_S = 256, REG_DP = 320, REG_DQ = 384;
  __host__ __device__ static constexpr uint32_t dq_col(int b) { return REG_DQ + 64u * uint32_t(b); }
  // smem: K_j, V_j, the half-tile slots (Q h x2, Q other, dO h, dO other), dS^T, L/D staging
  static constexpr int SMEM_BYTES = 2 * KV_BYTES + (QH_SLOTS + 3) * HALF_BYTES + DS_BYTES + LD_BYTES + 1024;
};

struct Shared256 {
  uint64_t kv_full;
  uint64_t qh_full[2], qh_empty[2];  // Q_i[:, h], slot n % 2
  uint64_t qo_full, qo_empty;        // Q_i, the other half
  uint64_t doh_full, doh_empty;      // dO_i[:, h]
  uint64_t doo_full, doo_empty;      // dO_i, the other half
  uint64_t s_full, dp_full, pa_ready, ds_ready, pv_done, acc_done, acc_free;
  uint64_t dq_full[2], dq_free[2];   // dQ^T buffer n & 1
  uint64_t mma_drain;                // the MMA thread's last commit: all its MMAs done before the CTA exits
  uint64_t item_full[kItemSlots], item_empty[kItemSlots];
  int item_ring[kItemSlots];
  uint32_t tmem_base;
  int abort_flag;
};

// Work item: key tile j of K/V head bh, half h of the head dimension. Its
// query stream is, for each of the g query heads that share the K/V head
// (query head bh*g + t), the 64-row query tiles i0 .. T64-1 (causal:
// i0 = 2j). Causal items are numbered most-work-first; the two halves of a
// key tile are adjacent (they read the same query stream).
template <bool CAUSAL>
struct Work256 {
  int bh, j, h, i0, T64, g;
  __device__ Work256(int item, int BHkv, int N, int group) {
    const int T = (N + 127) / 128;
    T64 = (N + 63) / 64;
    if (CAUSAL) {
      j = item / (2 * BHkv);
      const int rem = item - j * 2 * BHkv;
      bh = rem >> 1;
      h = rem & 1;
    } else {
      bh = item / (2 * T);
      const int rem = item - bh * 2 * T;
      j = rem >> 1;
      h = rem & 1;
    }
    i0 = CAUSAL ? 2 * j : 0;
    g = group;
  }
  __device__ int n_iter() const { return g * (T64 - i0); }
  struct Pos {
    int bh, i;  // query head, 64-row query tile
  };
  __device__ Pos first() const { return Pos{bh * g, i0}; }
  __device__ void advance(Pos& p) const {
    if (++p.i == T64) {
      p.i = i0;
      ++p.bh;
    }
  }
};

__device__ __forceinline__ int total_items256(const BwdLaunch& p) { return p.BHkv * ((p.N + 127) / 128) * 2; }

// Smem address of chunk c (0..3, 64 columns of the head dimension) of a
// query tile's Q (or dO) for an item of half h: in the h half's slot or in
// the other half's slot.
__device__ __forceinline__ uint32_t half_chunk(uint32_t h_slot, uint32_t o_slot, int h, int c) {
  return ((c >> 1) == h ? h_slot : o_slot) + (c & 1) * Cfg256::Q_CHUNK;
}

// TMA producer (one thread). Per query tile: Q's h half, Q's other half,
// dO's other half, dO's h half (the order in which their slots free up);
// per item K_j and V_j once every MMA of the previous item has completed.
template <bool CAUSAL>
__device__ void load_role(const BwdLaunch& p, Shared256& sh, uint8_t* sK, uint8_t* sV, uint8_t* sQh, uint8_t* sQo,
                          uint8_t* sDOh, uint8_t* sDOo) {
  using C = Cfg256;
  tma_prefetch_desc(&p.tmQ);
  tma_prefetch_desc(&p.tmK);
  tma_prefetch_desc(&p.tmV);
  tma_prefetch_desc(&p.tmdO);
  const int total = total_items256(p);
  const uint64_t lim = p.wait_limit_ns;
  int g = 0, items = 0, kv_issued = 0;
  int issued = 0;  // query tiles whose four half tiles were all issued
  int parts = 0;   // half tiles of tile `issued` issued before an abort (0..3)
  bool aborted = false;
  // the two 64-column chunks of half `half` of a 64-row tile of `map`
  auto load_half = [&](uint64_t* bar, uint8_t* dst, const CUtensorMap* map, int half, int i, int bh) {
    mbar_arrive_expect_tx(bar, C::HALF_BYTES);
    tma_load_3d(dst, map, bar, 128 * half, i * C::BQ, bh);
    tma_load_3d(dst + C::Q_CHUNK, map, bar, 128 * half + 64, i * C::BQ, bh);
  };
  auto load_tile = [&](int n, const typename Work256<CAUSAL>::Pos& pos, int h) -> bool {
    const int s = n % C::QH_SLOTS;
    parts = 0;
    if (n >= C::QH_SLOTS && !mbar_wait(&sh.qh_empty[s], ((n / C::QH_SLOTS) - 1) & 1, &sh.abort_flag, lim))
      return false;
    load_half(&sh.qh_full[s], sQh + s * C::HALF_BYTES, &p.tmQ, h, pos.i, pos.bh);
    ++parts;
    if (n > 0 && !mbar_wait(&sh.qo_empty, (n - 1) & 1, &sh.abort_flag, lim)) return false;
    load_half(&sh.qo_full, sQo, &p.tmQ, 1 - h, pos.i, pos.bh);
    ++parts;
    if (n > 0 && !mbar_wait(&sh.doo_empty, (n - 1) & 1, &sh.abort_flag, lim)) return false;
    load_half(&sh.doo_full, sDOo, &p.tmdO, 1 - h, pos.i, pos.bh);
    ++parts;
    if (n > 0 && !mbar_wait(&sh.doh_empty, (n - 1) & 1, &sh.abort_flag, lim)) return false;
    load_half(&sh.doh_full, sDOh, &p.tmdO, h, pos.i, pos.bh);
    parts = 0;
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
    const Work256<CAUSAL> wk(item, p.BHkv, p.N, p.group);
    const int n_iter = wk.n_iter();
    typename Work256<CAUSAL>::Pos pos = wk.first();
    if (!load_tile(g, pos, wk.h)) {
      aborted = true;
      break;
    }
    // K_j, V_j replace the previous item's once all its MMAs are done.
    if (items > 0 && !mbar_wait(&sh.acc_done, (items - 1) & 1, &sh.abort_flag, lim)) {
      aborted = true;
      break;
    }
    if (!debug_skip_here(p.debug_skip, WHERE_BWD_LOAD, items == 0)) {  // test hook
      mbar_arrive_expect_tx(&sh.kv_full, 2 * C::KV_BYTES);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        tma_load_3d(sK + c * C::KV_CHUNK, &p.tmK, &sh.kv_full, c * 64, wk.j * 128, wk.bh);
        tma_load_3d(sV + c * C::KV_CHUNK, &p.tmV, &sh.kv_full, c * 64, wk.j * 128, wk.bh);
      }
      ++kv_issued;
    }
    for (int n = 1; n < n_iter; ++n) {
      wk.advance(pos);
      if (!load_tile(g + n, pos, wk.h)) {
        aborted = true;
        break;
      }
    }
    if (aborted) break;
    g += n_iter;
    ++items;
    item = claim_item(p.sched);
  }
  finish_claiming(p.sched);
  if (aborted) record_timeout(p.status, &sh.abort_flag, WHERE_BWD_LOAD);
  // The copies already issued land before the CTA can exit (after an abort
  // no consumer may wait for them): the latest phase of every ring slot,
  // including the half tiles of a tile cut short by the abort.
  // Each slot waits for the latest phase issued into it only (an older phase
  // of a slot can no longer be told apart once a newer one has completed).
  const int last = issued - 1;  // last fully issued tile
  const int qh_last = parts >= 1 ? issued : last;
  for (int n = std::max(0, qh_last - C::QH_SLOTS + 1); n <= qh_last; ++n)
    drain_wait(&sh.qh_full[n % C::QH_SLOTS], (n / C::QH_SLOTS) & 1, lim);
  const int qo_last = parts >= 2 ? issued : last;
  const int doo_last = parts >= 3 ? issued : last;
  if (qo_last >= 0) drain_wait(&sh.qo_full, qo_last & 1, lim);
  if (doo_last >= 0) drain_wait(&sh.doo_full, doo_last & 1, lim);
  if (last >= 0) drain_wait(&sh.doh_full, last & 1, lim);
  if (kv_issued > 0) drain_wait(&sh.kv_full, (kv_issued - 1) & 1, lim);
}

// One thread issues every MMA (order in the file header).
template <bool CAUSAL, bool DQ>
__device__ void mma_role(const BwdLaunch& p, Shared256& sh, uint8_t* sK, uint8_t* sV, uint8_t* sQh, uint8_t* sQo,
                         uint8_t* sDOh, uint8_t* sDOo, uint8_t* sDS, uint32_t tmem) {
  using C = Cfg256;
  constexpr uint32_t kIdescS = make_idesc_bf16_f32(128, 64, false, false);  // S^T, dP^T: 128 keys x 64 queries
  constexpr uint32_t kIdescAcc = make_idesc_bf16_f32(128, 128, false, true);  // dV, dK halves
  constexpr uint32_t kIdescDq = make_idesc_bf16_f32(128, 64, true, true);     // dQ^T half: 128 d x 64 queries
  const uint32_t k_addr = smem_u32(sK), v_addr = smem_u32(sV), qh_addr = smem_u32(sQh), qo_addr = smem_u32(sQo),
                 doh_addr = smem_u32(sDOh), doo_addr = smem_u32(sDOo), ds_addr = smem_u32(sDS);
  const uint64_t lim = p.wait_limit_ns;
  const int total = total_items256(p);
  auto fail = [&]() {
    record_timeout(p.status, &sh.abort_flag, WHERE_BWD_MMA);
    drain_mmas(&sh.mma_drain, lim);
  };

  // D[tmem] = A (128 keys x 256, K-major, resident) * B (64 queries x 256,
  // K-major, in the h and other-half slots)^T, chunks of 64 columns in order.
  auto issue_sq = [&](uint32_t d_col, uint32_t a_addr, uint32_t b_h, uint32_t b_o, int h) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint64_t ad = make_smem_desc_sw128(a_addr + c * C::KV_CHUNK, 16, 1024);
      const uint64_t bd = make_smem_desc_sw128(half_chunk(b_h, b_o, h, c), 16, 1024);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_ss(tmem + d_col, desc_add(ad, ks * 32), desc_add(bd, ks * 32), kIdescS, (c > 0 || ks > 0) ? 1u : 0u);
    }
  };
  auto wait_s_operands = [&](int n) -> bool {
    return mbar_wait(&sh.qh_full[n % C::QH_SLOTS], (n / C::QH_SLOTS) & 1, &sh.abort_flag, lim) &&
           mbar_wait(&sh.qo_full, n & 1, &sh.abort_flag, lim);
  };
  auto wait_dp_operands = [&](int n) -> bool {
    return mbar_wait(&sh.doo_full, n & 1, &sh.abort_flag, lim) && mbar_wait(&sh.doh_full, n & 1, &sh.abort_flag, lim);
  };
  auto issue_s = [&](int n, int h) {
    issue_sq(C::REG_S, k_addr, qh_addr + (n % C::QH_SLOTS) * C::HALF_BYTES, qo_addr, h);
    umma_commit(&sh.s_full);
    umma_commit(&sh.qo_empty);  // the other half of Q_n is read by S^T(n) only
  };
  auto issue_dp = [&](int h) {
    issue_sq(C::REG_DP, v_addr, doh_addr, doo_addr, h);
    umma_commit(&sh.dp_full);
    umma_commit(&sh.doo_empty);
  };

  int g = 0, items = 0;
  while (true) {
    const int item = take_item(sh, items, lim);
    if (item < 0) return fail();
    if (item >= total) break;
    const Work256<CAUSAL> wk(item, p.BHkv, p.N, p.group);
    const int n_iter = wk.n_iter();
    const int h = wk.h;
    if (!mbar_wait(&sh.kv_full, items & 1, &sh.abort_flag, lim) || !wait_s_operands(g)) return fail();
    // S^T overwrites the previous item's last P^T: dV must have read it.
    if (g > 0 && !mbar_wait(&sh.pv_done, (g - 1) & 1, &sh.abort_flag, lim)) return fail();
    tc_fence_after_sync();
    issue_s(g, h);
    // dP^T overwrites the previous item's last dP^T, which phase B read
    // before ds_ready (waited for in the previous item's last step).
    if (!wait_dp_operands(g)) return fail();
    tc_fence_after_sync();
    issue_dp(h);

    for (int n = 0; n < n_iter; ++n, ++g) {
      const bool has_next = n + 1 < n_iter;
      if (!mbar_wait(&sh.pa_ready, g & 1, &sh.abort_flag, lim)) return fail();
      // the first dV / dK of an item overwrite the accumulators: the previous
      // item's epilogue must have read them
      if (n == 0 && items > 0 && !mbar_wait(&sh.acc_free, (items - 1) & 1, &sh.abort_flag, lim)) return fail();
      tc_fence_after_sync();
      // dV half += P^T dO_n[:, h]; P^T (bf16) in columns [0,16) and [32,48) of REG_S
      const uint64_t dod = make_smem_desc_sw128(doh_addr, C::Q_CHUNK, 1024);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_ts(tmem + C::DV_COL, tmem + C::REG_S + (ks >> 1) * 32 + (ks & 1) * 8, desc_add(dod, ks * 2048),
                kIdescAcc, (n > 0 || ks > 0) ? 1u : 0u);
      umma_commit(&sh.pv_done);
      umma_commit(&sh.doh_empty);
      if (has_next) {
        // S^T(n+1) overwrites P^T(n): wait until dV(n) has read it.
        if (!wait_s_operands(g + 1) || !mbar_wait(&sh.pv_done, g & 1, &sh.abort_flag, lim)) return fail();
        tc_fence_after_sync();
        issue_s(g + 1, h);
      }
      if (!mbar_wait(&sh.ds_ready, g & 1, &sh.abort_flag, lim)) return fail();
      tc_fence_after_sync();
      // dK half += dS^T Q_n[:, h]
      const uint32_t qh = qh_addr + (g % C::QH_SLOTS) * C::HALF_BYTES;
      const uint64_t dsk = make_smem_desc_sw128(ds_addr, 16, 1024), qmn = make_smem_desc_sw128(qh, C::Q_CHUNK, 1024);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_ss(tmem + C::DK_COL, desc_add(dsk, ks * 32), desc_add(qmn, ks * 2048), kIdescAcc,
                (n > 0 || ks > 0) ? 1u : 0u);
      umma_commit(&sh.qh_empty[g % C::QH_SLOTS]);
      if constexpr (DQ) {
        // dQ_n^T half = K_j[:, h]^T dS^T into buffer g & 1, once the drain of
        // tile g - 2 has read it
        const int b = g & 1;
        if (g >= 2 && !mbar_wait(&sh.dq_free[b], ((g >> 1) - 1) & 1, &sh.abort_flag, lim)) return fail();
        tc_fence_after_sync();
        const uint64_t kd = make_smem_desc_sw128(k_addr + 2 * h * C::KV_CHUNK, C::KV_CHUNK, 1024);
        const uint64_t dsm = make_smem_desc_sw128(ds_addr, C::DS_BYTES, 1024);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          umma_ss(tmem + C::dq_col(b), desc_add(kd, ks * 2048), desc_add(dsm, ks * 2048), kIdescDq, ks > 0 ? 1u : 0u);
        umma_commit(&sh.dq_full[b]);
      }
      if (has_next) {
        // dP^T(n+1): phase B(n) has read dP^T(n) (ds_ready above)
        if (!wait_dp_operands(g + 1)) return fail();
        tc_fence_after_sync();
        issue_dp(h);
      }
    }
    umma_commit(&sh.acc_done);
    ++items;
  }
  // Normally the epilogues have waited for the last products; if a softmax
  // warpgroup gave up, nothing has.
  drain_mmas(&sh.mma_drain, lim);
}

// Warpgroup w (w = 0, 1) owns queries [32w, 32w + 32) of every 64-row tile;
// thread r owns key r (TMEM lane r) in phases A and B and head-dim column
// 128h + r in the dQ drain. Order per tile n: B(n), A(n+1), drain(n). After
// an item's last tile warpgroup 0 writes its dK half and warpgroup 1 its dV
// half straight from TMEM.
template <bool CAUSAL, bool DQ>
__device__ void softmax_role(const BwdLaunch& p, Shared256& sh, uint8_t* sDS, float* sLD, uint32_t tmem, int w) {
  using C = Cfg256;
  const int r = threadIdx.x & 127;
  const uint32_t lane_base = static_cast<uint32_t>((threadIdx.x >> 5) & 3) << 21;
  const float c2 = p.scale_log2;
  const float sc = p.scale;
  const uint64_t lim = p.wait_limit_ns;
  float* ld_l2 = sLD + w * 64;  // 32 base-2 logsumexps, then 32 scaled D values
  float* ld_d = ld_l2 + 32;
  const uint32_t bar_id = 1 + w;
  const uint32_t tA = tmem + lane_base + C::REG_S + 32 * w;
  const uint32_t tB = tmem + lane_base + C::REG_DP + 32 * w;
  const int total = total_items256(p);
  bool alive = true;
  uint32_t pk[16];  // P^T of the current tile (bf16 pairs, as written to TMEM): dS uses the same rounding

  // thread r < 32 loads L2 of query 32w + r of the tile, 32 <= r < 64 its scaled D
  auto fetch_ld = [&](int bh, int i) -> float {
    const size_t row = static_cast<size_t>(bh) * p.Npad + i * C::BQ + 32 * w;
    if (r < 32) return __ldg(p.lse2 + row + r);
    if (r < 64) return __ldg(p.D + row + (r - 32)) * sc;
    return 0.f;
  };
  auto wait_all = [&](uint64_t* bar, int parity, int where) {
    alive = alive && __all_sync(0xffffffffu, mbar_wait(bar, parity, &sh.abort_flag, lim));
    if (!alive) record_timeout(p.status, &sh.abort_flag, where);
    tc_fence_after_sync();
  };

  // ---- phase A of query tile i (global tile g): P^T -> TMEM (bf16)
  auto phase_a = [&](const Work256<CAUSAL>& wk, int i, int g) {
    wait_all(&sh.s_full, g & 1, WHERE_BWD_SOFTMAX);
    if (!alive) return;
    uint32_t a[32];
    tmem_ld32(tA, a);
    tmem_ld_wait();
    // key 128j + r is seen by query 64i + 32w + c if it exists and (causal)
    // is not after the query: c >= c_lo
    const int key = wk.j * 128 + r;
    const bool key_valid = key < p.N;
    const int c_lo = CAUSAL ? key - i * C::BQ - 32 * w : 0;
    float pv[32];
#pragma unroll
    for (int c4 = 0; c4 < 32; c4 += 4) {
      const float4 l = *reinterpret_cast<const float4*>(ld_l2 + c4);
      const float2 x01 = ffma2_bcast_mul(__uint_as_float(a[c4]), __uint_as_float(a[c4 + 1]), c2, -l.x, -l.y);
      const float2 x23 = ffma2_bcast_mul(__uint_as_float(a[c4 + 2]), __uint_as_float(a[c4 + 3]), c2, -l.z, -l.w);
      pv[c4] = x01.x;
      pv[c4 + 1] = x01.y;
      pv[c4 + 2] = x23.x;
      pv[c4 + 3] = x23.y;
    }
#pragma unroll
    for (int c = 0; c < 32; ++c) pv[c] = ex2_approx(pv[c]);
    if (!key_valid || (CAUSAL && c_lo > 0)) {
#pragma unroll
      for (int c = 0; c < 32; ++c)
        if (!key_valid || c < c_lo) pv[c] = 0.f;
    }
#pragma unroll
    for (int c = 0; c < 16; ++c) pk[c] = pack_bf16x2(pv[2 * c], pv[2 * c + 1]);
    tmem_st16(tA, pk);  // columns [32w, 32w + 16): already read
    tmem_st_wait();
    tc_fence_before_sync();
    mbar_arrive(&sh.pa_ready);
  };

  // ---- phase B: dS^T = P^T o (dP^T - D) * scale -> smem row r, queries [32w, 32w + 32)
  auto phase_b = [&](int g) {
    wait_all(&sh.dp_full, g & 1, WHERE_BWD_SOFTMAX);
    if (!alive) return;
    uint32_t dpv[32];
    tmem_ld32(tB, dpv);
    tmem_ld_wait();
    uint32_t dk[16];
#pragma unroll
    for (int c4 = 0; c4 < 32; c4 += 4) {
      const float4 dd = *reinterpret_cast<const float4*>(ld_d + c4);
      const float2 p01 = unpack_bf16x2(pk[c4 / 2]);
      const float2 p23 = unpack_bf16x2(pk[c4 / 2 + 1]);
      const float2 g01 = ffma2_bcast_mul(__uint_as_float(dpv[c4]), __uint_as_float(dpv[c4 + 1]), sc, -dd.x, -dd.y);
      const float2 g23 = ffma2_bcast_mul(__uint_as_float(dpv[c4 + 2]), __uint_as_float(dpv[c4 + 3]), sc, -dd.z, -dd.w);
      const float2 ds01 = fmul2(p01, g01);
      const float2 ds23 = fmul2(p23, g23);
      dk[c4 / 2] = pack_bf16x2(ds01.x, ds01.y);
      dk[c4 / 2 + 1] = pack_bf16x2(ds23.x, ds23.y);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      st_shared_v4(smem_u32(sDS) + sw128_offset(r, 4 * w + u), dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
    fence_proxy_async_smem();
    tc_fence_before_sync();
    mbar_arrive(&sh.ds_ready);
  };

  // ---- dQ drain of query tile i (global tile g): lane r = head-dim column
  // 128h + r, this warpgroup's 32 queries along the columns; for a fixed
  // query a warp's 32 lanes add into 32 consecutive floats (one full line).
  auto drain = [&](int bh, int i, int h, int g) {
    const int b = g & 1;
    wait_all(&sh.dq_full[b], (g >> 1) & 1, WHERE_BWD_DQ);
    if (!alive) return;
    uint32_t v[32];
    tmem_ld32(tmem + lane_base + C::dq_col(b) + 32 * w, v);
    tmem_ld_wait();
    tc_fence_before_sync();
    mbar_arrive(&sh.dq_free[b]);
    float* dst = p.dq_acc + (static_cast<size_t>(bh) * p.Npad + i * C::BQ + 32 * w) * C::HD + 128 * h + r;
#pragma unroll
    for (int c = 0; c < 32; ++c) red_add_f32(dst + static_cast<size_t>(c) * C::HD, __uint_as_float(v[c]));
  };

  // ---- item epilogue: w = 0 writes the dK half, w = 1 the dV half; thread r
  // writes key row r (rows past N are skipped)
  auto epilogue = [&](const Work256<CAUSAL>& wk, int items) {
    wait_all(&sh.acc_done, items & 1, WHERE_BWD_SOFTMAX);
    if (!alive) return;
    const int key = wk.j * 128 + r;
    const uint32_t t = tmem + lane_base + (w == 0 ? C::DK_COL : C::DV_COL);
    __nv_bfloat16* dst = (w == 0 ? p.dk : p.dv) + (static_cast<size_t>(wk.bh) * p.N + key) * C::HD + 128 * wk.h;
#pragma unroll 1
    for (int c = 0; c < 128; c += 32) {
      uint32_t v[32];
      tmem_ld32(t + c, v);
      tmem_ld_wait();
      if (c + 32 == 128) {  // both accumulators read: the next item may overwrite them
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
  };

  // The next work item, agreed on by the whole warpgroup (as in fa_bwd.cu).
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
    const Work256<CAUSAL> wk0(item, p.BHkv, p.N, p.group);
    const typename Work256<CAUSAL>::Pos f0 = wk0.first();
    ld = fetch_ld(f0.bh, f0.i);
  }
  while (item < total) {
    const Work256<CAUSAL> wk(item, p.BHkv, p.N, p.group);
    const int n_iter = wk.n_iter();
    if (items > 0) named_barrier_sync(bar_id, 128);  // the previous item's L2 / D reads are done
    if (r < 64) sLD[w * 64 + r] = ld;
    named_barrier_sync(bar_id, 128);
    typename Work256<CAUSAL>::Pos cur = wk.first();
    phase_a(wk, cur.i, g);
    for (int n = 0; n < n_iter; ++n) {
      const bool has_next = n + 1 < n_iter;
      typename Work256<CAUSAL>::Pos nxt = cur;
      wk.advance(nxt);
      const float next_ld = has_next ? fetch_ld(nxt.bh, nxt.i) : 0.f;  // lands during phase B
      phase_b(g + n);
      if (has_next) {
        named_barrier_sync(bar_id, 128);  // every thread is done reading this tile's L2 / D
        if (r < 64) sLD[w * 64 + r] = next_ld;
        named_barrier_sync(bar_id, 128);
        phase_a(wk, nxt.i, g + n + 1);
      }
      if constexpr (DQ) drain(cur.bh, cur.i, wk.h, g + n);
      cur = nxt;
    }
    const int item_next = next_item(items + 1);
    if (item_next < total) {
      const Work256<CAUSAL> wk1(item_next, p.BHkv, p.N, p.group);
      const typename Work256<CAUSAL>::Pos f1 = wk1.first();
      ld = fetch_ld(f1.bh, f1.i);  // lands during the epilogue
    }
    epilogue(wk, items);
    g += n_iter;
    ++items;
    item = item_next;
  }
}

template <bool CAUSAL, bool DQ>
__global__ void __launch_bounds__(kThreads, 1) fa_bwd256_kernel(const __grid_constant__ BwdLaunch p) {
  using C = Cfg256;
  extern __shared__ uint8_t smem_dyn[];
  __shared__ Shared256 sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = sK + C::KV_BYTES;
  uint8_t* sQh = sV + C::KV_BYTES;                 // QH_SLOTS half tiles
  uint8_t* sQo = sQh + C::QH_SLOTS * C::HALF_BYTES;
  uint8_t* sDOh = sQo + C::HALF_BYTES;
  uint8_t* sDOo = sDOh + C::HALF_BYTES;
  uint8_t* sDS = sDOo + C::HALF_BYTES;
  float* sLD = reinterpret_cast<float*>(sDS + C::DS_BYTES);
  const int warp = threadIdx.x >> 5;
  // Without dQ this pass writes nothing the dQ kernel reads, so a dQ kernel
  // queued behind it may take SMs as soon as this grid's CTAs leave them.
  if constexpr (!DQ) griddep_launch_dependents();

  if (threadIdx.x == 0) {
    mbar_init(&sh.kv_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sh.qh_full[s], 1);
      mbar_init(&sh.qh_empty[s], 1);
      mbar_init(&sh.dq_full[s], 1);
      // test hook: buffer 0's dQ barrier waits for one arrival too many
      mbar_init(&sh.dq_free[s], 256 + (s == 0 ? debug_extra(p.debug_skip, WHERE_BWD_DQ) : 0u));
    }
    mbar_init(&sh.qo_full, 1);
    mbar_init(&sh.qo_empty, 1);
    mbar_init(&sh.doh_full, 1);
    mbar_init(&sh.doh_empty, 1);
    mbar_init(&sh.doo_full, 1);
    mbar_init(&sh.doo_empty, 1);
    // test hook: the S or P barrier waits for one arrival too many
    mbar_init(&sh.s_full, 1 + debug_extra(p.debug_skip, WHERE_BWD_MMA));
    mbar_init(&sh.dp_full, 1);
    mbar_init(&sh.pa_ready, 256 + debug_extra(p.debug_skip, WHERE_BWD_SOFTMAX));
    mbar_init(&sh.ds_ready, 256);
    mbar_init(&sh.pv_done, 1);
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
    if (lane_id() == 0) load_role<CAUSAL>(p, sh, sK, sV, sQh, sQo, sDOh, sDOo);
  } else if (warp == kMmaWarp) {
    if (lane_id() == 0) mma_role<CAUSAL, DQ>(p, sh, sK, sV, sQh, sQo, sDOh, sDOo, sDS, tmem);
  } else {
    softmax_role<CAUSAL, DQ>(p, sh, sDS, sLD, tmem, warp >> 2);
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

template <bool CAUSAL, bool DQ>
cudaError_t launch_t(const BwdLaunch& a, cudaStream_t stream) {
  auto kern = fa_bwd256_kernel<CAUSAL, DQ>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg256::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const long long items = static_cast<long long>(a.BHkv) * ((a.N + 127) / 128) * 2;
  // Persistent: one CTA per SM (the smem footprint allows no more).
  const long long grid = items < a.num_sms ? items : a.num_sms;
  kern<<<static_cast<unsigned>(grid), kThreads, Cfg256::SMEM_BYTES, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_main_d256(const BwdLaunch& a, cudaStream_t stream) {
  if (a.deterministic)
    return a.causal ? launch_t<true, false>(a, stream) : launch_t<false, false>(a, stream);
  return a.causal ? launch_t<true, true>(a, stream) : launch_t<false, true>(a, stream);
}

}  // namespace fa

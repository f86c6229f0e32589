// Forward pass of exact softmax attention for sm_103a: the kernel templates,
// instantiated by fa_fwd.cu (one head per tile) and fa_fwd_pack.cu (grouped
// query heads packed into a tile).
//
// Method (web pages on FlashAttention-2):
//   "FlashAttention 2: ..." reading note (papers.chlience.com) 5.1-5.2 and the
//   paper-graph-ui summary, "Algorithm 1 Walkthrough": for a query block Q_i
//   keep a running row max m, running sum l and an UNSCALED accumulator O~;
//   for each key block j: S = Q_i K_j^T, m' = max(m, rowmax S),
//   P~ = exp(S - m'), l = e^{m - m'} l + rowsum P~, O~ = e^{m - m'} O~ + P~ V_j;
//   at the end O = O~ / l and L = m + log l (the only statistics stored).
//   Causal key blocks entirely right of the diagonal are skipped and only the
//   diagonal block is masked element-wise (summary, "Causal masking
//   optimization"; reading note 5.6).
//
// GB300 mapping (our design; the pages' A100 warp layout does not apply):
//   - One CTA owns NT query tiles of 128 rows of one (batch, head) (NT = 2
//     for d <= 128, 1 for d = 256) and streams the 128-key K/V tiles of that
//     head through a TMA + mbarrier ring.
//   - Warp 9 (one thread) issues tcgen05 MMAs: S_t = Q_t K_j^T into TMEM
//     (SS, both operands K-major in 128-byte-swizzled smem) and
//     O~_t += P_t V_j (A = P_t read from TMEM, B = V_j MN-major in smem).
//   - Warp 8 (one thread) issues the TMA loads.
//   - Warpgroup t (warps 4t..4t+3) owns query tile t: thread r <-> query row r
//     <-> TMEM lane r. It reads its row of S from TMEM, keeps m (in base-2
//     units of the scaled scores) and l in registers, computes
//     P~ = 2^(S*scale*log2e - m) with one FFMA + ex2 per element, writes P~
//     as bf16 back to TMEM, and rescales its row of O~ in TMEM only when the
//     row max grew (by more than 8 in base-2 units for some row of the warp;
//     smaller growth is absorbed with P~ <= 2^8).
//   - While warpgroup 0 does softmax on tile 0 the tensor core works on
//     tile 1 and vice versa.
//   - Epilogue: O = O~ / l converted to bf16 into the (now free) Q tile's
//     smem in the TMA swizzle, one TMA store; L = ln2 * (m + log2 l).
//
// TMEM columns (512 allocated):
//   d=64 : S0 0, S1 128, O0 256, O1 320, P0 384, P1 448
//   d=128: S0 0, S1 128, O0 256, O1 384, P_t aliases the first 64 columns of
//          S_t, so S_t(j+1) is issued only after O_t += P_t V_j completed
//   d=256: S 0, P 128, O 256
#pragma once

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
constexpr float kLn2 = 0.69314718055994530942f;
// Largest growth of a row max (in base-2 units of the scaled scores) absorbed
// without rescaling: P~ <= 2^8 is exact in bf16's exponent range and l, O~
// stay far from fp32 overflow.
constexpr float kRescaleSlack = 8.0f;

template <int HD>
struct FwdCfg {
  static constexpr int NT = HD <= 128 ? 2 : 1;
  static constexpr int CHUNKS = HD / 64;             // 64-column (128-byte) swizzle chunks
  static constexpr int TILE_BYTES = 128 * HD * 2;    // one 128-row bf16 tile
  static constexpr int CHUNK_BYTES = 128 * 128;      // 128 rows x 128 bytes
  static constexpr int KST = HD == 64 ? 4 : (HD == 128 ? 2 : 1);
  static constexpr int VST = KST;
  static constexpr bool P_ALIAS = HD == 128;
  __host__ __device__ static constexpr uint32_t s_col(int t) { return HD == 256 ? 0u : uint32_t(t) * 128u; }
  __host__ __device__ static constexpr uint32_t o_col(int t) { return 256u + uint32_t(t) * HD; }
  __host__ __device__ static constexpr uint32_t p_col(int t) {
    return HD == 64 ? 384u + uint32_t(t) * 64u : (HD == 128 ? uint32_t(t) * 128u : 128u);
  }
  static constexpr int SMEM_BYTES = (NT + KST + VST) * TILE_BYTES + 1024;
};

struct FwdShared {
  uint64_t q_full[2], q_free[2];  // per query-tile slot
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2], p_full[2], pv_done[2], o_free[2];
  uint64_t mma_drain;  // the MMA thread's last commit: all its MMAs done before the CTA exits
  uint32_t tmem_base;
  int abort_flag;
};

// Rows per head and heads per tile: compile-time 128 and 1 unless the kernel
// is the instantiation that packs grouped query heads.
template <bool PACK>
__device__ __forceinline__ int rows_per_head(const FwdLaunch& p) {
  return PACK ? p.rph : 128;
}
template <bool PACK>
__device__ __forceinline__ int heads_per_tile(const FwdLaunch& p) {
  return PACK ? p.pack : 1;
}

// Work item: NT consecutive 128-row query tiles of query heads bh .. bh +
// pack - 1 and key range s (key tiles kv0 .. kv0 + kv_per_split - 1; one range
// covers every key unless the keys are split). A tile holds rph = 128 / pack
// positions of each of its pack heads, head-major: row r is position
// qt * rph + r % rph of head bh + r / rph. pack > 1 gathers the query heads
// that share one K/V head, so a short query block (decoding) reads each K/V
// tile once for the whole group. Items are numbered longest-first under a
// causal mask (the last query tiles see the most keys); non-causal items of
// one head are adjacent (K/V reuse in L2). Key-tile indices inside an item
// are relative to kv0.
template <int NT, bool CAUSAL, bool PACK>
struct FwdWork {
  int bh, s, kv0;
  int qt[NT];       // query tile indices
  int last_kv[NT];  // last key tile each query tile needs in this range; -1: none (or past the end)
  int nkv;          // number of key tiles streamed
  __device__ FwdWork(int item, const FwdLaunch& p) {
    const int rph = rows_per_head<PACK>(p), pack = heads_per_tile<PACK>(p);
    const int Tq = (p.Nq + rph - 1) / rph;
    const int Tk = (p.Nk + 127) / 128;
    const int n_w = (Tq + NT - 1) / NT;
    const int units = p.BH / pack;
    int w;
    if (CAUSAL) {
      const int u = item % (units * p.splits);
      w = n_w - 1 - item / (units * p.splits);
      bh = u / p.splits;
      s = u - bh * p.splits;
    } else {
      bh = item / (n_w * p.splits);
      const int rem = item - bh * (n_w * p.splits);
      w = rem / p.splits;
      s = rem - w * p.splits;
    }
    bh *= pack;
    kv0 = s * p.kv_per_split;
    const int kv_end = min(Tk, kv0 + p.kv_per_split) - 1;
    nkv = 0;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      qt[t] = w * NT + t;
      int last = -1;
      if (qt[t] < Tq) {
        int lim = kv_end;
        // causal: the tile's last row sees keys up to its index + causal_off
        if (CAUSAL) lim = min(lim, (min(qt[t] * rph + rph - 1, p.Nq - 1) + p.causal_off) / 128);
        last = max(lim - kv0, -1);
      }
      last_kv[t] = last;
      nkv = max(nkv, last + 1);
    }
  }
};

// Persistent schedule: CTA b of G takes items in rounds k = 0, 1, ...; round
// k holds items [kG, kG + G) and is walked forwards on even rounds and
// backwards on odd ones, so with items sorted longest-first every CTA gets a
// similar total.
__device__ __forceinline__ int sched_item(int k, int b, int G) { return k * G + ((k & 1) ? G - 1 - b : b); }

template <bool PACK>
__device__ __forceinline__ int total_items(const FwdLaunch& p, int NT) {
  const int rph = rows_per_head<PACK>(p);
  const int Tq = (p.Nq + rph - 1) / rph;
  return (p.BH / heads_per_tile<PACK>(p)) * ((Tq + NT - 1) / NT) * p.splits;
}

// Fetch one tile of a tensor map into L2 (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

// ---------------------------------------------------------------------------
// TMA producer (one thread)
// ---------------------------------------------------------------------------
template <int HD, bool CAUSAL, bool PACK>
__device__ void fwd_load_role(const FwdLaunch& p, FwdShared& sh, uint8_t* sQ, uint8_t* sK, uint8_t* sV) {
  using C = FwdCfg<HD>;
  tma_prefetch_desc(&p.tmQ);
  tma_prefetch_desc(&p.tmK);
  tma_prefetch_desc(&p.tmV);
  tma_prefetch_desc(&p.tmO);
  const int total = total_items<PACK>(p, C::NT);
  const int G = gridDim.x;
  const uint64_t lim = p.wait_limit_ns;
  int kv = 0;     // running count of K/V tiles loaded by this CTA
  int items = 0;  // items started
  int k_issued = 0, v_issued = 0;
  int q_item = -1;      // the latest item whose Q loads were issued ...
  unsigned q_mask = 0;  // ... and its slots
  bool aborted = false;
  for (int k = 0; k * G < total && !aborted; ++k) {
    const int item = sched_item(k, blockIdx.x, G);
    if (item >= total) continue;
    const FwdWork<C::NT, CAUSAL, PACK> wk(item, p);
    if (wk.nkv == 0) continue;  // a key range with nothing to do (every role skips it)
    const int kv_bh = wk.bh / p.group;  // grouped K/V heads: query head bh reads K/V head bh / g
    // Q_t's smem was the previous item's O staging: wait until its store read
    // it. The item's first K/V tile is issued before that wait so it loads
    // while the previous epilogue runs. Each slot has its own q_full, and the
    // two warpgroups' epilogues end at different times, so Q_0 (and with it
    // S_0(0)) does not wait for slot 1's epilogue. An empty slot's q_full
    // still completes one phase per item (an arrival without bytes).
    auto load_q = [&]() -> bool {
      q_mask = 0;
#pragma unroll
      for (int t = 0; t < C::NT; ++t) {
        if (items > 0 && !mbar_wait(&sh.q_free[t], (items - 1) & 1, &sh.abort_flag, lim)) return false;
        if (wk.last_kv[t] < 0) {
          mbar_arrive(&sh.q_full[t]);
          continue;
        }
        if (debug_skip_here(p.debug_skip, WHERE_FWD_LOAD, items == 0 && t == 0)) continue;  // test hook
        mbar_arrive_expect_tx(&sh.q_full[t], C::TILE_BYTES);
#pragma unroll
        for (int c = 0; c < C::CHUNKS; ++c)
          tma_load_3d(sQ + t * C::TILE_BYTES + c * C::CHUNK_BYTES, &p.tmQ, &sh.q_full[t], c * 64,
                      wk.qt[t] * rows_per_head<PACK>(p), wk.bh);
        q_item = items;
        q_mask |= 1u << t;
      }
      return true;
    };
    for (int j = 0; j < wk.nkv; ++j, ++kv) {
      const int ks = kv % C::KST;
      if (kv >= C::KST && !mbar_wait(&sh.k_empty[ks], ((kv / C::KST) - 1) & 1, &sh.abort_flag, lim)) {
        aborted = true;
        break;
      }
      mbar_arrive_expect_tx(&sh.k_full[ks], C::TILE_BYTES);
#pragma unroll
      for (int c = 0; c < C::CHUNKS; ++c)
        tma_load_3d(sK + ks * C::TILE_BYTES + c * C::CHUNK_BYTES, &p.tmK, &sh.k_full[ks], c * 64, (wk.kv0 + j) * 128,
                    kv_bh);
      ++k_issued;
      if (j == 0) {
        if (!load_q()) {
          aborted = true;
          break;
        }
        // The next item's Q tiles come from HBM (each query tile is read
        // once) and are loaded only after this item's epilogue: fetch them
        // into L2 now, so that load is an L2 hit. It matters for short
        // sequences, whose items hold only a few key tiles.
        const int next = (k + 1) * G < total ? sched_item(k + 1, blockIdx.x, G) : total;
        if (next < total) {
          const FwdWork<C::NT, CAUSAL, PACK> wn(next, p);
#pragma unroll
          for (int t = 0; t < C::NT; ++t) {
            if (wn.nkv == 0 || wn.last_kv[t] < 0) continue;
#pragma unroll
            for (int c = 0; c < C::CHUNKS; ++c)
              tma_prefetch_l2_3d(&p.tmQ, c * 64, wn.qt[t] * rows_per_head<PACK>(p), wn.bh);
          }
        }
      }
      const int vs = kv % C::VST;
      if (kv >= C::VST && !mbar_wait(&sh.v_empty[vs], ((kv / C::VST) - 1) & 1, &sh.abort_flag, lim)) {
        aborted = true;
        break;
      }
      mbar_arrive_expect_tx(&sh.v_full[vs], C::TILE_BYTES);
#pragma unroll
      for (int c = 0; c < C::CHUNKS; ++c)
        tma_load_3d(sV + vs * C::TILE_BYTES + c * C::CHUNK_BYTES, &p.tmV, &sh.v_full[vs], c * 64, (wk.kv0 + j) * 128,
                    kv_bh);
      ++v_issued;
    }
    if (aborted) break;
    ++items;
  }
  if (aborted) record_timeout(p.status, &sh.abort_flag, WHERE_FWD_LOAD);
  // The copies already issued land before the CTA can exit (after an abort
  // no consumer may wait for them).
  for (int jj = max(0, k_issued - C::KST); jj < k_issued; ++jj)
    drain_wait(&sh.k_full[jj % C::KST], (jj / C::KST) & 1, lim);
  for (int jj = max(0, v_issued - C::VST); jj < v_issued; ++jj)
    drain_wait(&sh.v_full[jj % C::VST], (jj / C::VST) & 1, lim);
  for (int t = 0; t < C::NT; ++t)
    if (q_mask >> t & 1) drain_wait(&sh.q_full[t], q_item & 1, lim);
}

// ---------------------------------------------------------------------------
// MMA issuer (one thread)
// ---------------------------------------------------------------------------
template <int HD, bool CAUSAL, bool PACK>
__device__ void fwd_mma_role(const FwdLaunch& p, FwdShared& sh, uint8_t* sQ, uint8_t* sK, uint8_t* sV,
                             uint32_t tmem) {
  using C = FwdCfg<HD>;
  constexpr uint32_t kIdescS = make_idesc_bf16_f32(128, 128, false, false);
  constexpr uint32_t kIdescPV = make_idesc_bf16_f32(128, HD, false, true);
  const uint32_t q_addr = smem_u32(sQ), k_addr = smem_u32(sK), v_addr = smem_u32(sV);
  const uint64_t lim = p.wait_limit_ns;
  const int total = total_items<PACK>(p, C::NT);
  const int G = gridDim.x;

  auto issue_s = [&](int t, int g) {  // g: running K/V tile index
    const uint32_t qa = q_addr + t * C::TILE_BYTES;
    const uint32_t ka = k_addr + (g % C::KST) * C::TILE_BYTES;
    const uint64_t qd = make_smem_desc_sw128(qa, 16, 1024), kd = make_smem_desc_sw128(ka, 16, 1024);
#pragma unroll
    for (int ks = 0; ks < HD / 16; ++ks) {
      const uint32_t off = (ks >> 2) * C::CHUNK_BYTES + (ks & 3) * 32;
      umma_ss(tmem + C::s_col(t), desc_add(qd, off), desc_add(kd, off), kIdescS, ks > 0 ? 1u : 0u);
    }
    umma_commit(&sh.s_full[t]);
  };
  auto issue_pv = [&](int t, int g, bool first) {
    const uint64_t vd = make_smem_desc_sw128(v_addr + (g % C::VST) * C::TILE_BYTES, C::CHUNK_BYTES, 1024);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      umma_ts(tmem + C::o_col(t), tmem + C::p_col(t) + ks * 8, desc_add(vd, ks * 2048), kIdescPV,
              (!first || ks > 0) ? 1u : 0u);
    umma_commit(&sh.pv_done[t]);
  };
  auto fail = [&]() {
    record_timeout(p.status, &sh.abort_flag, WHERE_FWD_MMA);
    drain_mmas(&sh.mma_drain, lim);
  };

  int kv = 0;             // running K/V tile index
  int items = 0;          // items processed
  int cnt[2] = {0, 0};    // running S / P / PV count per query-tile slot
  for (int k = 0; k * G < total; ++k) {
    const int item = sched_item(k, blockIdx.x, G);
    if (item >= total) continue;
    const FwdWork<C::NT, CAUSAL, PACK> wk(item, p);
    if (wk.nkv == 0) continue;
    if (!mbar_wait(&sh.k_full[kv % C::KST], (kv / C::KST) & 1, &sh.abort_flag, lim)) return fail();
    tc_fence_after_sync();
#pragma unroll
    for (int t = 0; t < C::NT; ++t) {
      if (wk.last_kv[t] < 0) continue;
      // S_t(0) overwrites S_t / P~_t of the previous item: its last PV must be done.
      if (C::P_ALIAS && cnt[t] > 0 && !mbar_wait(&sh.pv_done[t], (cnt[t] - 1) & 1, &sh.abort_flag, lim))
        return fail();
      if (!mbar_wait(&sh.q_full[t], items & 1, &sh.abort_flag, lim)) return fail();
      tc_fence_after_sync();
      issue_s(t, kv);
    }
    umma_commit(&sh.k_empty[kv % C::KST]);

    for (int j = 0; j < wk.nkv; ++j) {
      const int g = kv + j;
      const int vs = g % C::VST;
      if (!mbar_wait(&sh.v_full[vs], (g / C::VST) & 1, &sh.abort_flag, lim)) return fail();
      const bool has_next = j + 1 < wk.nkv;
      const int gn = g + 1;
      bool k_next_ready = false;
      auto wait_k_next = [&]() -> bool {
        if (k_next_ready) return true;
        if (!mbar_wait(&sh.k_full[gn % C::KST], (gn / C::KST) & 1, &sh.abort_flag, lim)) return false;
        tc_fence_after_sync();
        k_next_ready = true;
        return true;
      };
#pragma unroll
      for (int t = 0; t < C::NT; ++t) {
        if (j > wk.last_kv[t]) continue;
        if (!mbar_wait(&sh.p_full[t], (cnt[t] + j) & 1, &sh.abort_flag, lim)) return fail();
        // PV_t(0) overwrites O~_t: the previous item's epilogue must have read it.
        if (j == 0 && items > 0 && !mbar_wait(&sh.o_free[t], (items - 1) & 1, &sh.abort_flag, lim)) return fail();
        tc_fence_after_sync();
        issue_pv(t, g, j == 0);
        if (has_next && j + 1 <= wk.last_kv[t]) {
          if (!wait_k_next()) return fail();
          // d = 128: S_t(j+1) overwrites the TMEM columns P_t(j) is read
          // from, so it follows PV_t(j) directly, before the other tile's PV:
          // tile t's products then run while the other tile is in its
          // softmax (the two tiles alternate instead of moving in lockstep).
          if (C::P_ALIAS && !mbar_wait(&sh.pv_done[t], (cnt[t] + j) & 1, &sh.abort_flag, lim)) return fail();
          tc_fence_after_sync();
          issue_s(t, gn);
        }
      }
      if (has_next) umma_commit(&sh.k_empty[gn % C::KST]);
      umma_commit(&sh.v_empty[vs]);
    }
#pragma unroll
    for (int t = 0; t < C::NT; ++t)
      if (wk.last_kv[t] >= 0) cnt[t] += wk.last_kv[t] + 1;
    kv += wk.nkv;
    ++items;
  }
  // Normally the epilogues have waited for the last products; if a softmax
  // warpgroup gave up, nothing has.
  drain_mmas(&sh.mma_drain, lim);
}

// ---------------------------------------------------------------------------
// Softmax + correction + epilogue (warpgroup t owns query-tile slot t)
// ---------------------------------------------------------------------------
template <int HD, bool CAUSAL, bool PACK>
__device__ void fwd_softmax_role(const FwdLaunch& p, FwdShared& sh, uint8_t* sQ, uint32_t tmem, int t) {
  using C = FwdCfg<HD>;
  const int r = threadIdx.x & 127;
  const uint32_t lane_base = static_cast<uint32_t>((threadIdx.x >> 5) & 3) << 21;  // (warp % 4) * 32 lanes
  const uint32_t tS = tmem + lane_base + C::s_col(t);
  const uint32_t tP = tmem + lane_base + C::p_col(t);
  const uint32_t tO = tmem + lane_base + C::o_col(t);
  const int Nq = p.Nq, Nk = p.Nk;
  const int Tk = (Nk + 127) / 128;
  const float c2 = p.scale_log2;
  const uint64_t lim = p.wait_limit_ns;
  const int total = total_items<PACK>(p, C::NT);
  const int G = gridDim.x;
  uint8_t* stage = sQ + t * C::TILE_BYTES;  // O staging: Q_t once its last S MMA is done
  // After a timed-out wait a warp stops working but keeps passing every named
  // barrier and arrival, so the warpgroup's barrier counts stay matched.
  bool alive = true;
  int cnt = 0;    // running S / P count of this slot
  int items = 0;  // items processed (those with work)

  for (int k = 0; k * G < total; ++k) {
    const int item = sched_item(k, blockIdx.x, G);
    if (item >= total) continue;
    const FwdWork<C::NT, CAUSAL, PACK> wk(item, p);
    if (wk.nkv == 0) continue;
    const int qt = wk.qt[t];
    const int last_kv = wk.last_kv[t];
    // this thread's query: position `row` of head `head` (rph is a power of two)
    const int rph = rows_per_head<PACK>(p);
    const int row = qt * rph + (r & (rph - 1));
    const int head = wk.bh + r / rph;

    float m2 = -INFINITY;  // reference max of S * scale * log2(e)
    float l = 0.f;         // running sum of P~ (unrounded fp32)
    for (int j = 0; j <= last_kv; ++j) {
      alive = alive && __all_sync(0xffffffffu, mbar_wait(&sh.s_full[t], (cnt + j) & 1, &sh.abort_flag, lim));
      if (!alive) {
        record_timeout(p.status, &sh.abort_flag, WHERE_FWD_SOFTMAX);
        break;
      }
      tc_fence_after_sync();
      float s[128];
      {
        uint32_t a[32], b[32], c[32], d[32];
        tmem_ld32(tS + 0, a);
        tmem_ld32(tS + 32, b);
        tmem_ld32(tS + 64, c);
        tmem_ld32(tS + 96, d);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          s[i] = __uint_as_float(a[i]);
          s[32 + i] = __uint_as_float(b[i]);
          s[64 + i] = __uint_as_float(c[i]);
          s[96 + i] = __uint_as_float(d[i]);
        }
      }
      // Element-wise mask only on the key-tail tile and the tiles the causal
      // boundary crosses (key > row + causal_off).
      const int a = wk.kv0 + j;  // absolute key tile
      const bool mask_tail = (a == Tk - 1) && (Nk & 127);
      const bool mask_diag = CAUSAL && (a * 128 + 127 > qt * rph + p.causal_off);
      if (mask_tail || mask_diag) {
        int lim_col = Nk - 1 - a * 128;
        if (CAUSAL) lim_col = min(lim_col, row + p.causal_off - a * 128);
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (i > lim_col) s[i] = -INFINITY;
      }
      // columns 0-7 seed four accumulators, then 8-127 two at a time each
      float mx0 = fmaxf(s[0], s[1]), mx1 = fmaxf(s[2], s[3]), mx2 = fmaxf(s[4], s[5]), mx3 = fmaxf(s[6], s[7]);
#pragma unroll
      for (int i = 8; i < 128; i += 8) {
        mx0 = fmax3(mx0, s[i], s[i + 1]);
        mx1 = fmax3(mx1, s[i + 2], s[i + 3]);
        mx2 = fmax3(mx2, s[i + 4], s[i + 5]);
        mx3 = fmax3(mx3, s[i + 6], s[i + 7]);
      }
      const float mx = fmax3(fmaxf(mx0, mx1), mx2, mx3);
      // m2 is the reference max the exponentials and both accumulators are
      // relative to. It moves to the running max only when some row of the
      // warp has outgrown it by more than kRescaleSlack (then O~ and l are
      // rescaled); otherwise P~ = 2^(S c - m2) <= 2^kRescaleSlack. Either way
      // O~ / l is the same in exact arithmetic.
      const float m_run = fmaxf(m2, mx * c2);
      const bool move = __any_sync(0xffffffffu, m_run > m2 + kRescaleSlack);
      const float m_ref = move ? m_run : m2;
      const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
      const float alpha = ex2_approx(m2 - m_use);  // 0 on the first block, 1 when the reference is kept
      const float neg = -m_use;
      float2 sum_a = make_float2(0.f, 0.f), sum_b = make_float2(0.f, 0.f);
      uint32_t pk0[32], pk1[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float2 x = ffma2_bcast(s[2 * i], s[2 * i + 1], c2, neg);
        const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
        if (i & 1) sum_b = fadd2(sum_b, e); else sum_a = fadd2(sum_a, e);
        pk0[i] = pack_bf16x2(e.x, e.y);
      }
      tmem_st32(tP, pk0);  // first 64 keys of P~: frees registers for the second half
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float2 x = ffma2_bcast(s[64 + 2 * i], s[64 + 2 * i + 1], c2, neg);
        const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
        if (i & 1) sum_b = fadd2(sum_b, e); else sum_a = fadd2(sum_a, e);
        pk1[i] = pack_bf16x2(e.x, e.y);
      }
      const float2 sum2 = fadd2(sum_a, sum_b);
      l = l * alpha + (sum2.x + sum2.y);
      tmem_st32(tP + 32, pk1);
      // Rescale O~ only when the reference max moved.
      if (j > 0 && move) {
#pragma unroll 1
        for (int c = 0; c < HD; c += 32) {
          uint32_t o[32];
          tmem_ld32(tO + c, o);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tO + c, o);
        }
      }
      m2 = m_ref;
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&sh.p_full[t]);
    }

    // Epilogue: wait for the last O~ += P~ V, normalise, store through the
    // (now free) Q_t smem; then hand O~_t and Q_t's smem back to the MMA and
    // load threads for the next item.
    const bool active = last_kv >= 0;
    if (alive && active) {
      alive = __all_sync(0xffffffffu, mbar_wait(&sh.pv_done[t], (cnt + last_kv) & 1, &sh.abort_flag, lim));
      if (!alive) record_timeout(p.status, &sh.abort_flag, WHERE_FWD_SOFTMAX);
    }
    tc_fence_after_sync();
    // A row that saw no key of this range (possible only when the keys are
    // split) has l = 0: its partial is O = 0, L = -inf, and the combine step
    // never reads it.
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    const float lse_row = l > 0.f ? (m2 + log2f(l)) * kLn2 : -INFINITY;
    if (alive && active && p.splits > 1) {
      // fp32 partial of this key range, straight from TMEM to the workspace
      float* dst = p.o_part + ((static_cast<size_t>(wk.s) * p.BH + head) * Nq + row) * HD;
#pragma unroll 1
      for (int c = 0; c < HD; c += 32) {
        uint32_t o[32];
        tmem_ld32(tO + c, o);
        tmem_ld_wait();
        if (c + 32 >= HD) {
          tc_fence_before_sync();
          mbar_arrive(&sh.o_free[t]);
        }
        if (row < Nq) {
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<float4*>(dst + c + 4 * u) =
                make_float4(__uint_as_float(o[4 * u]) * inv_l, __uint_as_float(o[4 * u + 1]) * inv_l,
                            __uint_as_float(o[4 * u + 2]) * inv_l, __uint_as_float(o[4 * u + 3]) * inv_l);
        }
      }
      if (row < Nq) p.lse_part[(static_cast<size_t>(wk.s) * p.BH + head) * Nq + row] = lse_row;
    } else if (alive && active) {
      const uint32_t stage_addr = smem_u32(stage);
#pragma unroll 1
      for (int c = 0; c < HD; c += 32) {
        uint32_t o[32];
        tmem_ld32(tO + c, o);
        tmem_ld_wait();
        if (c + 32 >= HD) {  // O~_t fully read: the next item's first PV may overwrite it
          tc_fence_before_sync();
          mbar_arrive(&sh.o_free[t]);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int col = c + u * 8;
          const uint32_t w0 = pack_bf16x2(__uint_as_float(o[u * 8 + 0]) * inv_l, __uint_as_float(o[u * 8 + 1]) * inv_l);
          const uint32_t w1 = pack_bf16x2(__uint_as_float(o[u * 8 + 2]) * inv_l, __uint_as_float(o[u * 8 + 3]) * inv_l);
          const uint32_t w2 = pack_bf16x2(__uint_as_float(o[u * 8 + 4]) * inv_l, __uint_as_float(o[u * 8 + 5]) * inv_l);
          const uint32_t w3 = pack_bf16x2(__uint_as_float(o[u * 8 + 6]) * inv_l, __uint_as_float(o[u * 8 + 7]) * inv_l);
          st_shared_v4(stage_addr + (col >> 6) * C::CHUNK_BYTES + sw128_offset(r, (col & 63) >> 3), w0, w1, w2, w3);
        }
      }
      fence_proxy_async_smem();
      if (row < Nq) p.lse[static_cast<size_t>(head) * Nq + row] = lse_row;
    } else {
      // No query tile in this slot: nothing waits for this warpgroup, so it
      // first waits for the item's Q load. That keeps its q_free / o_free
      // arrivals one item at a time (a warpgroup that ran two items ahead
      // would complete a phase the load thread has not waited for yet).
      if (alive) {
        alive = __all_sync(0xffffffffu, mbar_wait(&sh.q_full[t], items & 1, &sh.abort_flag, lim));
        if (!alive) record_timeout(p.status, &sh.abort_flag, WHERE_FWD_SOFTMAX);
      }
      mbar_arrive(&sh.o_free[t]);
    }
    named_barrier_sync(1 + t, 128);
    if (r == 0) {
      if (alive && active && p.splits == 1 && !*reinterpret_cast<volatile int*>(&sh.abort_flag)) {
#pragma unroll
        for (int c = 0; c < C::CHUNKS; ++c)
          tma_store_3d(&p.tmO, stage + c * C::CHUNK_BYTES, c * 64, qt * rph, wk.bh);
        tma_store_commit();
        tma_store_wait_read_all();  // the staging can be overwritten by the next Q tile
      }
      mbar_arrive(&sh.q_free[t]);
    }
    if (active) cnt += last_kv + 1;
    ++items;
  }
  if (r == 0) tma_store_wait_all();  // O stores complete before the CTA can exit
}

template <int HD, bool CAUSAL, bool PACK>
__global__ void __launch_bounds__(kThreads, 1) fa_fwd_kernel(const __grid_constant__ FwdLaunch p) {
  using C = FwdCfg<HD>;
  extern __shared__ uint8_t smem_dyn[];
  __shared__ FwdShared sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + C::NT * C::TILE_BYTES;
  uint8_t* sV = sK + C::KST * C::TILE_BYTES;
  const int warp = threadIdx.x >> 5;
  // Split key ranges: the combine kernel queued next may take SMs as this
  // grid's CTAs leave them (it waits for this grid before it reads).
  if (p.splits > 1) griddep_launch_dependents();

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) mbar_init(&sh.q_full[t], 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(&sh.k_full[i], 1);
      mbar_init(&sh.k_empty[i], 1);
      mbar_init(&sh.v_full[i], 1);
      mbar_init(&sh.v_empty[i], 1);
    }
    for (int t = 0; t < 2; ++t) {
      // test hook: slot 0's S or P barrier waits for one arrival too many
      mbar_init(&sh.s_full[t], 1 + (t == 0 ? debug_extra(p.debug_skip, WHERE_FWD_MMA) : 0u));
      mbar_init(&sh.p_full[t], 128 + (t == 0 ? debug_extra(p.debug_skip, WHERE_FWD_SOFTMAX) : 0u));
      mbar_init(&sh.pv_done[t], 1);
      mbar_init(&sh.o_free[t], 128);
      mbar_init(&sh.q_free[t], 1);
    }
    mbar_init(&sh.mma_drain, 1);
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
    if (lane_id() == 0) fwd_load_role<HD, CAUSAL, PACK>(p, sh, sQ, sK, sV);
  } else if (warp == kMmaWarp) {
    if (lane_id() == 0) fwd_mma_role<HD, CAUSAL, PACK>(p, sh, sQ, sK, sV, tmem);
  } else if (warp < 4 * C::NT) {
    fwd_softmax_role<HD, CAUSAL, PACK>(p, sh, sQ, tmem, warp >> 2);
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

template <int HD, bool CAUSAL, bool PACK>
cudaError_t launch_fwd_t(const FwdLaunch& a, cudaStream_t stream) {
  using C = FwdCfg<HD>;
  auto kern = fa_fwd_kernel<HD, CAUSAL, PACK>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int rph = PACK ? a.rph : 128;
  const int Tq = (a.Nq + rph - 1) / rph;
  const long long items = static_cast<long long>(a.BH / (PACK ? a.pack : 1)) * ((Tq + C::NT - 1) / C::NT) * a.splits;
  // Persistent: one CTA per SM (the smem footprint allows no more), each
  // looping over its share of the items.
  const long long grid = items < a.num_sms ? items : a.num_sms;
  kern<<<static_cast<unsigned>(grid), kThreads, C::SMEM_BYTES, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace
}  // namespace fa

// dQ of the backward pass without atomics at head dimension 256, for sm_103a.
//
// Method (web pages on FlashAttention-2): the reading note (papers.chlience.com)
// 5.3-5.4 and the paper-graph-ui summary, "The Backward Pass", accumulate
// dQ_i += dS_ij K_j across key blocks with atomic adds, so dQ is not bitwise
// reproducible. As in fa_bwd_dq.cu (d = 64, 128), one work item here owns
// query tile i of one head and loops over the key tiles itself, so dQ_i is
// summed on chip in key order:
//   S = Q_i K_j^T, P = 2^(S scale log2e - L_i log2e), dP = dO_i V_j^T,
//   dS = P o (dP - D_i) * scale, dQ_i += dS K_j,
// with L and D from the preprocess kernel; the d = 256 main kernel then runs
// without its dQ products (fa_bwd256.cu, DQ = false).
//
// GB300 mapping: persistent, one CTA (320 threads) per SM taking items
// (query head, 128-row query tile) from a counter in the workspace (causal:
// the tiles that see the most keys first). Queries sit on the TMEM lanes:
// thread r of either softmax warpgroup owns query row r, so L_r and D_r are
// per-thread scalars; warpgroup w owns key columns [64w, 64w + 64).
//   - Q_i and dO_i (64 KB each) stay in shared memory for the item. K_j and
//     V_j stream through a ring of six 16-KB chunks (128 keys x 64 columns)
//     in the order the MMAs read them: K_0, V_0, then per key tile t:
//     K_{t+1} (for S(t+1)), K_t again (for the dQ product), V_{t+1} (for
//     dP(t+1)). K is read twice from L2 instead of held: holding it for the
//     dQ product would need more shared memory than the ring. Each item
//     loads 12 chunks per key tile, so every K_t read by the dQ product
//     lands in an even-aligned pair of slots, which its two N = 128 halves
//     read as one MN-major operand each.
//   - TMEM: S [0, 128); dP [128, 256), into whose first 32 columns of each
//     warpgroup's half phase B writes dS (bf16), the A operand of the dQ
//     product; dQ [256, 512) (128 rows x 256 columns, fp32).
//   - MMA order: S(0), dP(0); per key tile t: S(t+1) once phase A(t) has
//     read S(t) (P stays in registers); dQ += dS(t) K_t once phase B(t) has
//     written dS(t); dP(t+1) once the dQ product has read dS(t). The tensor
//     core thus runs S(t+1) while the softmax works on tile t.
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

struct Dq256Cfg {
  static constexpr int HD = 256;
  static constexpr int CHUNK_BYTES = 128 * 128;      // [128 rows][64 columns] bf16
  static constexpr int TILE_BYTES = 4 * CHUNK_BYTES;  // 64 KB
  static constexpr int RING = 6;                      // K / V chunk slots
  static constexpr uint32_t S_COL = 0, DP_COL = 128, DQ_COL = 256;
  // smem: Q_i, dO_i, the chunk ring
  static constexpr int SMEM_BYTES = 2 * TILE_BYTES + RING * CHUNK_BYTES + 1024;
};

struct Dq256Shared {
  uint64_t q_full, q_free;
  uint64_t ring_full[Dq256Cfg::RING], ring_empty[Dq256Cfg::RING];
  uint64_t s_full, s_free, dp_full, ds_ready, dq_done, acc_done, acc_free;
  uint64_t mma_drain;  // the MMA thread's last commit: all its MMAs done before the CTA exits
  uint64_t item_full[kItemSlots], item_empty[kItemSlots];
  int item_ring[kItemSlots];
  uint32_t tmem_base;
  int abort_flag;
};

// Work item: query tile i of query head bh; key tiles 0 .. nkv-1 (causal:
// up to the diagonal). Causal items are numbered most-work-first; non-causal
// items of one head are adjacent (K/V reuse in L2).
template <bool CAUSAL>
struct Dq256Work {
  int bh, i, nkv;
  __device__ Dq256Work(int item, int BH, int N) {
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

// The chunk stream of one item, in the MMA's reading order: K_0 and V_0
// (4 chunks each), then per key tile t: K_{t+1}, K_t, V_{t+1} (the first and
// last only when t + 1 < nkv). 12 nkv chunks in all.
struct ChunkStream {
  int nkv;
  // (tensor 0 = K / 1 = V, key tile, column chunk) of chunk k of the stream
  __device__ void at(int k, int& tensor, int& tile, int& col) const {
    col = k & 3;
    const int group = k >> 2;  // groups of 4 chunks
    if (group < 2) {
      tensor = group;
      tile = 0;
      return;
    }
    const int t = (group - 2) / 3, part = (group - 2) % 3;
    if (t == nkv - 1) {  // the last key tile has only the dQ product's K_t
      tensor = 0;
      tile = t;
      return;
    }
    tensor = part == 2 ? 1 : 0;
    tile = part == 1 ? t : t + 1;
  }
  __device__ int count() const { return 12 * nkv; }
};

// TMA producer (one thread): per item K_0, then Q_i and dO_i once the
// previous item's last S and dP products have read theirs, then the rest of
// the chunk stream through the ring.
template <bool CAUSAL>
__device__ void dq256_load_role(const BwdLaunch& p, Dq256Shared& sh, uint8_t* sQ, uint8_t* sdO, uint8_t* sRing) {
  using C = Dq256Cfg;
  tma_prefetch_desc(&p.tmQ);
  tma_prefetch_desc(&p.tmdO);
  tma_prefetch_desc(&p.tmK);
  tma_prefetch_desc(&p.tmV);
  const int T = (p.N + 127) / 128;
  const int total = p.BH * T;
  const uint64_t lim = p.wait_limit_ns;
  int u = 0, pos = 0, q_issued = 0;  // pos: ring chunks issued
  bool aborted = false;
  auto load_chunk = [&](const ChunkStream& cs, int k, int kvh) -> bool {
    int tensor, tile, col;
    cs.at(k, tensor, tile, col);
    const int s = pos % C::RING;
    if (pos >= C::RING && !mbar_wait(&sh.ring_empty[s], ((pos / C::RING) - 1) & 1, &sh.abort_flag, lim)) return false;
    mbar_arrive_expect_tx(&sh.ring_full[s], C::CHUNK_BYTES);
    tma_load_3d(sRing + s * C::CHUNK_BYTES, tensor == 0 ? &p.tmK : &p.tmV, &sh.ring_full[s], col * 64, tile * 128, kvh);
    ++pos;
    return true;
  };
  int item = blockIdx.x;  // the grid never exceeds the item count
  while (!aborted) {
    if (!publish_item(sh, u, item, lim)) {
      aborted = true;
      break;
    }
    if (item >= total) break;
    const Dq256Work<CAUSAL> wk(item, p.BH, p.N);
    const int kvh = wk.bh / p.group;  // grouped K/V heads
    const ChunkStream cs{wk.nkv};
    const int n = cs.count();
    int k = 0;
    // K_0 loads while the previous item still reads Q_i, dO_i. V_0 follows
    // Q_i: its last chunks wait for S(0) to free ring slots, and S(0) needs Q_i.
    for (; k < 4 && !aborted; ++k) aborted = !load_chunk(cs, k, kvh);
    if (aborted || (u > 0 && !mbar_wait(&sh.q_free, (u - 1) & 1, &sh.abort_flag, lim))) {
      aborted = true;
      break;
    }
    if (!debug_skip_here(p.debug_skip, WHERE_BWD_LOAD, u == 0)) {  // test hook
      // The Q and dO maps have 64-row boxes (the main kernel's query tiles):
      // two boxes fill one 128-row chunk, in the same swizzled layout.
      mbar_arrive_expect_tx(&sh.q_full, 2 * C::TILE_BYTES);
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const uint32_t off = c * C::CHUNK_BYTES + hh * (C::CHUNK_BYTES / 2);
          tma_load_3d(sQ + off, &p.tmQ, &sh.q_full, c * 64, wk.i * 128 + 64 * hh, wk.bh);
          tma_load_3d(sdO + off, &p.tmdO, &sh.q_full, c * 64, wk.i * 128 + 64 * hh, wk.bh);
        }
      ++q_issued;
    }
    for (; k < n && !aborted; ++k) aborted = !load_chunk(cs, k, kvh);
    if (aborted) break;
    ++u;
    item = claim_item(p.sched + 2);
  }
  finish_claiming(p.sched + 2);
  if (aborted) record_timeout(p.status, &sh.abort_flag, WHERE_BWD_LOAD);
  // The copies already issued land before the CTA can exit (after an abort
  // no consumer may wait for them): the latest phase of each ring slot.
  for (int k = std::max(0, pos - C::RING); k < pos; ++k) drain_wait(&sh.ring_full[k % C::RING], (k / C::RING) & 1, lim);
  if (q_issued > 0) drain_wait(&sh.q_full, (q_issued - 1) & 1, lim);
}

// One thread issues every MMA (order in the file header).
template <bool CAUSAL>
__device__ void dq256_mma_role(const BwdLaunch& p, Dq256Shared& sh, uint8_t* sQ, uint8_t* sdO, uint8_t* sRing,
                               uint32_t tmem) {
  using C = Dq256Cfg;
  constexpr uint32_t kIdescSq = make_idesc_bf16_f32(128, 128, false, false);  // S, dP: A, B K-major
  constexpr uint32_t kIdescDq = make_idesc_bf16_f32(128, 128, false, true);   // A = dS (TMEM), B = K MN-major
  const uint32_t q_addr = smem_u32(sQ), do_addr = smem_u32(sdO), ring_addr = smem_u32(sRing);
  const uint64_t lim = p.wait_limit_ns;
  const int T = (p.N + 127) / 128;
  const int total = p.BH * T;
  auto fail = [&]() {
    record_timeout(p.status, &sh.abort_flag, WHERE_BWD_MMA);
    drain_mmas(&sh.mma_drain, lim);
  };
  int pos = 0;  // ring chunks consumed
  auto wait_chunk = [&](int k) -> bool {
    return mbar_wait(&sh.ring_full[k % C::RING], (k / C::RING) & 1, &sh.abort_flag, lim);
  };
  auto slot_addr = [&](int k) -> uint32_t { return ring_addr + (k % C::RING) * C::CHUNK_BYTES; };
  // D = A (128 x 256 resident, K-major) * (4 ring chunks, K-major)^T; each
  // chunk's slot is released once the product has read it
  auto issue_sq = [&](uint32_t d_col, uint32_t a_addr) -> bool {
#pragma unroll 1
    for (int c = 0; c < 4; ++c, ++pos) {
      if (!wait_chunk(pos)) return false;
      tc_fence_after_sync();
      const uint64_t ad = make_smem_desc_sw128(a_addr + c * C::CHUNK_BYTES, 16, 1024);
      const uint64_t bd = make_smem_desc_sw128(slot_addr(pos), 16, 1024);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_ss(tmem + d_col, desc_add(ad, ks * 32), desc_add(bd, ks * 32), kIdescSq, (c > 0 || ks > 0) ? 1u : 0u);
      umma_commit(&sh.ring_empty[pos % C::RING]);
    }
    return true;
  };
  // dQ += dS K_t: two N = 128 halves of the head dimension, each reading an
  // even-aligned pair of ring chunks as one MN-major B operand.
  auto issue_dq = [&](bool first) -> bool {
#pragma unroll 1
    for (int half = 0; half < 2; ++half, pos += 2) {
      if (!wait_chunk(pos) || !wait_chunk(pos + 1)) return false;
      tc_fence_after_sync();
      const uint64_t kd = make_smem_desc_sw128(slot_addr(pos), C::CHUNK_BYTES, 1024);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma_ts(tmem + C::DQ_COL + 128 * half, tmem + C::DP_COL + (ks >> 2) * 64 + (ks & 3) * 8,
                desc_add(kd, ks * 2048), kIdescDq, (!first || ks > 0) ? 1u : 0u);
      umma_commit(&sh.ring_empty[pos % C::RING]);
      umma_commit(&sh.ring_empty[(pos + 1) % C::RING]);
    }
    return true;
  };

  int u = 0, t = 0;  // items, key tiles (global)
  while (true) {
    const int item = take_item(sh, u, lim);
    if (item < 0) return fail();
    if (item >= total) break;
    const Dq256Work<CAUSAL> wk(item, p.BH, p.N);
    if (!mbar_wait(&sh.q_full, u & 1, &sh.abort_flag, lim)) return fail();
    // S(first): the previous item's last dQ product has read dS from the dP
    // columns, and phase A read its S, before that product was issued.
    if (t > 0 && !mbar_wait(&sh.s_free, (t - 1) & 1, &sh.abort_flag, lim)) return fail();
    tc_fence_after_sync();
    if (!issue_sq(C::S_COL, q_addr)) return fail();
    umma_commit(&sh.s_full);
    // dP(first) overwrites the previous item's last dS: its dQ product is done
    if (t > 0 && !mbar_wait(&sh.dq_done, (t - 1) & 1, &sh.abort_flag, lim)) return fail();
    tc_fence_after_sync();
    if (!issue_sq(C::DP_COL, do_addr)) return fail();
    umma_commit(&sh.dp_full);
    if (wk.nkv == 1) umma_commit(&sh.q_free);
    for (int j = 0; j < wk.nkv; ++j, ++t) {
      const bool has_next = j + 1 < wk.nkv;
      if (has_next) {
        // S(t+1) once phase A(t) has read S(t)
        if (!mbar_wait(&sh.s_free, t & 1, &sh.abort_flag, lim)) return fail();
        tc_fence_after_sync();
        if (!issue_sq(C::S_COL, q_addr)) return fail();
        umma_commit(&sh.s_full);
      }
      if (!mbar_wait(&sh.ds_ready, t & 1, &sh.abort_flag, lim)) return fail();
      // the first dQ product of an item overwrites the accumulator: the
      // previous item's epilogue must have read it
      if (j == 0 && u > 0 && !mbar_wait(&sh.acc_free, (u - 1) & 1, &sh.abort_flag, lim)) return fail();
      tc_fence_after_sync();
      if (!issue_dq(j == 0)) return fail();
      umma_commit(&sh.dq_done);
      if (has_next) {
        // dP(t+1) overwrites dS(t): wait for the dQ product to have read it
        if (!mbar_wait(&sh.dq_done, t & 1, &sh.abort_flag, lim)) return fail();
        tc_fence_after_sync();
        if (!issue_sq(C::DP_COL, do_addr)) return fail();
        umma_commit(&sh.dp_full);
        if (j + 2 == wk.nkv) umma_commit(&sh.q_free);  // the item's last S and dP are issued
      }
    }
    umma_commit(&sh.acc_done);
    ++u;
  }
  // Normally the epilogues have waited for the last products; if a softmax
  // warpgroup gave up, nothing has.
  drain_mmas(&sh.mma_drain, lim);
}

// Warpgroup w owns key columns [64w, 64w + 64) of every key tile; thread r
// owns query row r. Phase A: P = 2^(S scale log2e - L2_r) (bf16-rounded,
// kept in registers). Phase B: dS = P o (dP scale - D_r scale) into the dP
// columns. At the end of an item warpgroup w writes dQ columns
// [128w, 128w + 128).
template <bool CAUSAL>
__device__ void dq256_softmax_role(const BwdLaunch& p, Dq256Shared& sh, uint32_t tmem, int w) {
  using C = Dq256Cfg;
  const int r = threadIdx.x & 127;
  const uint32_t lane_base = static_cast<uint32_t>((threadIdx.x >> 5) & 3) << 21;
  const float c2 = p.scale_log2;
  const float sc = p.scale;
  const uint64_t lim = p.wait_limit_ns;
  const uint32_t tS = tmem + lane_base + C::S_COL + 64 * w;
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
    const Dq256Work<CAUSAL> wk(item, p.BH, p.N);
    const int row = wk.i * 128 + r;
    const size_t srow = static_cast<size_t>(wk.bh) * p.Npad + row;
    const float l2 = __ldg(p.lse2 + srow);  // +inf on padding rows: their P is 0
    const float dsc = __ldg(p.D + srow) * sc;
    for (int j = 0; j < wk.nkv; ++j, ++t) {
      // ---- phase A: P of this warpgroup's 64 keys; S is released once read
      wait_all(&sh.s_full, t & 1, WHERE_BWD_SOFTMAX);
      float pv[64];
      if (alive) {
        uint32_t a[32], b[32];
        tmem_ld32(tS, a);
        tmem_ld32(tS + 32, b);
        tmem_ld_wait();
        tc_fence_before_sync();
        mbar_arrive(&sh.s_free);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          pv[c] = __uint_as_float(a[c]);
          pv[32 + c] = __uint_as_float(b[c]);
        }
        // key 128j + 64w + c is seen if it is < N and (causal) <= the query row
        const int kbase = j * 128 + 64 * w;
        int c_hi = min(64, p.N - kbase);
        if (CAUSAL && j == wk.i) c_hi = min(c_hi, row - kbase + 1);
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
      // ---- phase B: dS into the first 32 columns of this warpgroup's half
      // of the dP columns (already read)
      wait_all(&sh.dp_full, t & 1, WHERE_BWD_SOFTMAX);
      if (alive) {
        uint32_t ds[32];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          uint32_t dpv[32];
          tmem_ld32(tDP + 32 * h2, dpv);
          tmem_ld_wait();
#pragma unroll
          for (int c4 = 0; c4 < 32; c4 += 4) {
            const float2 p01 = unpack_bf16x2(pk[16 * h2 + c4 / 2]);
            const float2 p23 = unpack_bf16x2(pk[16 * h2 + c4 / 2 + 1]);
            const float2 g01 = ffma2_bcast(__uint_as_float(dpv[c4]), __uint_as_float(dpv[c4 + 1]), sc, -dsc);
            const float2 g23 = ffma2_bcast(__uint_as_float(dpv[c4 + 2]), __uint_as_float(dpv[c4 + 3]), sc, -dsc);
            const float2 d01 = fmul2(p01, g01);
            const float2 d23 = fmul2(p23, g23);
            ds[16 * h2 + c4 / 2] = pack_bf16x2(d01.x, d01.y);
            ds[16 * h2 + c4 / 2 + 1] = pack_bf16x2(d23.x, d23.y);
          }
        }
        tmem_st32(tDP, ds);
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(&sh.ds_ready);
      }
    }
    const int item_next = next_item(u + 1);
    // ---- epilogue: dQ (fp32, TMEM) -> bf16 -> dq; rows past N are skipped
    wait_all(&sh.acc_done, u & 1, WHERE_BWD_SOFTMAX);
    if (alive) {
      const uint32_t tq = tmem + lane_base + C::DQ_COL + w * 128;
      __nv_bfloat16* dst = p.dq + (static_cast<size_t>(wk.bh) * p.N + row) * C::HD + w * 128;
#pragma unroll 1
      for (int c = 0; c < 128; c += 32) {
        uint32_t v[32];
        tmem_ld32(tq + c, v);
        tmem_ld_wait();
        if (c + 32 == 128) {  // the next item may overwrite the accumulator
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

template <bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1) fa_bwd_dq256_kernel(const __grid_constant__ BwdLaunch p) {
  using C = Dq256Cfg;
  extern __shared__ uint8_t smem_dyn[];
  __shared__ Dq256Shared sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sdO = sQ + C::TILE_BYTES;
  uint8_t* sRing = sdO + C::TILE_BYTES;
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    mbar_init(&sh.q_full, 1);
    mbar_init(&sh.q_free, 1);
    for (int s = 0; s < C::RING; ++s) {
      mbar_init(&sh.ring_full[s], 1);
      mbar_init(&sh.ring_empty[s], 1);
    }
    // test hook: the S or dS barrier waits for one arrival too many
    mbar_init(&sh.s_full, 1 + debug_extra(p.debug_skip, WHERE_BWD_MMA));
    mbar_init(&sh.s_free, 256);
    mbar_init(&sh.dp_full, 1);
    mbar_init(&sh.ds_ready, 256 + debug_extra(p.debug_skip, WHERE_BWD_SOFTMAX));
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
    if (lane_id() == 0) dq256_load_role<CAUSAL>(p, sh, sQ, sdO, sRing);
  } else if (warp == kMmaWarp) {
    if (lane_id() == 0) dq256_mma_role<CAUSAL>(p, sh, sQ, sdO, sRing, tmem);
  } else {
    dq256_softmax_role<CAUSAL>(p, sh, tmem, warp >> 2);
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
  // Launched to overlap the dK/dV pass (overlap_prev), this grid must not
  // complete before that pass has: work queued after it may read dK and dV.
  if (threadIdx.x == 0) griddep_wait();
}

template <bool CAUSAL>
cudaError_t launch_t(const BwdLaunch& a, cudaStream_t stream) {
  using C = Dq256Cfg;
  auto kern = fa_bwd_dq256_kernel<CAUSAL>;
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

cudaError_t launch_bwd_dq256(const BwdLaunch& a, cudaStream_t stream) {
  return a.causal ? launch_t<true>(a, stream) : launch_t<false>(a, stream);
}

}  // namespace fa

// Backward main kernel for head dimension 256 on sm_103a.
//
// Same method as fa_bwd.cu (reading note 5.3; paper-graph-ui summary, "The
// Backward Pass": key blocks outer, recompute S and P = exp(S - L), dV += P^T
// dO, dP = dO V^T, dS = P o (dP - D), dK += dS^T Q, dQ += dS K with atomic
// adds), with a different split because at d = 256 the fp32 dK and dV of one
// 128-key tile alone would fill all 512 TMEM columns, and the bf16 K, V, Q
// and dO tiles alone would fill shared memory:
//   - Two CTAs per 128-key tile j: CTA h accumulates columns [128h, 128h+128)
//     of dK_j and dV_j and adds columns [128h, 128h+128) of every dQ_i. Both
//     recompute S^T and dP^T over the full head dimension.
//   - Query tiles have 64 rows, and each is loaded once (one stage): K_j, V_j
//     (64 KB each), Q_i, dO_i (32 KB each) and dS^T (16 KB) fill the smem.
// TMEM columns (512 allocated): dK half [0, 128), dV half [128, 256),
// S^T then P^T [256, 320), dP^T [320, 384), dQ half transposed [384, 448)
// (head-dim columns on the lanes, so each warp's reductions cover whole
// 128-byte lines).
// Warpgroup w (w = 0, 1) owns query columns [32w, 32w + 32) of each tile;
// thread r owns key r (phases A, B) and head-dim column 128h + r (dQ drain).
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

struct Cfg256 {
  static constexpr int HD = 256;
  static constexpr int BQ = 64;                        // query rows per tile
  static constexpr int KV_CHUNK = 128 * 128;           // [128 keys][64 d] bf16
  static constexpr int KV_BYTES = 4 * KV_CHUNK;        // 64 KB
  static constexpr int Q_CHUNK = BQ * 128;             // [64 rows][64 d] bf16
  static constexpr int Q_BYTES = 4 * Q_CHUNK;          // 32 KB
  static constexpr int DS_BYTES = 128 * BQ * 2;        // [128 keys][64 queries] bf16
  static constexpr int LD_BYTES = 2 * 64 * 4;          // per warpgroup: 32 L2 + 32 D
  static constexpr uint32_t DK_COL = 0, DV_COL = 128, REG_S = 256, REG_DP = 320, REG_DQ = 384;
  static constexpr int SMEM_BYTES = 2 * KV_BYTES + 2 * Q_BYTES + DS_BYTES + LD_BYTES + 1024;
};

struct Shared256 {
  uint64_t kv_full, q_full, q_empty, do_full, do_empty;
  uint64_t s_full, dp_full, pa_ready, ds_ready, pv_done, dq_full, dq_free, acc_done;
  uint64_t mma_drain;  // the MMA thread's last commit: all its MMAs done before the CTA exits
  uint32_t tmem_base;
  int abort_flag;
};

// Key tile j of K/V head bh, half h of the head dimension. The query stream
// is, for each of the g query heads that share this K/V head (query head
// bh*g + t), 64-row query tiles i0..T64-1 (causal: i0 = 2j).
template <bool CAUSAL>
struct Work256 {
  int bh, j, h, i0, T64, nq, g;
  __device__ Work256(int block, int BHkv, int N, int group) {
    const int T = (N + 127) / 128;
    T64 = (N + 63) / 64;
    if (CAUSAL) {  // key tiles with the most query tiles first
      j = block / (2 * BHkv);
      const int rem = block % (2 * BHkv);
      bh = rem >> 1;
      h = rem & 1;
    } else {
      bh = block / (2 * T);
      const int rem = block % (2 * T);
      j = rem >> 1;
      h = rem & 1;
    }
    i0 = CAUSAL ? 2 * j : 0;
    nq = T64 - i0;
    g = group;
  }
  __device__ int n_iter() const { return g * nq; }
  // (query head, 64-row query tile) of a step, advanced in order
  struct Pos {
    int bh, i;
  };
  __device__ Pos first() const { return Pos{bh * g, i0}; }
  __device__ void advance(Pos& p) const {
    if (++p.i == T64) {
      p.i = i0;
      ++p.bh;
    }
  }
};

template <bool CAUSAL>
__device__ void load_role(const BwdLaunch& p, Shared256& sh, uint8_t* sK, uint8_t* sV, uint8_t* sQ, uint8_t* sdO,
                          const Work256<CAUSAL>& wk) {
  using C = Cfg256;
  tma_prefetch_desc(&p.tmQ);
  tma_prefetch_desc(&p.tmK);
  tma_prefetch_desc(&p.tmV);
  tma_prefetch_desc(&p.tmdO);
  mbar_arrive_expect_tx(&sh.kv_full, 2 * C::KV_BYTES);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    tma_load_3d(sK + c * C::KV_CHUNK, &p.tmK, &sh.kv_full, c * 64, wk.j * 128, wk.bh);
    tma_load_3d(sV + c * C::KV_CHUNK, &p.tmV, &sh.kv_full, c * 64, wk.j * 128, wk.bh);
  }
  const int n_iter = wk.n_iter();
  int q_issued = 0, do_issued = 0;
  bool aborted = false;
  typename Work256<CAUSAL>::Pos pos = wk.first();
  for (int n = 0; n < n_iter && !aborted; ++n, wk.advance(pos)) {
    const int i = pos.i, qbh = pos.bh;
    if (n > 0 && !mbar_wait(&sh.q_empty, (n - 1) & 1, &sh.abort_flag, p.wait_limit_ns)) {
      aborted = true;
      break;
    }
    mbar_arrive_expect_tx(&sh.q_full, C::Q_BYTES);
#pragma unroll
    for (int c = 0; c < 4; ++c) tma_load_3d(sQ + c * C::Q_CHUNK, &p.tmQ, &sh.q_full, c * 64, i * C::BQ, qbh);
    ++q_issued;
    if (n > 0 && !mbar_wait(&sh.do_empty, (n - 1) & 1, &sh.abort_flag, p.wait_limit_ns)) {
      aborted = true;
      break;
    }
    mbar_arrive_expect_tx(&sh.do_full, C::Q_BYTES);
#pragma unroll
    for (int c = 0; c < 4; ++c) tma_load_3d(sdO + c * C::Q_CHUNK, &p.tmdO, &sh.do_full, c * 64, i * C::BQ, qbh);
    ++do_issued;
  }
  if (aborted) record_timeout(p.status, &sh.abort_flag, WHERE_BWD_LOAD);
  // The copies already issued land before the CTA can exit.
  if (q_issued > 0) drain_wait(&sh.q_full, (q_issued - 1) & 1, p.wait_limit_ns);
  if (do_issued > 0) drain_wait(&sh.do_full, (do_issued - 1) & 1, p.wait_limit_ns);
  drain_wait(&sh.kv_full, 0, p.wait_limit_ns);
}

template <bool CAUSAL>
__device__ void mma_role(const BwdLaunch& p, Shared256& sh, uint8_t* sK, uint8_t* sV, uint8_t* sQ, uint8_t* sdO,
                         uint8_t* sDS, uint32_t tmem, const Work256<CAUSAL>& wk) {
  using C = Cfg256;
  constexpr uint32_t kIdescS = make_idesc_bf16_f32(128, 64, false, false);  // S^T, dP^T: 128 keys x 64 queries
  constexpr uint32_t kIdescAcc = make_idesc_bf16_f32(128, 128, false, true);  // dV, dK halves
  constexpr uint32_t kIdescDq = make_idesc_bf16_f32(128, 64, true, true);     // dQ^T half: 128 d x 64 queries
  const uint32_t k_addr = smem_u32(sK), v_addr = smem_u32(sV), q_addr = smem_u32(sQ), do_addr = smem_u32(sdO),
                 ds_addr = smem_u32(sDS);
  const uint64_t lim = p.wait_limit_ns;
  const int n_iter = wk.n_iter();
  auto fail = [&]() {
    record_timeout(p.status, &sh.abort_flag, WHERE_BWD_MMA);
    drain_mmas(&sh.mma_drain, lim);
  };

  // D = A (128 x 256, K-major) * B (64 x 256, K-major)^T
  auto issue_sq = [&](uint32_t d_col, uint32_t a_addr, uint32_t b_addr) {
#pragma unroll
    for (int ks = 0; ks < 16; ++ks) {
      const uint32_t koff = (ks & 3) * 32;
      umma_ss(tmem + d_col, make_smem_desc_sw128(a_addr + (ks >> 2) * C::KV_CHUNK + koff, 16, 1024),
              make_smem_desc_sw128(b_addr + (ks >> 2) * C::Q_CHUNK + koff, 16, 1024), kIdescS, ks > 0 ? 1u : 0u);
    }
  };

  if (!mbar_wait(&sh.kv_full, 0, &sh.abort_flag, lim)) return fail();
  for (int n = 0; n < n_iter; ++n) {
    const uint32_t par = n & 1;
    if (!mbar_wait(&sh.q_full, par, &sh.abort_flag, lim)) return fail();
    if (n > 0 && !mbar_wait(&sh.pv_done, (n - 1) & 1, &sh.abort_flag, lim)) return fail();
    tc_fence_after_sync();
    issue_sq(C::REG_S, k_addr, q_addr);  // S^T(n), over P^T(n-1) once dV(n-1) is done
    umma_commit(&sh.s_full);
    if (!mbar_wait(&sh.do_full, par, &sh.abort_flag, lim)) return fail();
    tc_fence_after_sync();
    issue_sq(C::REG_DP, v_addr, do_addr);  // dP^T(n); phase B(n-1) finished reading dP^T(n-1)
    umma_commit(&sh.dp_full);
    if (!mbar_wait(&sh.pa_ready, par, &sh.abort_flag, lim)) return fail();
    tc_fence_after_sync();
    // dV half += P^T dO_i[:, 128h : 128h + 128]; P^T in columns [0,16) and [32,48) of REG_S
    const uint32_t do_half = do_addr + 2 * wk.h * C::Q_CHUNK;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      umma_ts(tmem + C::DV_COL, tmem + C::REG_S + (ks >> 1) * 32 + (ks & 1) * 8,
              make_smem_desc_sw128(do_half + ks * 2048, C::Q_CHUNK, 1024), kIdescAcc, (n > 0 || ks > 0) ? 1u : 0u);
    umma_commit(&sh.pv_done);
    umma_commit(&sh.do_empty);
    if (!mbar_wait(&sh.ds_ready, par, &sh.abort_flag, lim)) return fail();
    tc_fence_after_sync();
    // dK half += dS^T Q_i[:, 128h : 128h + 128]
    const uint32_t q_half = q_addr + 2 * wk.h * C::Q_CHUNK;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      umma_ss(tmem + C::DK_COL, make_smem_desc_sw128(ds_addr + ks * 32, 16, 1024),
              make_smem_desc_sw128(q_half + ks * 2048, C::Q_CHUNK, 1024), kIdescAcc, (n > 0 || ks > 0) ? 1u : 0u);
    umma_commit(&sh.q_empty);
    // dQ half^T = K_j[:, 128h : 128h + 128]^T dS^T, once the previous one was drained
    if (n > 0 && !mbar_wait(&sh.dq_free, (n - 1) & 1, &sh.abort_flag, lim)) return fail();
    tc_fence_after_sync();
    const uint32_t k_half = k_addr + 2 * wk.h * C::KV_CHUNK;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      umma_ss(tmem + C::REG_DQ, make_smem_desc_sw128(k_half + ks * 2048, C::KV_CHUNK, 1024),
              make_smem_desc_sw128(ds_addr + ks * 2048, C::DS_BYTES, 1024), kIdescDq, ks > 0 ? 1u : 0u);
    umma_commit(&sh.dq_full);
  }
  umma_commit(&sh.acc_done);
  drain_mmas(&sh.mma_drain, lim);  // if a softmax warpgroup gave up, nothing waits for the last products
}

template <bool CAUSAL>
__device__ void softmax_role(const BwdLaunch& p, Shared256& sh, uint8_t* sDS, float* sLD, uint32_t tmem, int w,
                             const Work256<CAUSAL>& wk) {
  using C = Cfg256;
  const int r = threadIdx.x & 127;
  const uint32_t lane_base = static_cast<uint32_t>((threadIdx.x >> 5) & 3) << 21;
  const int key = wk.j * 128 + r;
  const bool key_valid = key < p.N;
  const float c2 = p.scale_log2;
  const float sc = p.scale;
  const uint64_t lim = p.wait_limit_ns;
  float* ld_l2 = sLD + w * 64;
  float* ld_d = ld_l2 + 32;
  const int n_iter = wk.n_iter();
  const uint32_t bar_id = 1 + w;
  bool alive = true;

  // thread r < 32 holds L2 of query 32w + r of a step's tile, 32 <= r < 64 its scaled D
  auto fetch_ld = [&](const typename Work256<CAUSAL>::Pos& q) -> float {
    const size_t row = static_cast<size_t>(q.bh) * p.Npad + q.i * C::BQ + 32 * w;
    if (r < 32) return __ldg(p.lse2 + row + r);
    if (r < 64) return __ldg(p.D + row + (r - 32)) * sc;
    return 0.f;
  };
  typename Work256<CAUSAL>::Pos cur = wk.first();
  {
    const float v = fetch_ld(cur);
    if (r < 64) sLD[w * 64 + r] = v;
    named_barrier_sync(bar_id, 128);
  }

  for (int n = 0; n < n_iter; ++n) {
    const int i = cur.i;
    const bool has_next = n + 1 < n_iter;
    typename Work256<CAUSAL>::Pos nxt = cur;
    wk.advance(nxt);
    const float next_ld = has_next ? fetch_ld(nxt) : 0.f;
    const uint32_t tS = tmem + lane_base + C::REG_S + 32 * w;
    const uint32_t tDP = tmem + lane_base + C::REG_DP + 32 * w;
    // ---- phase A: P^T for this warpgroup's 32 queries, bf16 back into TMEM
    alive = alive && __all_sync(0xffffffffu, mbar_wait(&sh.s_full, n & 1, &sh.abort_flag, lim));
    if (!alive) record_timeout(p.status, &sh.abort_flag, WHERE_BWD_SOFTMAX);
    tc_fence_after_sync();
    float pv[32];
    if (alive) {
      uint32_t a[32];
      tmem_ld32(tS, a);
      tmem_ld_wait();
      // causal: query 64i + 32w + c sees key 128j + r only if it is not smaller
      const int c_lo = CAUSAL ? wk.j * 128 + r - i * C::BQ - 32 * w : 0;
      uint32_t pk[16];
#pragma unroll
      for (int c4 = 0; c4 < 32; c4 += 4) {
        const float4 l = *reinterpret_cast<const float4*>(ld_l2 + c4);
        const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = c4 + u;
          float e = ex2_approx(fmaf(__uint_as_float(a[c]), c2, -lv[u]));
          if (!key_valid || c < c_lo) e = 0.f;
          pv[c] = e;
        }
        pk[c4 / 2] = pack_bf16x2(pv[c4], pv[c4 + 1]);
        pk[c4 / 2 + 1] = pack_bf16x2(pv[c4 + 2], pv[c4 + 3]);
      }
      tmem_st16(tS, pk);  // columns [32w, 32w + 16): already read
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&sh.pa_ready);
    }
    // ---- phase B: dS^T = P^T o (dP^T - D) * scale -> smem row r, queries [32w, 32w + 32)
    alive = alive && __all_sync(0xffffffffu, mbar_wait(&sh.dp_full, n & 1, &sh.abort_flag, lim));
    if (!alive) record_timeout(p.status, &sh.abort_flag, WHERE_BWD_SOFTMAX);
    tc_fence_after_sync();
    if (alive) {
      uint32_t dpv[32];
      tmem_ld32(tDP, dpv);
      tmem_ld_wait();
      uint32_t dk[16];
#pragma unroll
      for (int c4 = 0; c4 < 32; c4 += 4) {
        const float4 dd = *reinterpret_cast<const float4*>(ld_d + c4);
        const float dv4[4] = {dd.x, dd.y, dd.z, dd.w};
        float ds[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) ds[u] = pv[c4 + u] * fmaf(__uint_as_float(dpv[c4 + u]), sc, -dv4[u]);
        dk[c4 / 2] = pack_bf16x2(ds[0], ds[1]);
        dk[c4 / 2 + 1] = pack_bf16x2(ds[2], ds[3]);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        st_shared_v4(smem_u32(sDS) + sw128_offset(r, 4 * w + u), dk[4 * u], dk[4 * u + 1], dk[4 * u + 2],
                     dk[4 * u + 3]);
      fence_proxy_async_smem();
      tc_fence_before_sync();
      mbar_arrive(&sh.ds_ready);
    }
    // ---- dQ drain: lane r = head-dim column 128h + r, this warpgroup's 32 queries
    alive = alive && __all_sync(0xffffffffu, mbar_wait(&sh.dq_full, n & 1, &sh.abort_flag, lim));
    if (!alive) record_timeout(p.status, &sh.abort_flag, WHERE_BWD_DQ);
    tc_fence_after_sync();
    if (alive) {
      uint32_t v[32];
      tmem_ld32(tmem + lane_base + C::REG_DQ + 32 * w, v);
      tmem_ld_wait();
      tc_fence_before_sync();
      mbar_arrive(&sh.dq_free);
      float* dst = p.dq_acc + (static_cast<size_t>(cur.bh) * p.Npad + i * C::BQ + 32 * w) * C::HD + 128 * wk.h + r;
#pragma unroll
      for (int c = 0; c < 32; ++c) red_add_f32(dst + static_cast<size_t>(c) * C::HD, __uint_as_float(v[c]));
    }
    if (has_next) {
      named_barrier_sync(bar_id, 128);  // this tile's L2 / D are no longer read
      if (r < 64) sLD[w * 64 + r] = next_ld;
      named_barrier_sync(bar_id, 128);
    }
    cur = nxt;
  }
}

// Warpgroup 0 stores the dK half, warpgroup 1 the dV half (bf16 via smem
// over the first half of K_j / V_j, then TMA).
template <bool CAUSAL>
__device__ void epilogue(const BwdLaunch& p, Shared256& sh, uint8_t* sK, uint8_t* sV, uint32_t tmem, int w,
                         const Work256<CAUSAL>& wk) {
  using C = Cfg256;
  const int r = threadIdx.x & 127;
  const uint32_t lane_base = static_cast<uint32_t>((threadIdx.x >> 5) & 3) << 21;
  bool ok = !*reinterpret_cast<volatile int*>(&sh.abort_flag);
  if (ok) {
    ok = __all_sync(0xffffffffu, mbar_wait(&sh.acc_done, 0, &sh.abort_flag, p.wait_limit_ns));
    if (!ok) record_timeout(p.status, &sh.abort_flag, WHERE_BWD_SOFTMAX);
  }
  tc_fence_after_sync();
  uint8_t* stage = w == 0 ? sK : sV;
  if (ok) {
    const uint32_t t = tmem + lane_base + (w == 0 ? C::DK_COL : C::DV_COL);
    const uint32_t st = smem_u32(stage);
#pragma unroll 1
    for (int c = 0; c < 128; c += 32) {
      uint32_t v[32];
      tmem_ld32(t + c, v);
      tmem_ld_wait();
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int col = c + u * 8;
        st_shared_v4(st + (col >> 6) * C::KV_CHUNK + sw128_offset(r, (col & 63) >> 3),
                     pack_bf16x2(__uint_as_float(v[u * 8 + 0]), __uint_as_float(v[u * 8 + 1])),
                     pack_bf16x2(__uint_as_float(v[u * 8 + 2]), __uint_as_float(v[u * 8 + 3])),
                     pack_bf16x2(__uint_as_float(v[u * 8 + 4]), __uint_as_float(v[u * 8 + 5])),
                     pack_bf16x2(__uint_as_float(v[u * 8 + 6]), __uint_as_float(v[u * 8 + 7])));
      }
    }
    fence_proxy_async_smem();
  }
  named_barrier_sync(1 + w, 128);
  if (ok && r == 0 && !*reinterpret_cast<volatile int*>(&sh.abort_flag)) {
    const CUtensorMap* map = w == 0 ? &p.tmdK : &p.tmdV;
#pragma unroll
    for (int c = 0; c < 2; ++c)
      tma_store_3d(map, stage + c * C::KV_CHUNK, 128 * wk.h + 64 * c, wk.j * 128, wk.bh);
    tma_store_commit();
    tma_store_wait_all();
  }
}

template <bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1) fa_bwd256_kernel(const __grid_constant__ BwdLaunch p) {
  using C = Cfg256;
  extern __shared__ uint8_t smem_dyn[];
  __shared__ Shared256 sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = sK + C::KV_BYTES;
  uint8_t* sQ = sV + C::KV_BYTES;
  uint8_t* sdO = sQ + C::Q_BYTES;
  uint8_t* sDS = sdO + C::Q_BYTES;
  float* sLD = reinterpret_cast<float*>(sDS + C::DS_BYTES);
  const int warp = threadIdx.x >> 5;
  const Work256<CAUSAL> wk(blockIdx.x, p.BHkv, p.N, p.group);

  if (threadIdx.x == 0) {
    mbar_init(&sh.kv_full, 1);
    mbar_init(&sh.q_full, 1);
    mbar_init(&sh.q_empty, 1);
    mbar_init(&sh.do_full, 1);
    mbar_init(&sh.do_empty, 1);
    mbar_init(&sh.s_full, 1);
    mbar_init(&sh.dp_full, 1);
    mbar_init(&sh.pa_ready, 256);
    mbar_init(&sh.ds_ready, 256);
    mbar_init(&sh.pv_done, 1);
    mbar_init(&sh.dq_full, 1);
    mbar_init(&sh.dq_free, 256);
    mbar_init(&sh.acc_done, 1);
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
    if (lane_id() == 0) load_role<CAUSAL>(p, sh, sK, sV, sQ, sdO, wk);
  } else if (warp == kMmaWarp) {
    if (lane_id() == 0) mma_role<CAUSAL>(p, sh, sK, sV, sQ, sdO, sDS, tmem, wk);
  } else {
    const int w = warp >> 2;
    softmax_role<CAUSAL>(p, sh, sDS, sLD, tmem, w, wk);
    epilogue<CAUSAL>(p, sh, sK, sV, tmem, w, wk);
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

template <bool CAUSAL>
cudaError_t launch_t(const BwdLaunch& a, cudaStream_t stream) {
  auto kern = fa_bwd256_kernel<CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg256::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int T = (a.N + 127) / 128;
  kern<<<static_cast<unsigned>(static_cast<long long>(a.BHkv) * T * 2), kThreads, Cfg256::SMEM_BYTES, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_main_d256(const BwdLaunch& a, cudaStream_t stream) {
  return a.causal ? launch_t<true>(a, stream) : launch_t<false>(a, stream);
}

}  // namespace fa

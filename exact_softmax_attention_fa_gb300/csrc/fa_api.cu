// C ABI of the attention library: argument validation, TMA tensor-map
// construction, per-device state and the device status word. All compute is
// in the kernels of fa_fwd.cu / fa_bwd.cu.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

// Per-device status word written by kernels whose bounded waits gave up.
__device__ uint32_t g_status_word[4];

// One thread waits on an mbarrier that nothing arrives at; the bounded wait
// gives up after limit_ns and records FA_ERR_TIMEOUT.
__global__ void timeout_probe_kernel(uint32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, &abort_flag, limit_ns)) {
    if (atomicCAS(status, 0u, static_cast<uint32_t>(FA_ERR_TIMEOUT)) == 0u) {
      status[1] = WHERE_PROBE;
      status[2] = blockIdx.x;
      status[3] = threadIdx.x;
    }
  }
}

cudaError_t launch_timeout_probe(uint32_t* status, uint64_t limit_ns, cudaStream_t stream) {
  timeout_probe_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

// Argument checks shared by every entry point (the conventions of fa.h).
fa_status_t check_common(int B, int H, int N, int d, int causal, float scale, bool* empty) {
  if (B < 0 || H < 0 || N < 0) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  // [BH] is a TMA coordinate (int32) and the tensor byte size must fit.
  const long long bh = static_cast<long long>(B) * H;
  if (bh > INT32_MAX) return FA_ERR_INVALID_ARG;
  if (bh * N > (1ll << 40)) return FA_ERR_INVALID_ARG;
  *empty = (bh * N == 0);
  return FA_OK;
}

namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultWaitLimitNs = 4000000000ull;
constexpr uint64_t kMaxWaitLimitNs = 10000000000ull;
constexpr double kLog2e = 1.4426950408889634074;

std::atomic<unsigned long long> g_wait_limit_ns{kDefaultWaitLimitNs};
// Test hook (fa_debug_skip_arrival): role whose first arrival block 0 of the
// next launches leaves out; 0 = none.
std::atomic<uint32_t> g_debug_skip{0};

struct DeviceState {
  std::once_flag once;
  cudaError_t init_error = cudaSuccess;
  int num_sms = 0;
  int cc_major = 0, cc_minor = 0;
  uint32_t* status = nullptr;  // device address of g_status_word
};
DeviceState g_dev[kMaxDevices];

std::once_flag g_encode_once;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

// Current device's cached state; nullptr (and *err set) on failure.
DeviceState* device_state(fa_status_t* err) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *err = FA_ERR_CUDA;
    return nullptr;
  }
  DeviceState& s = g_dev[dev];
  std::call_once(s.once, [&s, dev] {
    cudaError_t e = cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&s.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&s.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e == cudaSuccess) e = cudaGetSymbolAddress(reinterpret_cast<void**>(&s.status), g_status_word);
    s.init_error = e;
  });
  if (s.init_error != cudaSuccess) {
    *err = FA_ERR_CUDA;
    return nullptr;
  }
  if (s.cc_major != 10 || s.cc_minor != 3) {  // kernels are built for sm_103a only
    *err = FA_ERR_UNSUPPORTED;
    return nullptr;
  }
  return &s;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// [BH][N][d] bf16, boxes of 128 rows x 64 columns, 128-byte swizzle; rows
// past N read as zero and are not written by stores.
bool make_map(CUtensorMap* m, const void* base, int BH, int N, int d, unsigned box_rows = 128,
              unsigned box_heads = 1) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2};
  cuuint32_t box[3] = {64, box_rows, box_heads};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The fp32 dQ accumulator [BH][Npad][d]: boxes of 128 rows x 32 columns
// (128 bytes), 128-byte swizzle, used by TMA reduce-adds.
bool make_map_f32_acc(CUtensorMap* m, void* base, int BH, int Npad, int d) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(Npad), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(Npad) * d * 4};
  cuuint32_t box[3] = {32, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


// Grouped K/V heads: Hkv >= 1 dividing Hq (nothing to check when Hq == 0).
fa_status_t check_heads(int Hq, int Hkv) {
  if (Hkv < 0) return FA_ERR_INVALID_ARG;
  if (Hq > 0 && (Hkv == 0 || Hq % Hkv != 0)) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

int round_up_128(int n) { return (n + 127) / 128 * 128; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct BwdWorkspaceLayout {
  size_t D_off, lse2_off, dq_off, sched_off, total;
};

BwdWorkspaceLayout bwd_layout(long long BH, int N, int d) {
  const size_t rows = static_cast<size_t>(BH) * round_up_128(N);
  BwdWorkspaceLayout w;
  w.D_off = 0;
  w.lse2_off = align_up(w.D_off + rows * 4, 256);
  w.dq_off = align_up(w.lse2_off + rows * 4, 256);
  w.sched_off = align_up(w.dq_off + rows * static_cast<size_t>(d) * 4, 256);
  w.total = w.sched_off + 256;
  return w;
}

// Key ranges of the split-key forward: fp32 O and L partials per range.
constexpr int kMaxSplits = 256;

size_t splitkv_bytes(long long BH, int Nq, int d, int splits) {
  return align_up(static_cast<size_t>(splits) * BH * Nq * d * 4, 256) +
         align_up(static_cast<size_t>(splits) * BH * Nq * 4, 256);
}

// Automatic number of key ranges. Work items are (query-tile pair, key
// range); the persistent grid runs them in rounds of one per SM, so the
// busiest CTA processes ceil(items * s / SMs) items of ceil(Tk / s) key tiles
// each, plus a fixed cost per item (its Q load, first S product and
// epilogue, about two key tiles' time). The count minimising that estimate
// is taken (a larger one must win by 1 %), among counts whose fp32 partials
// fit the workspace and stay below a sixteenth of the K/V bytes the call
// reads (short query blocks such as decoding; a long query block keeps one
// range). units: query-head units (heads, or packed head groups), tq: query
// tiles per unit; BH, Nq size the partials, BHkv the K/V heads.
int auto_splits(long long units, long long tq, int Nk, int d, int sms, long long BH, int Nq, long long BHkv,
                size_t room) {
  constexpr double kItemCost = 2.0;  // key tiles' time
  const long long nt = d <= 128 ? 2 : 1;  // query tiles per CTA
  const long long items = units * ((tq + nt - 1) / nt);
  const int Tk = (Nk + 127) / 128;
  if (Tk < 2 || sms <= 0 || items <= 0) return 1;
  const double kv_bytes = static_cast<double>(BHkv) * Nk * d * 2 * 2;
  int best = 1;
  double best_t = 1e300;
  for (int s = 1; s <= std::min(Tk, kMaxSplits); ++s) {
    const int per = (Tk + s - 1) / s;
    if ((Tk + per - 1) / per != s) continue;  // the count the call would actually use differs
    if (s > 1 && (splitkv_bytes(BH, Nq, d, s) > room || splitkv_bytes(BH, Nq, d, s) * 16.0 > kv_bytes)) break;
    const double rounds = static_cast<double>((items * s + sms - 1) / sms);
    const double t = rounds * (per + kItemCost);
    if (t < best_t * 0.99) {
      best_t = t;
      best = s;
    }
  }
  return best;
}

// fp32 partial dK + dV of one chunk of a group, for every K/V head.
size_t kv_part_bytes(long long BHkv, int N, int d) { return static_cast<size_t>(BHkv) * N * d * 4 * 2; }

// How many work items share one (K/V head, key tile) when g query heads read
// the same K/V head. One item per group keeps dK, dV on chip; splitting the
// group adds items and, under a causal mask, shortens the longest item (key
// tile 0 meets every query tile of every head of the group), at the price of
// fp32 partials that the main kernel writes and a post kernel reads. The
// estimate, in 128x128xd products at ~6 TFLOP/s per SM: the longest item
// against the average per SM, with the dQ kernel's 3 products per tile pair
// counted into the average when it runs after the dK/dV pass and takes the
// SMs that pass leaves idle (dq_separate); without it, non-causal items of
// equal length run in whole rounds. A split must win by 2 %. d = 256 keeps
// one item per group.
int choose_kv_chunks(long long BHkv, int g, int N, int d, int causal, int sms, size_t part_room, bool dq_separate) {
  if (g <= 1 || d == 256 || sms <= 0) return 1;
  const double T = static_cast<double>((N + 127) / 128);
  const double t_prod = 2.0 * 128 * 128 * d / 6.0e12;
  const double pairs = static_cast<double>(BHkv) * g * (causal ? T * (T + 1) / 2 : T * T);
  const double per_pair = dq_separate ? 4.0 : 5.0;  // products per tile pair in the kernel holding dK, dV
  int best = 1;
  double best_t = 1e300;
  for (int chunks = 1; chunks <= g; ++chunks) {
    if (g % chunks != 0) continue;
    if (chunks > 1 && static_cast<size_t>(chunks) * kv_part_bytes(BHkv, N, d) > part_room) break;
    const double gs = g / chunks;
    const double items = static_cast<double>(BHkv) * chunks * T;
    const double longest = per_pair * gs * T;
    double work;
    if (dq_separate)
      work = std::max(longest, (per_pair + 3.0) * pairs / sms);
    else
      work = causal ? std::max(longest, per_pair * pairs / sms) : std::ceil(items / sms) * longest;
    const double t = work * t_prod + (chunks > 1 ? 2.0 * chunks * kv_part_bytes(BHkv, N, d) / 6.0e12 : 0.0);
    if (t < best_t * 0.98) {
      best_t = t;
      best = chunks;
    }
  }
  return best;
}

fa_status_t from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return FA_OK;
  if (e == cudaErrorLaunchFailure || e == cudaErrorInvalidConfiguration || e == cudaErrorLaunchOutOfResources ||
      e == cudaErrorInvalidDeviceFunction || e == cudaErrorNoKernelImageForDevice)
    return FA_ERR_LAUNCH;
  return FA_ERR_CUDA;
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" {

int fa_version(void) { return 100; }

const char* fa_status_string(fa_status_t s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: null pointer, negative size, or bad scale/flag";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: head dimension must be 64, 128 or 256 on an sm_103a device";
    case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED: bf16 tensors need 16-byte, lse 4-byte, workspace 256-byte alignment";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE: backward workspace missing or smaller than fa_bwd_workspace_size()";
    case FA_ERR_LAUNCH: return "FA_ERR_LAUNCH: kernel launch failed";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a device-side pipeline wait exceeded its limit";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: CUDA runtime error";
  }
  return "unknown fa_status_t";
}

void fa_set_wait_limit_ns(unsigned long long limit_ns) {
  // 0 restores the default; larger values are capped, so a stalled pipeline
  // still gives up within kMaxWaitLimitNs instead of holding the GPU.
  g_wait_limit_ns.store(limit_ns == 0 ? kDefaultWaitLimitNs : std::min<unsigned long long>(limit_ns, kMaxWaitLimitNs));
}

fa_status_t fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                           int Nq, int Nk, int d, int causal, float scale, int num_splits, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream) {
  bool empty = false, empty_k = false;
  fa_status_t st = check_common(B, Hq, Nq, d, causal, scale, &empty);
  if (st != FA_OK) return st;
  st = check_common(B, Hkv, Nk, d, causal, scale, &empty_k);
  if (st != FA_OK) return st;
  st = check_heads(Hq, Hkv);
  if (st != FA_OK) return st;
  if (num_splits < 0 || num_splits > kMaxSplits) return FA_ERR_INVALID_ARG;
  if (empty) return FA_OK;
  // every query row must see at least one key
  if (Nk == 0 || (causal && Nq > Nk)) return FA_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return FA_ERR_MISALIGNED;
  const int BH = B * Hq, BHkv = B * Hkv;
  const int Tk = (Nk + 127) / 128;
  // A query block shorter than a tile shares its tiles among the query heads
  // of a K/V group (a power-of-two group of at most 128 heads).
  const int g = Hq / Hkv;
  const int pack = (Nq < 128 && g >= 2 && g <= 128 && (g & (g - 1)) == 0) ? g : 1;
  int splits = num_splits;
  if (splits == 0) {
    DeviceState* ds0 = device_state(&st);
    if (!ds0) return st;
    splits = auto_splits(BH / pack, (Nq + 128 / pack - 1) / (128 / pack), Nk, d, ds0->num_sms, BH, Nq, BHkv,
                         workspace ? workspace_bytes : 0);
  }
  int per = (Tk + splits - 1) / splits;  // key tiles per range; no range is empty
  splits = (Tk + per - 1) / per;
  if (splits > 1) {
    if (!workspace || workspace_bytes < splitkv_bytes(BH, Nq, d, splits)) return FA_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return FA_ERR_MISALIGNED;
  }
  DeviceState* ds = device_state(&st);
  if (!ds) return st;
  FwdLaunch a{};
  if (!make_map(&a.tmQ, q, BH, Nq, d, 128 / pack, pack) || !make_map(&a.tmK, k, BHkv, Nk, d) ||
      !make_map(&a.tmV, v, BHkv, Nk, d) || !make_map(&a.tmO, o, BH, Nq, d, 128 / pack, pack))
    return FA_ERR_CUDA;
  a.lse = lse;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.pack = pack;
  a.rph = 128 / pack;
  a.status = ds->status;
  a.Nq = Nq;
  a.Nk = Nk;
  a.causal_off = Nk - Nq;
  a.BH = BH;
  a.d = d;
  a.causal = causal;
  a.group = Hq / Hkv;
  a.splits = splits;
  a.kv_per_split = per;
  if (splits > 1) {
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    a.o_part = reinterpret_cast<float*>(ws);
    a.lse_part = reinterpret_cast<float*>(ws + align_up(static_cast<size_t>(splits) * BH * Nq * d * 4, 256));
  }
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * kLog2e);
  a.wait_limit_ns = g_wait_limit_ns.load();
  a.num_sms = ds->num_sms;
  a.debug_skip = g_debug_skip.load();
  cudaError_t e = launch_fwd(a, stream);
  if (e == cudaSuccess && splits > 1) e = launch_fwd_combine(a, stream);
  return from_cuda(e);
}

size_t fa_fwd_splitkv_workspace_size(int B, int Hq, int Nq, int d, int num_splits) {
  bool empty = false;
  if (check_common(B, Hq, Nq, d, 0, 1.0f, &empty) != FA_OK || empty || num_splits < 2 || num_splits > kMaxSplits)
    return 0;
  return splitkv_bytes(static_cast<long long>(B) * Hq, Nq, d, num_splits);
}

fa_status_t fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                       int N, int d, int causal, float scale, cudaStream_t stream) {
  return fa_fwd_splitkv(q, k, v, o, lse, B, Hq, Hkv, N, N, d, causal, scale, 1, nullptr, 0, stream);
}

fa_status_t fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                   int causal, float scale, cudaStream_t stream) {
  return fa_fwd_gqa(q, k, v, o, lse, B, H, H, N, d, causal, scale, stream);
}

size_t fa_bwd_gqa_workspace_size(int B, int Hq, int Hkv, int N, int d) {
  bool empty = false;
  if (check_common(B, Hq, N, d, 0, 1.0f, &empty) != FA_OK || check_heads(Hq, Hkv) != FA_OK || empty) return 0;
  const size_t base = bwd_layout(static_cast<long long>(B) * Hq, N, d).total;
  const int g = Hq / Hkv;
  if (g <= 1 || d == 256) return base;
  return base + static_cast<size_t>(g) * kv_part_bytes(static_cast<long long>(B) * Hkv, N, d);
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
  bool empty = false;
  if (check_common(B, H, N, d, 0, 1.0f, &empty) != FA_OK || empty) return 0;
  return bwd_layout(static_cast<long long>(B) * H, N, d).total;
}

}  // extern "C"

namespace {

// Validation and launch-argument setup shared by fa_bwd and its phases. A
// null entry in `need` means the phase does not use that tensor.
struct BwdTensors {
  const void *q, *k, *v, *o, *dO;
  const float* lse;
  void *dq, *dk, *dv;
};

// dq_separate: the call forms dQ with the separate dQ kernel after the dK/dV
// pass (the deterministic route), which the work-item split takes into account.
fa_status_t prepare_bwd(const BwdTensors& t, int B, int H, int Hkv, int N, int d, int causal, float scale,
                        void* workspace, size_t workspace_bytes, bool* empty, BwdLaunch* a,
                        bool dq_separate = false) {
  fa_status_t st = check_common(B, H, N, d, causal, scale, empty);
  if (st != FA_OK) return st;
  st = check_heads(H, Hkv);
  if (st != FA_OK || *empty) return st;
  const void* bf16_ptrs[] = {t.q, t.k, t.v, t.o, t.dO, t.dq, t.dk, t.dv};
  for (const void* p : bf16_ptrs)
    if (p && !aligned(p, 16)) return FA_ERR_MISALIGNED;
  if (t.lse && !aligned(t.lse, 4)) return FA_ERR_MISALIGNED;
  const int BH = B * H;
  const BwdWorkspaceLayout wl = bwd_layout(BH, N, d);
  if (!workspace || workspace_bytes < wl.total) return FA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return FA_ERR_MISALIGNED;
  DeviceState* ds = device_state(&st);
  if (!ds) return st;
  *a = BwdLaunch{};
  const int BHkv = B * Hkv;
  auto map = [&](CUtensorMap* m, const void* ptr, int heads, unsigned rows) {
    return !ptr || make_map(m, ptr, heads, N, d, rows);
  };
  // d = 256 streams Q and dO in 64-row query tiles (smem budget); all other
  // tiles are 128 rows. Q, dO have BH heads, K, V, dK, dV have BHkv.
  const unsigned q_rows = d == 256 ? 64 : 128;
  if (!map(&a->tmQ, t.q, BH, q_rows) || !map(&a->tmK, t.k, BHkv, 128) || !map(&a->tmV, t.v, BHkv, 128) ||
      !map(&a->tmdO, t.dO, BH, q_rows) || !map(&a->tmdK, t.dk, BHkv, 128) || !map(&a->tmdV, t.dv, BHkv, 128))
    return FA_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a->o = static_cast<const __nv_bfloat16*>(t.o);
  a->dO = static_cast<const __nv_bfloat16*>(t.dO);
  a->lse = t.lse;
  a->dq = static_cast<__nv_bfloat16*>(t.dq);
  a->dk = static_cast<__nv_bfloat16*>(t.dk);
  a->dv = static_cast<__nv_bfloat16*>(t.dv);
  a->D = reinterpret_cast<float*>(ws + wl.D_off);
  a->lse2 = reinterpret_cast<float*>(ws + wl.lse2_off);
  a->dq_acc = reinterpret_cast<float*>(ws + wl.dq_off);
  a->sched = reinterpret_cast<uint32_t*>(ws + wl.sched_off);
  // Room after the fixed layout holds the split groups' dK, dV partials.
  const size_t part_room = workspace_bytes > wl.total ? workspace_bytes - wl.total : 0;
  a->chunks = choose_kv_chunks(BHkv, H / (Hkv > 0 ? Hkv : 1), N, d, causal, ds->num_sms, part_room, dq_separate);
  a->kv_part = reinterpret_cast<float*>(ws + wl.total);
  if (!make_map_f32_acc(&a->tmdQacc, a->dq_acc, BH, round_up_128(N), d)) return FA_ERR_CUDA;
  a->status = ds->status;
  a->N = N;
  a->Npad = round_up_128(N);
  a->BH = BH;
  a->BHkv = BHkv;
  a->group = H / Hkv;
  a->d = d;
  a->causal = causal;
  a->scale = scale;
  a->scale_log2 = static_cast<float>(static_cast<double>(scale) * kLog2e);
  a->wait_limit_ns = g_wait_limit_ns.load();
  a->num_sms = ds->num_sms;
  a->debug_skip = g_debug_skip.load();
  return FA_OK;
}

}  // namespace

extern "C" {

fa_status_t fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const float* lse,
                       const void* dO, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N, int d,
                       int causal, float scale, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  bool empty = false;
  fa_status_t st = check_common(B, Hq, N, d, causal, scale, &empty);
  if (st != FA_OK) return st;
  st = check_heads(Hq, Hkv);
  if (st != FA_OK) return st;
  if (empty) return FA_OK;
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  // d = 128: dQ from the per-query-tile kernel (measured faster than the
  // atomic accumulation at this head dimension, and reproducible); d = 64,
  // 256: atomic accumulation in the main kernel.
  if (d == 128)
    return fa_bwd_gqa_deterministic(q, k, v, o, lse, dO, dq, dk, dv, B, Hq, Hkv, N, d, causal, scale, workspace,
                                    workspace_bytes, stream);
  BwdLaunch a;
  st = prepare_bwd(BwdTensors{q, k, v, o, dO, lse, dq, dk, dv}, B, Hq, Hkv, N, d, causal, scale, workspace,
                   workspace_bytes, &empty, &a);
  if (st != FA_OK || empty) return st;
  cudaError_t e = launch_bwd_pre(a, stream);
  if (e == cudaSuccess) e = launch_bwd_main(a, stream);
  if (e == cudaSuccess) e = launch_bwd_post(a, stream);
  return from_cuda(e);
}

fa_status_t fa_bwd_gqa_deterministic(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                     const void* dO, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N,
                                     int d, int causal, float scale, void* workspace, size_t workspace_bytes,
                                     cudaStream_t stream) {
  bool empty = false;
  fa_status_t st = check_common(B, Hq, N, d, causal, scale, &empty);
  if (st != FA_OK) return st;
  st = check_heads(Hq, Hkv);
  if (st != FA_OK) return st;
  if (empty) return FA_OK;
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  BwdLaunch a;
  st = prepare_bwd(BwdTensors{q, k, v, o, dO, lse, dq, dk, dv}, B, Hq, Hkv, N, d, causal, scale, workspace,
                   workspace_bytes, &empty, &a, true);
  if (st != FA_OK || empty) return st;
  a.deterministic = 1;
  cudaError_t e = launch_bwd_pre(a, stream);
  if (e == cudaSuccess) e = launch_bwd_main(a, stream);  // dK, dV only
  // The dQ kernel reads nothing the dK/dV pass writes: it may take the SMs
  // that pass leaves idle in its last round.
  a.overlap_prev = 1;
  if (e == cudaSuccess) e = launch_bwd_dq(a, stream);
  a.overlap_prev = 0;
  if (e == cudaSuccess) e = launch_bwd_post(a, stream);  // split groups' dK, dV sums, if any
  return from_cuda(e);
}

fa_status_t fa_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                 const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal,
                                 float scale, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return fa_bwd_gqa_deterministic(q, k, v, o, lse, dO, dq, dk, dv, B, H, H, N, d, causal, scale, workspace,
                                  workspace_bytes, stream);
}

fa_status_t fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                   void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal, float scale,
                   void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return fa_bwd_gqa(q, k, v, o, lse, dO, dq, dk, dv, B, H, H, N, d, causal, scale, workspace, workspace_bytes,
                    stream);
}

fa_status_t fa_bwd_preprocess(const void* o, const float* lse, const void* dO, int B, int H, int N, int d,
                              void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  bool empty = false;
  fa_status_t st = check_common(B, H, N, d, 0, 1.0f, &empty);
  if (st != FA_OK) return st;
  if (empty) return FA_OK;
  if (!o || !lse || !dO) return FA_ERR_INVALID_ARG;
  BwdLaunch a;
  st = prepare_bwd(BwdTensors{nullptr, nullptr, nullptr, o, dO, lse, nullptr, nullptr, nullptr}, B, H, H, N, d, 0, 1.0f,
                   workspace, workspace_bytes, &empty, &a);
  if (st != FA_OK || empty) return st;
  return from_cuda(launch_bwd_pre(a, stream));
}

fa_status_t fa_bwd_preprocess_stats(const void* o, const float* lse, const void* dO, int B, int H, int N, int d,
                                    void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  bool empty = false;
  fa_status_t st = check_common(B, H, N, d, 0, 1.0f, &empty);
  if (st != FA_OK) return st;
  if (empty) return FA_OK;
  if (!o || !lse || !dO) return FA_ERR_INVALID_ARG;
  BwdLaunch a;
  st = prepare_bwd(BwdTensors{nullptr, nullptr, nullptr, o, dO, lse, nullptr, nullptr, nullptr}, B, H, H, N, d, 0, 1.0f,
                   workspace, workspace_bytes, &empty, &a);
  if (st != FA_OK || empty) return st;
  a.deterministic = 1;  // the accumulator is not zeroed: the dQ kernel does not use it
  return from_cuda(launch_bwd_pre(a, stream));
}

fa_status_t fa_bwd_main(const void* q, const void* k, const void* v, const void* dO, void* dk, void* dv, int B,
                        int H, int N, int d, int causal, float scale, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream) {
  bool empty = false;
  fa_status_t st = check_common(B, H, N, d, causal, scale, &empty);
  if (st != FA_OK) return st;
  if (empty) return FA_OK;
  if (!q || !k || !v || !dO || !dk || !dv) return FA_ERR_INVALID_ARG;
  BwdLaunch a;
  st = prepare_bwd(BwdTensors{q, k, v, nullptr, dO, nullptr, nullptr, dk, dv}, B, H, H, N, d, causal, scale, workspace,
                   workspace_bytes, &empty, &a);
  if (st != FA_OK || empty) return st;
  return from_cuda(launch_bwd_main(a, stream));
}

fa_status_t fa_bwd_dkdv(const void* q, const void* k, const void* v, const void* dO, void* dk, void* dv, int B,
                        int H, int N, int d, int causal, float scale, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream) {
  bool empty = false;
  fa_status_t st = check_common(B, H, N, d, causal, scale, &empty);
  if (st != FA_OK) return st;
    if (empty) return FA_OK;
  if (!q || !k || !v || !dO || !dk || !dv) return FA_ERR_INVALID_ARG;
  BwdLaunch a;
  st = prepare_bwd(BwdTensors{q, k, v, nullptr, dO, nullptr, nullptr, dk, dv}, B, H, H, N, d, causal, scale,
                   workspace, workspace_bytes, &empty, &a);
  if (st != FA_OK || empty) return st;
  a.deterministic = 1;
  return from_cuda(launch_bwd_main(a, stream));
}

fa_status_t fa_bwd_dq(const void* q, const void* k, const void* v, const void* dO, void* dq, int B, int H, int N,
                      int d, int causal, float scale, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  bool empty = false;
  fa_status_t st = check_common(B, H, N, d, causal, scale, &empty);
  if (st != FA_OK) return st;
    if (empty) return FA_OK;
  if (!q || !k || !v || !dO || !dq) return FA_ERR_INVALID_ARG;
  BwdLaunch a;
  st = prepare_bwd(BwdTensors{q, k, v, nullptr, dO, nullptr, dq, nullptr, nullptr}, B, H, H, N, d, causal, scale,
                   workspace, workspace_bytes, &empty, &a);
  if (st != FA_OK || empty) return st;
  a.deterministic = 1;
  return from_cuda(launch_bwd_dq(a, stream));
}

fa_status_t fa_bwd_postprocess(void* dq, int B, int H, int N, int d, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream) {
  bool empty = false;
  fa_status_t st = check_common(B, H, N, d, 0, 1.0f, &empty);
  if (st != FA_OK) return st;
  if (empty) return FA_OK;
  if (!dq) return FA_ERR_INVALID_ARG;
  BwdLaunch a;
  st = prepare_bwd(BwdTensors{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, dq, nullptr, nullptr}, B, H, H, N,
                   d, 0, 1.0f, workspace, workspace_bytes, &empty, &a);
  if (st != FA_OK || empty) return st;
  return from_cuda(launch_bwd_post(a, stream));
}

fa_status_t fa_get_device_status_detail(unsigned int* word, cudaStream_t stream) {
  if (!word) return FA_ERR_INVALID_ARG;
  fa_status_t st = FA_OK;
  DeviceState* ds = device_state(&st);
  if (!ds) return st;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
  uint32_t w[4] = {0, 0, 0, 0};
  if (cudaMemcpy(w, ds->status, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  if (w[0] != 0) {
    const uint32_t zero[4] = {0, 0, 0, 0};
    if (cudaMemcpy(ds->status, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_CUDA;
  }
  for (int i = 0; i < 4; ++i) word[i] = w[i];
  return static_cast<fa_status_t>(w[0]);
}

fa_status_t fa_get_device_status(cudaStream_t stream) {
  unsigned int word[4];
  return fa_get_device_status_detail(word, stream);
}

fa_status_t fa_debug_skip_arrival(unsigned int role) {
  switch (role) {
    case 0:
    case WHERE_FWD_LOAD:
    case WHERE_FWD_MMA:
    case WHERE_FWD_SOFTMAX:
    case WHERE_BWD_LOAD:
    case WHERE_BWD_MMA:
    case WHERE_BWD_SOFTMAX:
    case WHERE_BWD_DQ:
      g_debug_skip.store(role);
      return FA_OK;
    default:
      return FA_ERR_INVALID_ARG;
  }
}

fa_status_t fa_debug_timeout_probe(unsigned long long limit_ns, cudaStream_t stream) {
  fa_status_t st = FA_OK;
  DeviceState* ds = device_state(&st);
  if (!ds) return st;
  if (limit_ns == 0 || limit_ns > kMaxWaitLimitNs) return FA_ERR_INVALID_ARG;
  return from_cuda(launch_timeout_probe(ds->status, limit_ns, stream));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free backward: a fixed scratch array compiled into the library
// stands in for the caller's workspace.
// ---------------------------------------------------------------------------
namespace fa {

static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_BWD_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of g_noalloc_scratch per device, looked up on the first
// call that finds the device usable. A failed lookup is not remembered, so a
// later call tries again.
struct NoAllocState {
  std::mutex mu;
  void* scratch = nullptr;
};
NoAllocState g_noalloc[kMaxDevices];

}  // namespace
}  // namespace fa

extern "C" fa_status_t fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                      const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                                      int causal, float scale, cudaStream_t stream) {
  bool empty = false;
  fa_status_t st = check_common(B, H, N, d, causal, scale, &empty);
  if (st != FA_OK) return st;
  if (empty) return FA_OK;
  if (fa_bwd_workspace_size(B, H, N, d) > FA_BWD_NOALLOC_SCRATCH_BYTES) return FA_ERR_WORKSPACE;
  // The device must be one the kernels run on (sm_103a) before its copy of
  // the array is looked up.
  DeviceState* ds = device_state(&st);
  if (!ds) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  NoAllocState& ns = g_noalloc[dev];
  void* scratch = nullptr;
  {
    // Once per device, with that device current: the array's device address.
    // In host code the symbol itself is only a host-side stand-in.
    std::lock_guard<std::mutex> lock(ns.mu);
    if (!ns.scratch && cudaGetSymbolAddress(&ns.scratch, g_noalloc_scratch) != cudaSuccess) ns.scratch = nullptr;
    scratch = ns.scratch;
  }
  if (!scratch) return FA_ERR_CUDA;
  return fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, causal, scale, scratch, FA_BWD_NOALLOC_SCRATCH_BYTES,
                stream);
}


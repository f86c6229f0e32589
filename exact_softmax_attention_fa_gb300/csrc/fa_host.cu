// Host-buffer entry points: a forward (and backward) pass of a problem whose
// inputs and outputs live in host memory. The library owns, per device, two
// copy streams (host->device, device->host), two forward streams at the
// greatest stream priority and two streams per head group for the backward,
// and orders them against the caller's stream with events, so the copies
// overlap the kernels. Rows of different heads are independent problems, and
// a head's result does not depend on which launch computes it, so
// fa_fwd_bwd_host splits the heads into groups that flow through the copies
// and kernels one after another (default plan: four groups, the middle two
// with their forward in two launches):
//
//   h2d:      QKV g0 | dO g0 | QKV g1 (2 chunks) | dO g1 | QKV g2 ... | dO g3
//   fwd 0,1:    fwd g0 |  fwd g1 chunks  |  fwd g2 chunks  | fwd g3
//   bwd g:             D g | dK,dV g         (one stream per group)
//   bwd_dq g:              | dQ g            (one stream per group)
//   d2h:         O,L | dK,dV | dQ of each group, in the order they are final
//
// Each group has its own slice of the backward workspace, so no kernel of one
// group waits for another group's kernels, and a group's dK/dV and dQ kernels
// (both read only Q, K, V, dO and the preprocess's D, L) run side by side.
// The persistent kernels fill every SM: a kernel queued on another stream
// takes the SMs a running one frees in its last round, so the partly empty
// last rounds of the many launches fill with other launches' work, and the
// forward chunks, whose results every later step needs, are dispatched first
// (no kernel waits on another's progress). The plan (make_plan) keeps the
// first group small, so the device starts after a short upload, and the last
// group small, so little work and little read-back remain once its dO has
// arrived (every byte crosses the host link, which is slower than the kernels
// consume them). Nothing here computes: the work is the same sequence of
// kernels fa_fwd and fa_bwd launch.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxGroups = 4;  // head groups of fa_fwd_bwd_host, at most
constexpr int kMaxChunks = 2;  // forward launches per group, at most

// Events of one fa_fwd_bwd_host call.
enum : int {
  EV_START,
  EV_DONE,
  EV_DO0,                               // per group: its dO is on the device
  EV_PRE0 = EV_DO0 + kMaxGroups,        // per group: its D and L are in its workspace
  EV_DKDV0 = EV_PRE0 + kMaxGroups,      // per group: its dK and dV are final
  EV_BWD0 = EV_DKDV0 + kMaxGroups,      // per group: its dQ is final
  EV_IN0 = EV_BWD0 + kMaxGroups,        // per forward chunk: its Q, K, V are on the device
  EV_OUT0 = EV_IN0 + kMaxGroups * kMaxChunks,  // per forward chunk: its O and L are final
  EV_COUNT = EV_OUT0 + kMaxGroups * kMaxChunks
};

constexpr int kFwdOnlyChunks = 8;  // fa_fwd_host: uploads, forwards and read-backs pipelined over 8 head chunks

struct CopyState {
  std::once_flag once;
  cudaError_t error = cudaSuccess;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaStream_t fwd[2] = {};                  // forward chunks, at the greatest stream priority
  cudaStream_t bwd[kMaxGroups] = {};         // per group: preprocess, dK/dV (or the whole backward)
  cudaStream_t bwd_dq[kMaxGroups] = {};      // per group: the dQ kernel
  cudaEvent_t ev[EV_COUNT] = {};
  cudaEvent_t fwd_in[kFwdOnlyChunks] = {}, fwd_out[kFwdOnlyChunks] = {};
  int num_sms = 0;
  std::mutex mu;  // one call at a time per device enqueues on the shared streams and events
};
CopyState g_copy[kMaxDevices];

CopyState* copy_state(int dev) {
  CopyState& cs = g_copy[dev];
  std::call_once(cs.once, [&cs, dev] {
    cudaError_t e = cudaDeviceGetAttribute(&cs.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&cs.h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&cs.d2h, cudaStreamNonBlocking);
    int least = 0, greatest = 0;
    if (e == cudaSuccess) e = cudaDeviceGetStreamPriorityRange(&least, &greatest);
    for (int i = 0; i < 2 && e == cudaSuccess; ++i)
      e = cudaStreamCreateWithPriority(&cs.fwd[i], cudaStreamNonBlocking, greatest);
    for (int i = 0; i < kMaxGroups && e == cudaSuccess; ++i) {
      e = cudaStreamCreateWithFlags(&cs.bwd[i], cudaStreamNonBlocking);
      if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&cs.bwd_dq[i], cudaStreamNonBlocking);
    }
    for (int i = 0; i < EV_COUNT && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&cs.ev[i], cudaEventDisableTiming);
    for (int i = 0; i < kFwdOnlyChunks && e == cudaSuccess; ++i) {
      e = cudaEventCreateWithFlags(&cs.fwd_in[i], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&cs.fwd_out[i], cudaEventDisableTiming);
    }
    cs.error = e;
  });
  return cs.error == cudaSuccess ? &cs : nullptr;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// How fa_fwd_bwd_host splits B*H heads: group g holds heads
// [first[g], first[g + 1]) and runs its forward in chunks[g] launches.
struct Plan {
  int groups;
  long long first[kMaxGroups + 1];
  int chunks[kMaxGroups];
};

// A small first group (an eighth of the heads) starts the device after a
// short upload; a small last group (another eighth) leaves little work and
// little read-back after the last upload; the heads between form two middle
// groups, each with its forward in two launches that follow its uploads.
Plan make_plan(long long BH) {
  Plan p{};
  const long long g0 = (BH + 7) / 8;
  const long long last = BH - g0 >= 2 ? (BH + 7) / 8 : BH - g0;
  const long long mid = BH - g0 - last;
  p.first[0] = 0;
  p.groups = 0;
  p.first[++p.groups] = g0;
  if (mid >= 2) p.first[++p.groups] = g0 + mid / 2;
  if (mid >= 1) p.first[++p.groups] = g0 + mid;
  if (last > 0) p.first[++p.groups] = BH;
  for (int g = 0; g < p.groups; ++g) {
    const long long h = p.first[g + 1] - p.first[g];
    p.chunks[g] = static_cast<int>(std::min<long long>(g == 0 || g == p.groups - 1 ? 1 : 2, h));
  }
  return p;
}

// Device buffer: q, k, v, dO, o, dq, dk, dv (bf16), lse (fp32), then one
// backward workspace per group of the plan; every part starts on a 256-byte
// boundary.
struct HostLayout {
  size_t q, k, v, dO, o, dq, dk, dv, lse, ws[kMaxGroups], ws_bytes[kMaxGroups], total;
};

HostLayout host_layout(int B, int H, int N, int d, const Plan& P) {
  HostLayout L{};
  const size_t rows = static_cast<size_t>(B) * H * N;
  const size_t tb = align256(rows * d * 2), lb = align256(rows * 4);
  size_t off = 0;
  for (size_t* f : {&L.q, &L.k, &L.v, &L.dO, &L.o, &L.dq, &L.dk, &L.dv}) {
    *f = off;
    off += tb;
  }
  L.lse = off;
  off += lb;
  for (int g = 0; g < P.groups; ++g) {
    L.ws[g] = off;
    L.ws_bytes[g] = fa_bwd_workspace_size(1, static_cast<int>(P.first[g + 1] - P.first[g]), N, d);
    off += align256(L.ws_bytes[g]);
  }
  L.total = off;
  return L;
}

// fa_fwd_host's device buffer: q, k, v, o (bf16), lse (fp32).
struct FwdHostLayout {
  size_t q, k, v, o, lse, total;
};

FwdHostLayout fwd_host_layout(int B, int H, int N, int d) {
  FwdHostLayout L{};
  const size_t rows = static_cast<size_t>(B) * H * N;
  const size_t tb = align256(rows * d * 2);
  L.q = 0;
  L.k = tb;
  L.v = 2 * tb;
  L.o = 3 * tb;
  L.lse = 4 * tb;
  L.total = 4 * tb + align256(rows * 4);
  return L;
}

}  // namespace
}  // namespace fa

extern "C" {

size_t fa_fwd_host_device_bytes(int B, int H, int N, int d) {
  bool empty = false;
  if (fa::check_common(B, H, N, d, 0, 1.0f, &empty) != FA_OK || empty) return 0;
  return fa::fwd_host_layout(B, H, N, d).total;
}

// Forward of host tensors, pipelined over chunks of heads: chunk c uploads
// while chunk c - 1 computes and chunk c - 2 is read back.
fa_status_t fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                        int causal, float scale, void* device_buffer, size_t device_bytes, cudaStream_t stream) {
  using namespace fa;
  bool empty = false;
  fa_status_t st = check_common(B, H, N, d, causal, scale, &empty);
  if (st != FA_OK) return st;
  if (empty) return FA_OK;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  const FwdHostLayout L = fwd_host_layout(B, H, N, d);
  if (!device_buffer || device_bytes < L.total) return FA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(device_buffer) % 256 != 0) return FA_ERR_MISALIGNED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  CopyState* cs = copy_state(dev);
  if (!cs) return FA_ERR_CUDA;

  uint8_t* base = static_cast<uint8_t*>(device_buffer);
  uint8_t *Qd = base + L.q, *Kd = base + L.k, *Vd = base + L.v, *Od = base + L.o;
  float* Ld = reinterpret_cast<float*>(base + L.lse);
  const long long BH = static_cast<long long>(B) * H;
  const size_t head_bytes = static_cast<size_t>(N) * d * 2, head_lse = static_cast<size_t>(N) * 4;
  const auto* hq = static_cast<const uint8_t*>(q);
  const auto* hk = static_cast<const uint8_t*>(k);
  const auto* hv = static_cast<const uint8_t*>(v);
  auto* ho = static_cast<uint8_t*>(o);
  auto* hl = reinterpret_cast<uint8_t*>(lse);

  std::lock_guard<std::mutex> lock(cs->mu);
  cudaError_t e = cudaSuccess;
  auto ok = [&e](cudaError_t x) {
    if (e == cudaSuccess) e = x;
  };
  ok(cudaEventRecord(cs->ev[EV_START], stream));
  ok(cudaStreamWaitEvent(cs->h2d, cs->ev[EV_START], 0));
  const int chunks = static_cast<int>(std::min<long long>(kFwdOnlyChunks, BH));
  for (int c = 0; c < chunks; ++c) {
    const long long h0 = BH * c / chunks, h1 = BH * (c + 1) / chunks;
    const size_t off = h0 * head_bytes, n = (h1 - h0) * head_bytes;
    ok(cudaMemcpyAsync(Qd + off, hq + off, n, cudaMemcpyHostToDevice, cs->h2d));
    ok(cudaMemcpyAsync(Kd + off, hk + off, n, cudaMemcpyHostToDevice, cs->h2d));
    ok(cudaMemcpyAsync(Vd + off, hv + off, n, cudaMemcpyHostToDevice, cs->h2d));
    ok(cudaEventRecord(cs->fwd_in[c], cs->h2d));
  }
  for (int c = 0; c < chunks; ++c) {
    const long long h0 = BH * c / chunks, h1 = BH * (c + 1) / chunks;
    const size_t off = h0 * head_bytes, n = (h1 - h0) * head_bytes;
    cudaStream_t fs = cs->fwd[c & 1];  // a chunk's launch fills the last round of the one before
    ok(cudaStreamWaitEvent(fs, cs->fwd_in[c], 0));
    if (st == FA_OK && e == cudaSuccess)
      st = fa_fwd(Qd + off, Kd + off, Vd + off, Od + off, Ld + h0 * N, 1, static_cast<int>(h1 - h0), N, d, causal,
                  scale, fs);
    ok(cudaEventRecord(cs->fwd_out[c], fs));
    ok(cudaStreamWaitEvent(cs->d2h, cs->fwd_out[c], 0));
    ok(cudaMemcpyAsync(ho + off, Od + off, n, cudaMemcpyDeviceToHost, cs->d2h));
    ok(cudaMemcpyAsync(hl + h0 * head_lse, Ld + h0 * N, (h1 - h0) * head_lse, cudaMemcpyDeviceToHost, cs->d2h));
  }
  ok(cudaEventRecord(cs->ev[EV_DONE], cs->d2h));
  ok(cudaStreamWaitEvent(stream, cs->ev[EV_DONE], 0));
  if (st != FA_OK) return st;
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

size_t fa_fwd_bwd_host_device_bytes(int B, int H, int N, int d) {
  bool empty = false;
  if (fa::check_common(B, H, N, d, 0, 1.0f, &empty) != FA_OK || empty) return 0;
  return fa::host_layout(B, H, N, d, fa::make_plan(static_cast<long long>(B) * H)).total;
}

fa_status_t fa_fwd_bwd_host(const void* q, const void* k, const void* v, const void* dO, void* o, float* lse,
                            void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal, float scale,
                            void* device_buffer, size_t device_bytes, cudaStream_t stream) {
  using namespace fa;
  bool empty = false;
  fa_status_t st = check_common(B, H, N, d, causal, scale, &empty);
  if (st != FA_OK) return st;
  if (empty) return FA_OK;
  if (!q || !k || !v || !dO || !o || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(B) * H;
  const Plan P = make_plan(BH);
  const HostLayout L = host_layout(B, H, N, d, P);
  if (!device_buffer || device_bytes < L.total) return FA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(device_buffer) % 256 != 0) return FA_ERR_MISALIGNED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  CopyState* cs = copy_state(dev);
  if (!cs) return FA_ERR_CUDA;

  // Device copies: Qd, Kd, Vd, dOd in; Od, Ld, dQd, dKd, dVd out.
  uint8_t* base = static_cast<uint8_t*>(device_buffer);
  uint8_t *Qd = base + L.q, *Kd = base + L.k, *Vd = base + L.v, *dOd = base + L.dO, *Od = base + L.o;
  uint8_t *dQd = base + L.dq, *dKd = base + L.dk, *dVd = base + L.dv;
  float* Ld = reinterpret_cast<float*>(base + L.lse);
  const size_t head_bytes = static_cast<size_t>(N) * d * 2;
  const auto* hq = static_cast<const uint8_t*>(q);
  const auto* hk = static_cast<const uint8_t*>(k);
  const auto* hv = static_cast<const uint8_t*>(v);

  std::lock_guard<std::mutex> lock(cs->mu);
  cudaError_t e = cudaSuccess;
  auto ok = [&e](cudaError_t x) {
    if (e == cudaSuccess) e = x;
  };
  auto run = [&st, &e](fa_status_t x) {
    if (st == FA_OK && e == cudaSuccess) st = x;
  };
  const auto H2D = cudaMemcpyHostToDevice;
  const auto D2H = cudaMemcpyDeviceToHost;
  // Earlier work on `stream` may still read the device buffer: the uploads wait for it.
  ok(cudaEventRecord(cs->ev[EV_START], stream));
  ok(cudaStreamWaitEvent(cs->h2d, cs->ev[EV_START], 0));
  auto chunk_first = [&P](int g, int c) { return P.first[g] + (P.first[g + 1] - P.first[g]) * c / P.chunks[g]; };
  // Uploads, in the order the kernels consume them.
  for (int g = 0; g < P.groups; ++g) {
    for (int c = 0; c < P.chunks[g]; ++c) {
      const long long h0 = chunk_first(g, c), h1 = chunk_first(g, c + 1);
      const size_t off = h0 * head_bytes, n = (h1 - h0) * head_bytes;
      ok(cudaMemcpyAsync(Qd + off, hq + off, n, H2D, cs->h2d));
      ok(cudaMemcpyAsync(Kd + off, hk + off, n, H2D, cs->h2d));
      ok(cudaMemcpyAsync(Vd + off, hv + off, n, H2D, cs->h2d));
      ok(cudaEventRecord(cs->ev[EV_IN0 + g * kMaxChunks + c], cs->h2d));
    }
    const size_t off = P.first[g] * head_bytes, n = (P.first[g + 1] - P.first[g]) * head_bytes;
    ok(cudaMemcpyAsync(dOd + off, static_cast<const uint8_t*>(dO) + off, n, H2D, cs->h2d));
    ok(cudaEventRecord(cs->ev[EV_DO0 + g], cs->h2d));
  }

  // Forward, one launch per chunk of heads (a [1][h1 - h0] problem),
  // alternately on the two forward streams.
  int alt = 0;
  for (int g = 0; g < P.groups; ++g) {
    for (int c = 0; c < P.chunks[g]; ++c) {
      const long long h0 = chunk_first(g, c), h1 = chunk_first(g, c + 1);
      const size_t off = h0 * head_bytes;
      cudaStream_t fs = cs->fwd[alt++ & 1];
      ok(cudaStreamWaitEvent(fs, cs->ev[EV_IN0 + g * kMaxChunks + c], 0));
      run(fa_fwd(Qd + off, Kd + off, Vd + off, Od + off, Ld + h0 * N, 1, static_cast<int>(h1 - h0), N, d, causal,
                 scale, fs));
      ok(cudaEventRecord(cs->ev[EV_OUT0 + g * kMaxChunks + c], fs));
    }
  }

  // Backward per group, on the group's own streams and workspace: the phases
  // fa_bwd runs for this head dimension (d = 128: dQ side by side with dK,
  // dV). The read-backs are queued in the order their data is final.
  auto* ho = static_cast<uint8_t*>(o);
  auto* hl = reinterpret_cast<uint8_t*>(lse);
  auto* hdq = static_cast<uint8_t*>(dq);
  auto* hdk = static_cast<uint8_t*>(dk);
  auto* hdv = static_cast<uint8_t*>(dv);
  const size_t head_lse = static_cast<size_t>(N) * 4;
  for (int g = 0; g < P.groups && e == cudaSuccess && st == FA_OK; ++g) {
    const long long g0 = P.first[g], Hg = P.first[g + 1] - g0;
    const int hg = static_cast<int>(Hg);
    const size_t off = g0 * head_bytes, n = Hg * head_bytes;
    void* ws = base + L.ws[g];
    const size_t wsb = L.ws_bytes[g];
    cudaStream_t bs = cs->bwd[g], qs = cs->bwd_dq[g];
    for (int c = 0; c < P.chunks[g]; ++c) {
      const long long h0 = chunk_first(g, c), h1 = chunk_first(g, c + 1);
      ok(cudaStreamWaitEvent(bs, cs->ev[EV_OUT0 + g * kMaxChunks + c], 0));
      ok(cudaStreamWaitEvent(cs->d2h, cs->ev[EV_OUT0 + g * kMaxChunks + c], 0));
      ok(cudaMemcpyAsync(ho + h0 * head_bytes, Od + h0 * head_bytes, (h1 - h0) * head_bytes, D2H, cs->d2h));
      ok(cudaMemcpyAsync(hl + h0 * head_lse, Ld + h0 * N, (h1 - h0) * head_lse, D2H, cs->d2h));
    }
    ok(cudaStreamWaitEvent(bs, cs->ev[EV_DO0 + g], 0));
    uint8_t *q_g = Qd + off, *k_g = Kd + off, *v_g = Vd + off, *do_g = dOd + off;
    // d = 128 runs the dQ kernel, which needs no zeroed accumulator
    if (d == 128) run(fa_bwd_preprocess_stats(Od + off, Ld + g0 * N, do_g, 1, hg, N, d, ws, wsb, bs));
    else run(fa_bwd_preprocess(Od + off, Ld + g0 * N, do_g, 1, hg, N, d, ws, wsb, bs));
    if (d == 128) {
      ok(cudaEventRecord(cs->ev[EV_PRE0 + g], bs));
      ok(cudaStreamWaitEvent(qs, cs->ev[EV_PRE0 + g], 0));
      run(fa_bwd_dq(q_g, k_g, v_g, do_g, dQd + off, 1, hg, N, d, causal, scale, ws, wsb, qs));
      ok(cudaEventRecord(cs->ev[EV_BWD0 + g], qs));
      run(fa_bwd_dkdv(q_g, k_g, v_g, do_g, dKd + off, dVd + off, 1, hg, N, d, causal, scale, ws, wsb, bs));
      ok(cudaEventRecord(cs->ev[EV_DKDV0 + g], bs));
    } else {
      run(fa_bwd_main(q_g, k_g, v_g, do_g, dKd + off, dVd + off, 1, hg, N, d, causal, scale, ws, wsb, bs));
      ok(cudaEventRecord(cs->ev[EV_DKDV0 + g], bs));
      run(fa_bwd_postprocess(dQd + off, 1, hg, N, d, ws, wsb, bs));
      ok(cudaEventRecord(cs->ev[EV_BWD0 + g], bs));
    }
    ok(cudaStreamWaitEvent(cs->d2h, cs->ev[EV_DKDV0 + g], 0));
    ok(cudaMemcpyAsync(hdk + off, dKd + off, n, D2H, cs->d2h));
    ok(cudaMemcpyAsync(hdv + off, dVd + off, n, D2H, cs->d2h));
    ok(cudaStreamWaitEvent(cs->d2h, cs->ev[EV_BWD0 + g], 0));
    ok(cudaMemcpyAsync(hdq + off, dQd + off, n, D2H, cs->d2h));
  }

  // Work queued on `stream` after this call sees the outputs in host memory.
  ok(cudaEventRecord(cs->ev[EV_DONE], cs->d2h));
  ok(cudaStreamWaitEvent(stream, cs->ev[EV_DONE], 0));
  if (st != FA_OK) return st;
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"

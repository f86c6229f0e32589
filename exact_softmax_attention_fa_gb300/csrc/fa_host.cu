// Host-buffer entry point: one forward and backward pass of a problem whose
// inputs and outputs live in host memory. The library owns two copy streams
// per device (host->device and device->host) and orders them against the
// caller's stream with events, so the copies overlap the kernels:
//
//   h2d:    Q,K,V heads chunk 0 | chunk 1 | ... | chunk C-1 | dO
//   stream:          fwd chunk 0 | fwd chunk 1 | ... | fwd C-1 | D, L2 | dK,dV | dQ part 0 | dQ part 1
//   d2h:                                                  O, L | dK, dV   | dQ part 0 | dQ part 1
//
// d = 128: the dQ kernel runs in two launches over the first three quarters
// and the last quarter of the heads, so only the last quarter of dQ is read
// back after the last kernel.
// The forward runs per chunk of heads as soon as that chunk is on the device
// (rows of different heads are independent problems, and a head's result does
// not depend on which launch computes it). The backward needs every head's
// dO before its first kernel, so it runs unchunked. Nothing here computes:
// the work is the same sequence of kernels fa_fwd and fa_bwd launch.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kFwdChunks = 4;

enum : int { EV_START, EV_DO, EV_FWD, EV_DKDV, EV_DQ0, EV_BWD, EV_DONE, EV_IN0, EV_COUNT = EV_IN0 + kFwdChunks };

constexpr int kFwdOnlyChunks = 8;  // fa_fwd_host: uploads, forwards and read-backs pipelined over 8 head chunks

struct CopyState {
  std::once_flag once;
  cudaError_t error = cudaSuccess;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t ev[EV_COUNT] = {};
  cudaEvent_t fwd_in[kFwdOnlyChunks] = {}, fwd_out[kFwdOnlyChunks] = {};
  std::mutex mu;  // one call at a time per device enqueues on the shared streams and events
};
CopyState g_copy[kMaxDevices];

CopyState* copy_state(int dev) {
  CopyState& cs = g_copy[dev];
  std::call_once(cs.once, [&cs] {
    cudaError_t e = cudaStreamCreateWithFlags(&cs.h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&cs.d2h, cudaStreamNonBlocking);
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

// Device buffer: q, k, v, dO, o, dq, dk, dv (bf16), lse (fp32), then the
// backward workspace; every part starts on a 256-byte boundary.
struct HostLayout {
  size_t q, k, v, dO, o, dq, dk, dv, lse, ws, ws_bytes, total;
};

HostLayout host_layout(int B, int H, int N, int d) {
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
  L.ws = off;
  L.ws_bytes = fa_bwd_workspace_size(B, H, N, d);
  L.total = off + align256(L.ws_bytes);
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
    ok(cudaStreamWaitEvent(stream, cs->fwd_in[c], 0));
    if (st == FA_OK && e == cudaSuccess)
      st = fa_fwd(Qd + off, Kd + off, Vd + off, Od + off, Ld + h0 * N, 1, static_cast<int>(h1 - h0), N, d, causal,
                  scale, stream);
    ok(cudaEventRecord(cs->fwd_out[c], stream));
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
  return fa::host_layout(B, H, N, d).total;
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
  const HostLayout L = host_layout(B, H, N, d);
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
  void* ws = base + L.ws;
  const long long BH = static_cast<long long>(B) * H;
  const size_t head_bytes = static_cast<size_t>(N) * d * 2, all_bytes = BH * head_bytes;
  const size_t lse_bytes = static_cast<size_t>(BH) * N * 4;
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
  const int chunks = static_cast<int>(std::min<long long>(kFwdChunks, BH));
  for (int c = 0; c < chunks; ++c) {
    const long long h0 = BH * c / chunks, h1 = BH * (c + 1) / chunks;
    const size_t off = h0 * head_bytes, n = (h1 - h0) * head_bytes;
    ok(cudaMemcpyAsync(Qd + off, hq + off, n, H2D, cs->h2d));
    ok(cudaMemcpyAsync(Kd + off, hk + off, n, H2D, cs->h2d));
    ok(cudaMemcpyAsync(Vd + off, hv + off, n, H2D, cs->h2d));
    ok(cudaEventRecord(cs->ev[EV_IN0 + c], cs->h2d));
  }
  ok(cudaMemcpyAsync(dOd, dO, all_bytes, H2D, cs->h2d));
  ok(cudaEventRecord(cs->ev[EV_DO], cs->h2d));

  // Forward, one launch per chunk of heads (a [1][h1 - h0] problem).
  for (int c = 0; c < chunks && e == cudaSuccess && st == FA_OK; ++c) {
    const long long h0 = BH * c / chunks, h1 = BH * (c + 1) / chunks;
    const size_t off = h0 * head_bytes;
    ok(cudaStreamWaitEvent(stream, cs->ev[EV_IN0 + c], 0));
    run(fa_fwd(Qd + off, Kd + off, Vd + off, Od + off, Ld + h0 * N, 1, static_cast<int>(h1 - h0), N, d,
               causal, scale, stream));
  }
  ok(cudaEventRecord(cs->ev[EV_FWD], stream));
  ok(cudaStreamWaitEvent(cs->d2h, cs->ev[EV_FWD], 0));
  ok(cudaMemcpyAsync(o, Od, all_bytes, D2H, cs->d2h));
  ok(cudaMemcpyAsync(lse, Ld, lse_bytes, D2H, cs->d2h));

  // Backward: the phases fa_bwd runs for this head dimension, with dK and dV
  // read back while dQ is still being computed.
  ok(cudaStreamWaitEvent(stream, cs->ev[EV_DO], 0));
  run(fa_bwd_preprocess(Od, Ld, dOd, B, H, N, d, ws, L.ws_bytes, stream));
  if (d == 128) {
    run(fa_bwd_dkdv(Qd, Kd, Vd, dOd, dKd, dVd, B, H, N, d, causal, scale, ws, L.ws_bytes, stream));
  } else {
    run(fa_bwd_main(Qd, Kd, Vd, dOd, dKd, dVd, B, H, N, d, causal, scale, ws, L.ws_bytes, stream));
  }
  ok(cudaEventRecord(cs->ev[EV_DKDV], stream));
  ok(cudaStreamWaitEvent(cs->d2h, cs->ev[EV_DKDV], 0));
  ok(cudaMemcpyAsync(dk, dKd, all_bytes, D2H, cs->d2h));
  ok(cudaMemcpyAsync(dv, dVd, all_bytes, D2H, cs->d2h));
  long long dq_first = BH;  // heads whose dQ is read back while the rest is computed
  if (d == 128) {
    dq_first = BH >= 4 ? BH - (BH + 3) / 4 : BH;
    run(bwd_dq_heads(Qd, Kd, Vd, dOd, dQd, B, H, N, d, causal, scale, ws, L.ws_bytes, 0, static_cast<int>(dq_first),
                     stream));
    if (dq_first < BH) {
      ok(cudaEventRecord(cs->ev[EV_DQ0], stream));
      ok(cudaStreamWaitEvent(cs->d2h, cs->ev[EV_DQ0], 0));
      ok(cudaMemcpyAsync(dq, dQd, dq_first * head_bytes, D2H, cs->d2h));
      run(bwd_dq_heads(Qd, Kd, Vd, dOd, dQd, B, H, N, d, causal, scale, ws, L.ws_bytes, static_cast<int>(dq_first),
                       static_cast<int>(BH - dq_first), stream));
    }
  } else {
    run(fa_bwd_postprocess(dQd, B, H, N, d, ws, L.ws_bytes, stream));
  }
  const long long dq_rest = d == 128 && dq_first < BH ? dq_first : 0;  // heads already read back
  ok(cudaEventRecord(cs->ev[EV_BWD], stream));
  ok(cudaStreamWaitEvent(cs->d2h, cs->ev[EV_BWD], 0));
  ok(cudaMemcpyAsync(static_cast<uint8_t*>(dq) + dq_rest * head_bytes, dQd + dq_rest * head_bytes,
                     (BH - dq_rest) * head_bytes, D2H, cs->d2h));

  // Work queued on `stream` after this call sees the outputs in host memory.
  ok(cudaEventRecord(cs->ev[EV_DONE], cs->d2h));
  ok(cudaStreamWaitEvent(stream, cs->ev[EV_DONE], 0));
  if (st != FA_OK) return st;
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"

// Forward pass of exact softmax attention for sm_103a: launches of the kernel
// in fa_fwd_kernel.cuh with one query head per tile, and the combine kernel
// that merges split key ranges.
#include "fa_fwd_kernel.cuh"

namespace fa {

namespace {

// Merge of the key ranges' partials (reading note 5.2: the running max and
// sum make softmax blocks combinable; the same identity merges whole ranges):
// with L_s and O_s of range s, each normalised by its own sum,
//   L = log sum_s e^{L_s},   O = sum_s e^{L_s - L} O_s.
// One warp per query row, HD / 32 consecutive columns per lane; ranges that
// hold no key the row sees are not read. HBM-bound.
template <int HD>
__global__ void __launch_bounds__(256) fwd_combine_kernel(const float* __restrict__ o_part,
                                                          const float* __restrict__ lse_part,
                                                          __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                                                          int BH, int Nq, int Nk, int causal, int causal_off,
                                                          int splits, int keys_per_split) {
  constexpr int PER = HD / 32;
  // Launched to overlap the forward's last round: its partials are final
  // only once that grid has completed.
  griddep_wait();
  const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= static_cast<long long>(BH) * Nq) return;
  const int i = static_cast<int>(row % Nq);
  const int last_key = causal ? min(Nk - 1, i + causal_off) : Nk - 1;
  const int n = min(splits, last_key / keys_per_split + 1);
  const size_t plane = static_cast<size_t>(BH) * Nq;
  float m = -INFINITY;
  for (int s = 0; s < n; ++s) m = fmaxf(m, __ldg(lse_part + s * plane + row));
  float acc[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) acc[k] = 0.f;
  float sum = 0.f;
  for (int s = 0; s < n; ++s) {
    const float wgt = expf(__ldg(lse_part + s * plane + row) - m);
    sum += wgt;
    const float* src = o_part + (s * plane + row) * HD + lane * PER;
#pragma unroll
    for (int k = 0; k < PER; k += 2) {
      const float2 v = __ldg(reinterpret_cast<const float2*>(src + k));
      acc[k] = fmaf(wgt, v.x, acc[k]);
      acc[k + 1] = fmaf(wgt, v.y, acc[k + 1]);
    }
  }
  const float inv = 1.f / sum;
  uint32_t packed[PER / 2];
#pragma unroll
  for (int k = 0; k < PER; k += 2) packed[k / 2] = pack_bf16x2(acc[k] * inv, acc[k + 1] * inv);
  __nv_bfloat16* dst = o + row * HD + lane * PER;
  if constexpr (PER == 2) {
    *reinterpret_cast<uint32_t*>(dst) = packed[0];
  } else if constexpr (PER == 4) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
  } else {
    *reinterpret_cast<uint4*>(dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  }
  if (lane == 0) lse[row] = m + logf(sum);
}

template <int HD>
cudaError_t launch_combine_t(const FwdLaunch& a, cudaStream_t stream) {
  const long long threads = static_cast<long long>(a.BH) * a.Nq * 32;
  // Programmatic dependent launch: the forward (splits > 1) signals at its
  // start, so these blocks are queued as its CTAs leave SMs and wait in
  // griddep_wait for its completion instead of for a launch after it.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((threads + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fwd_combine_kernel<HD>, static_cast<const float*>(a.o_part),
                            static_cast<const float*>(a.lse_part), a.o, a.lse, a.BH, a.Nq, a.Nk, a.causal,
                            a.causal_off, a.splits, a.kv_per_split * 128);
}

}  // namespace

cudaError_t launch_fwd_combine(const FwdLaunch& a, cudaStream_t stream) {
  switch (a.d) {
    case 64: return launch_combine_t<64>(a, stream);
    case 128: return launch_combine_t<128>(a, stream);
    case 256: return launch_combine_t<256>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_fwd(const FwdLaunch& a, cudaStream_t stream) {
  if (a.pack > 1) return launch_fwd_packed(a, stream);
  switch (a.d) {
    case 64: return a.causal ? launch_fwd_t<64, true, false>(a, stream) : launch_fwd_t<64, false, false>(a, stream);
    case 128: return a.causal ? launch_fwd_t<128, true, false>(a, stream) : launch_fwd_t<128, false, false>(a, stream);
    case 256: return a.causal ? launch_fwd_t<256, true, false>(a, stream) : launch_fwd_t<256, false, false>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fa

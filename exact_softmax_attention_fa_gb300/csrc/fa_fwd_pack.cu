// Forward pass with grouped query heads packed into a tile (short query
// blocks such as decoding): instantiations of the kernel in
// fa_fwd_kernel.cuh, compiled apart from the unpacked ones.
#include "fa_fwd_kernel.cuh"

namespace fa {

cudaError_t launch_fwd_packed(const FwdLaunch& a, cudaStream_t stream) {
  switch (a.d) {
    case 64: return a.causal ? launch_fwd_t<64, true, true>(a, stream) : launch_fwd_t<64, false, true>(a, stream);
    case 128: return a.causal ? launch_fwd_t<128, true, true>(a, stream) : launch_fwd_t<128, false, true>(a, stream);
    case 256: return a.causal ? launch_fwd_t<256, true, true>(a, stream) : launch_fwd_t<256, false, true>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fa

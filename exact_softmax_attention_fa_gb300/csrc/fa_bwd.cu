// Backward pass (placeholder until the kernels land).
#include "fa_internal.h"

namespace fa {
cudaError_t launch_bwd(const BwdLaunch&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace fa

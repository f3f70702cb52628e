// Backward pass (placeholder until the kernels land): reports "not supported".
#include "fa_internal.h"

namespace fa {
cudaError_t launch_bwd(const BwdLaunch&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace fa

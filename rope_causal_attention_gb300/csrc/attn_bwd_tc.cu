// Tensor-core backward (placeholder until the tcgen05 kernels land).
#include <cuda_runtime.h>

#include "internal.h"

namespace ra {
cudaError_t launch_attn_bwd_tc(const BwdArgs &, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace ra

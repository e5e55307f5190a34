// Tensor-core decode split kernel (placeholder until the tcgen05 variant lands).
#include <cuda_runtime.h>

#include "internal.h"

namespace ra {
cudaError_t launch_attn_decode_tc(const DecodeArgs &, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace ra

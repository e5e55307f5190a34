// Tensor-core (tcgen05) causal attention with RoPE fused in.
#include <cuda_runtime.h>

#include "internal.h"

namespace ra {
cudaError_t launch_attn_tc(const AttnArgs &, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace ra

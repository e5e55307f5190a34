// Tensor maps (TMA descriptors) for the tensor-core kernels: 16-bit tensors
// whose rows of D elements are contiguous, addressed by up to three outer
// coordinates.  Host code only.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "internal.h"

namespace ra {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's encoder, looked up once through the runtime (no -lcuda).
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

}  // namespace

cudaError_t make_row_tile_map(const void *base, bool bf16, int D, int n_outer,
                              const int64_t size[3], const int64_t stride[3], CUtensorMap *map,
                              int perm[3]) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  if (n_outer < 1 || n_outer > 3) return cudaErrorInvalidValue;
  struct Dim { uint64_t size, stride; int logical; };
  Dim d[3];
  for (int i = 0; i < n_outer; ++i) d[i] = {(uint64_t)size[i], (uint64_t)stride[i] * 2, i};
  // increasing stride, size-1 dims last (their stride is never used)
  std::stable_sort(d, d + n_outer, [](const Dim &x, const Dim &y) {
    if ((x.size == 1) != (y.size == 1)) return y.size == 1;
    return x.stride < y.stride;
  });
  uint64_t prev_extent = (uint64_t)D * 2;
  for (int i = 0; i < n_outer; ++i) {
    if (d[i].size == 1 || d[i].stride == 0) d[i].stride = (prev_extent + 15) & ~uint64_t(15);
    prev_extent = d[i].stride * d[i].size;
    perm[i] = d[i].logical;
  }
  cuuint64_t gdim[4] = {(cuuint64_t)D, 1, 1, 1};
  cuuint64_t gstride[3] = {0, 0, 0};
  cuuint32_t box[4] = {64, 1, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  for (int i = 0; i < n_outer; ++i) {
    gdim[1 + i] = d[i].size;
    gstride[i] = d[i].stride;
    if (d[i].logical == 0) box[1 + i] = 128;  // 128 rows, whichever map dim holds them
  }
  const CUtensorMapDataType t =
      bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUresult r = enc(map, t, (cuuint32_t)(1 + n_outer), const_cast<void *>(base), gdim,
                         gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace ra

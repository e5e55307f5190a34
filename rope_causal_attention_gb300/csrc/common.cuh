// Small device helpers shared by the kernels: element conversion and status
// recording.  Tensor-core specific PTX lives in tc_ptx.cuh.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ra {

__device__ __forceinline__ void record_status(int *status, int code) {
  if (status) atomicCAS(status, 0, code);
}

template <typename T> struct Elem;
template <> struct Elem<float> {
  static __device__ __forceinline__ float load(float x) { return x; }
  static __device__ __forceinline__ float store(float x) { return x; }
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float load(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 store(float x) { return __float2bfloat16_rn(x); }
};
template <> struct Elem<__half> {
  static __device__ __forceinline__ float load(__half x) { return __half2float(x); }
  static __device__ __forceinline__ __half store(float x) { return __float2half_rn(x); }
};

__device__ __forceinline__ int64_t load_position(const void *positions, int is64, int64_t t) {
  return is64 ? static_cast<const int64_t *>(positions)[t]
              : static_cast<int64_t>(static_cast<const int32_t *>(positions)[t]);
}

}  // namespace ra

// Small device helpers shared by the kernels: element conversion and status
// recording.  Tensor-core specific PTX lives in tc_ptx.cuh.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/rope_attn.h"

namespace ra {

__device__ __forceinline__ void record_status(int *status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// Nonzero when either fp16 half of w is an infinity or a NaN (exponent field
// all ones): adding one to a saturated 5-bit exponent carries into the sign
// position of that half.
__device__ __forceinline__ uint32_t f16x2_nonfinite(uint32_t w) {
  return ((w & 0x7c007c00u) + 0x04000400u) & 0x80008000u;
}

// Records RA_ERR_RANGE once per warp when any lane's flag is set.
__device__ __forceinline__ void record_range_flag(int *status, uint32_t flag) {
  if (__any_sync(0xffffffffu, flag != 0u) && (threadIdx.x & 31) == 0)
    record_status(status, RA_ERR_RANGE);
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

// 16-byte vector access: VecN<T>::N elements per uint4.
template <typename T> struct VecN { static constexpr int N = 16 / (int)sizeof(T); };

template <typename T>
__device__ __forceinline__ void unpack16(const uint4 &u, float *f) {
  const T *e = reinterpret_cast<const T *>(&u);
#pragma unroll
  for (int i = 0; i < VecN<T>::N; ++i) f[i] = Elem<T>::load(e[i]);
}

template <typename T>
__device__ __forceinline__ uint4 pack16(const float *f) {
  uint4 u;
  T *e = reinterpret_cast<T *>(&u);
#pragma unroll
  for (int i = 0; i < VecN<T>::N; ++i) e[i] = Elem<T>::store(f[i]);
  return u;
}

// Loads n consecutive fp32 table values (n = 2, 4 or 8) starting at p.
template <int n>
__device__ __forceinline__ void load_table(const float *__restrict__ p, float *out) {
  if constexpr (n == 2) {
    const float2 a = __ldg(reinterpret_cast<const float2 *>(p));
    out[0] = a.x; out[1] = a.y;
  } else {
#pragma unroll
    for (int j = 0; j < n / 4; ++j) {
      const float4 a = __ldg(reinterpret_cast<const float4 *>(p) + j);
      out[4 * j] = a.x; out[4 * j + 1] = a.y; out[4 * j + 2] = a.z; out[4 * j + 3] = a.w;
    }
  }
}

}  // namespace ra

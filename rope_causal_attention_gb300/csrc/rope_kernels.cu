// RoPE table build and the standalone Q+K rotation (decode / continuous
// batching).
//
// What is computed ("Write Triton Rope Kernel", Required reasoning process
// steps 1-10 and Kernel design rules; "RoPE and FlashAttention: relative
// positions and online softmax", sections 1-2):
//   theta_i = base^(-2i/F); table row p holds cos/sin(p * theta_i), fp32.
//   NeoX pairs (i, i + r/2), GPT-J pairs (2i, 2i+1), i < r/2:
//     lo' = lo*c - hi*s,  hi' = hi*c + lo*s   (fp32, rounded once on store).
//   Positions come from positions[t]; dims past rot_dim stay untouched.
//
// GB300 design: the rotation is a pure stream (read Q/K once, write once), so
// it is bound by HBM bandwidth.  Each thread owns one 16-byte slice (NeoX: a
// 16-byte piece of the low half plus the matching piece of the high half;
// GPT-J: 16 contiguous bytes, i.e. whole pairs) of up to four heads of one
// token: threadIdx.x = slice, threadIdx.y = head group, threadIdx.z = token
// within the block, so a warp touches consecutive slices of consecutive heads
// -- contiguous 128-bit accesses.  A thread issues all its heads' loads before
// its first store, and loads the token's cos/sin slice once (read-only path)
// for all of them; Q and K heads share one launch.  Q/K rows are read and
// written with the streaming (evict-first) cache hint: each is touched once,
// so they should not displace the cos/sin rows that nearby tokens share.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace ra {
namespace {

// ------------------------------------------------------------------ tables
__global__ void rope_table_build_kernel(float *__restrict__ cos_out,
                                        float *__restrict__ sin_out, int64_t rows, int half,
                                        double base, int F, double pos_scale) {
  const int64_t n = rows * half;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < n;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t p = idx / half;
    const int i = (int)(idx - p * half);
    const double theta = pow(base, -(2.0 * i) / (double)F);
    const double angle = ((double)p / pos_scale) * theta;  // p / 1.0 == p exactly
    double s, c;
    sincos(angle, &s, &c);
    cos_out[idx] = (float)c;
    sin_out[idx] = (float)s;
  }
}

// ------------------------------------------------------------ rope (vector)
struct RopeKParams {
  void *q, *k, *qo, *ko;
  int64_t sq_t, sq_h, sk_t, sk_h, sqo_t, sqo_h, sko_t, sko_h;
  int64_t T;
  int Hq, Htot, half, rot_dim, s_rot, s_tail;
  const void *positions;
  int is64;
  const float *cos_t, *sin_t;
  int64_t table_rows;
  int *status;
};

// Heads handled by one thread per token, loaded together before any store
// (in place, a store may alias a later head's load, so the compiler cannot
// overlap heads on its own).
constexpr int kHeadsPerThread = 4;

template <typename T, int LAYOUT>
__global__ void __launch_bounds__(512) rope_apply_vec_kernel(RopeKParams p) {
  constexpr int V = VecN<T>::N;                         // elements per 16 bytes
  constexpr int NP = (LAYOUT == RA_NEOX) ? V : V / 2;   // pairs per slice
  constexpr int NH = kHeadsPerThread;
  constexpr int LD = (LAYOUT == RA_NEOX) ? 2 : 1;       // 16-byte loads per head
  const int s = threadIdx.x;
  const int hy = blockDim.y;  // heads of a token are h = threadIdx.y + k * hy, k < NH
  const bool rot_slice = s < p.s_rot, tail_slice = !rot_slice && s < p.s_rot + p.s_tail;
  const int i0 = s * NP;  // first pair index of a rotated slice
  // NeoX: low-half and high-half pieces; GPT-J: whole pairs; tail: a copy
  const int off0 = rot_slice ? ((LAYOUT == RA_NEOX) ? i0 : 2 * i0) : p.rot_dim + (s - p.s_rot) * V;
  const int off1 = i0 + p.half;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.z + threadIdx.z; t < p.T;
       t += (int64_t)gridDim.x * blockDim.z) {
    const T *src[NH];
    T *dst[NH];
    bool ok[NH];
#pragma unroll
    for (int k = 0; k < NH; ++k) {
      const int h = threadIdx.y + k * hy;
      ok[k] = h < p.Htot;
      const bool isq = h < p.Hq;
      const int hh = isq ? h : h - p.Hq;
      src[k] = static_cast<const T *>(isq ? p.q : p.k) + t * (isq ? p.sq_t : p.sk_t) +
               hh * (isq ? p.sq_h : p.sk_h);
      dst[k] = static_cast<T *>(isq ? p.qo : p.ko) + t * (isq ? p.sqo_t : p.sko_t) +
               hh * (isq ? p.sqo_h : p.sko_h);
    }
    // the token's rows are read before its position, so that the position
    // (and then the cos/sin row) is fetched while the rows are in flight
    uint4 raw[NH][LD];
#pragma unroll
    for (int k = 0; k < NH; ++k) {
      if (!ok[k] || !(rot_slice || tail_slice)) continue;
      raw[k][0] = __ldcs(reinterpret_cast<const uint4 *>(src[k] + off0));
      if (LD == 2 && rot_slice) raw[k][LD - 1] = __ldcs(reinterpret_cast<const uint4 *>(src[k] + off1));
    }
    const int64_t pos = load_position(p.positions, p.is64, t);
    if (pos < 0 || pos >= p.table_rows) {
      if (s == 0 && threadIdx.y == 0) record_status(p.status, RA_ERR_POSITION_RANGE);
      continue;
    }
    if (rot_slice) {
      float c[NP], sn[NP];
      load_table<NP>(p.cos_t + pos * p.half + i0, c);
      load_table<NP>(p.sin_t + pos * p.half + i0, sn);
#pragma unroll
      for (int k = 0; k < NH; ++k) {
        if (!ok[k]) continue;
        if constexpr (LAYOUT == RA_NEOX) {
          float lo[V], hi[V], olo[V], ohi[V];
          unpack16<T>(raw[k][0], lo);
          unpack16<T>(raw[k][LD - 1], hi);
#pragma unroll
          for (int j = 0; j < V; ++j) {
            olo[j] = lo[j] * c[j] - hi[j] * sn[j];
            ohi[j] = hi[j] * c[j] + lo[j] * sn[j];
          }
          __stcs(reinterpret_cast<uint4 *>(dst[k] + off0), pack16<T>(olo));
          __stcs(reinterpret_cast<uint4 *>(dst[k] + off1), pack16<T>(ohi));
        } else {
          float x[V], y[V];
          unpack16<T>(raw[k][0], x);
#pragma unroll
          for (int j = 0; j < NP; ++j) {
            y[2 * j] = x[2 * j] * c[j] - x[2 * j + 1] * sn[j];
            y[2 * j + 1] = x[2 * j + 1] * c[j] + x[2 * j] * sn[j];
          }
          __stcs(reinterpret_cast<uint4 *>(dst[k] + off0), pack16<T>(y));
        }
      }
    } else if (tail_slice) {  // out of place: copy the unrotated tail
#pragma unroll
      for (int k = 0; k < NH; ++k)
        if (ok[k]) __stcs(reinterpret_cast<uint4 *>(dst[k] + off0), raw[k][0]);
    }
  }
}

// ------------------------------------------------------------ rope (scalar)
// Any even D / rot_dim, any alignment: one thread per (pair or tail element,
// head) of a token.
template <typename T>
__global__ void __launch_bounds__(256) rope_apply_scalar_kernel(RopeKParams p, int layout,
                                                                int tail) {
  const int per_head = p.half + tail;
  for (int64_t t = blockIdx.x; t < p.T; t += gridDim.x) {
    const int64_t pos = load_position(p.positions, p.is64, t);
    if (pos < 0 || pos >= p.table_rows) {
      if (threadIdx.x == 0 && threadIdx.y == 0) record_status(p.status, RA_ERR_POSITION_RANGE);
      continue;
    }
    for (int h = threadIdx.y; h < p.Htot; h += blockDim.y) {
      const bool isq = h < p.Hq;
      const int hh = isq ? h : h - p.Hq;
      const T *src = static_cast<const T *>(isq ? p.q : p.k) + t * (isq ? p.sq_t : p.sk_t) +
                     hh * (isq ? p.sq_h : p.sk_h);
      T *dst = static_cast<T *>(isq ? p.qo : p.ko) + t * (isq ? p.sqo_t : p.sko_t) +
               hh * (isq ? p.sqo_h : p.sko_h);
      for (int j = threadIdx.x; j < per_head; j += blockDim.x) {
        if (j < p.half) {
          const int lo = layout == RA_NEOX ? j : 2 * j;
          const int hi = layout == RA_NEOX ? j + p.half : 2 * j + 1;
          const float c = __ldg(p.cos_t + pos * p.half + j);
          const float sn = __ldg(p.sin_t + pos * p.half + j);
          const float a = Elem<T>::load(src[lo]), b = Elem<T>::load(src[hi]);
          dst[lo] = Elem<T>::store(a * c - b * sn);
          dst[hi] = Elem<T>::store(b * c + a * sn);
        } else {
          const int e = p.rot_dim + (j - p.half);
          dst[e] = src[e];
        }
      }
    }
  }
}


template <typename T>
cudaError_t launch_vec(const RopeKParams &kp, ra_layout layout, cudaStream_t s) {
  const int slices = kp.s_rot + kp.s_tail;
  // every head of a token must be reachable: blockDim.y * kHeadsPerThread >= Htot
  const int hy = (kp.Htot + kHeadsPerThread - 1) / kHeadsPerThread;
  if (slices * hy > 512) return cudaErrorNotSupported;
  // several tokens per block (z) so that a block has ~256 threads
  int tz = 256 / (slices * hy);
  if (tz < 1) tz = 1;
  if (tz > 64) tz = 64;
  const dim3 block(slices, hy, tz);
  const int64_t max_grid = (int64_t)sm_count_current() * 64;
  const int64_t need = (kp.T + tz - 1) / tz;
  const unsigned grid = (unsigned)(need < max_grid ? need : max_grid);
  if (layout == RA_NEOX)
    rope_apply_vec_kernel<T, RA_NEOX><<<grid, block, 0, s>>>(kp);
  else
    rope_apply_vec_kernel<T, RA_GPTJ><<<grid, block, 0, s>>>(kp);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_scalar(const RopeKParams &kp, ra_layout layout, int tail, cudaStream_t s) {
  const dim3 block(32, 8);
  const int64_t max_grid = (int64_t)sm_count_current() * 64;
  const unsigned grid = (unsigned)(kp.T < max_grid ? kp.T : max_grid);
  rope_apply_scalar_kernel<T><<<grid, block, 0, s>>>(kp, (int)layout, tail);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_table_build(const TableArgs &a, cudaStream_t s) {
  const int half = a.rot_dim / 2;
  const int F = a.freq_dim > 0 ? a.freq_dim : a.rot_dim;
  const int64_t n = a.rows * half;
  if (n == 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = (int64_t)sm_count_current() * 32;
  if (blocks > cap) blocks = cap;
  rope_table_build_kernel<<<(unsigned)blocks, 256, 0, s>>>(a.cos_out, a.sin_out, a.rows, half,
                                                          a.base, F, a.pos_scale);
  return cudaGetLastError();
}

cudaError_t launch_rope_apply(const RopeArgs &a, bool vectorized, cudaStream_t s) {
  RopeKParams kp{};
  const bool qin = a.q_out == nullptr || a.q_out == a.q;
  const bool kin = a.k_out == nullptr || a.k_out == a.k;
  kp.q = a.q; kp.k = a.k;
  kp.qo = qin ? a.q : a.q_out;
  kp.ko = kin ? a.k : a.k_out;
  kp.sq_t = a.sq[0]; kp.sq_h = a.sq[1];
  kp.sk_t = a.sk[0]; kp.sk_h = a.sk[1];
  kp.sqo_t = qin ? a.sq[0] : a.sqo[0]; kp.sqo_h = qin ? a.sq[1] : a.sqo[1];
  kp.sko_t = kin ? a.sk[0] : a.sko[0]; kp.sko_h = kin ? a.sk[1] : a.sko[1];
  kp.T = a.T; kp.Hq = a.Hq; kp.Htot = a.Hq + a.Hkv;
  kp.half = a.rot_dim / 2; kp.rot_dim = a.rot_dim;
  kp.positions = a.positions; kp.is64 = a.pos_is_int64;
  kp.cos_t = a.cos_t; kp.sin_t = a.sin_t; kp.table_rows = a.table_rows;
  kp.status = a.status;
  // Out of place (for either tensor) copies the tail; the in-place tensor then
  // copies its tail onto itself, which is harmless.
  const bool copy_tail = !(qin && kin);
  const int tail = copy_tail ? (a.D - a.rot_dim) : 0;
  if (a.T == 0 || kp.Htot == 0) return cudaSuccess;
  if (vectorized) {
    const int es = a.dt == RA_F32 ? 4 : 2;
    const int V = 16 / es;
    kp.s_rot = a.layout == RA_NEOX ? kp.half / V : a.rot_dim / V;
    kp.s_tail = tail / V;
    const int hy = (kp.Htot + kHeadsPerThread - 1) / kHeadsPerThread;
    vectorized = (kp.s_rot + kp.s_tail) * hy <= 512;  // else the scalar kernel
  }
  if (vectorized) {
    switch (a.dt) {
      case RA_F32: return launch_vec<float>(kp, a.layout, s);
      case RA_BF16: return launch_vec<__nv_bfloat16>(kp, a.layout, s);
      default: return launch_vec<__half>(kp, a.layout, s);
    }
  }
  switch (a.dt) {
    case RA_F32: return launch_scalar<float>(kp, a.layout, tail, s);
    case RA_BF16: return launch_scalar<__nv_bfloat16>(kp, a.layout, tail, s);
    default: return launch_scalar<__half>(kp, a.layout, tail, s);
  }
}

}  // namespace ra

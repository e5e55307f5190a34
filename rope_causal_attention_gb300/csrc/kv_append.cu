// Decoder-step KV append: rotate the new tokens' Q, write their rotated K and
// raw V into the KV cache ("RoPE and FlashAttention: relative positions and
// online softmax", section 2: new K is cached already rotated, V is never
// rotated, cached K is never rotated again; positions come from the cache
// position of each token).
//
// Same rotation as rope_apply_qk (section 1; "Write Triton Rope Kernel",
// Kernel design rules): NeoX pairs (i, i + r/2) or GPT-J pairs (2i, 2i+1),
// fp32 arithmetic, one rounding on store; dims past rot_dim copied.
//
// GB300 design: a pure stream like rope_apply (read each new row once, write
// it once), so the same thread layout: one 16-byte slice of up to four heads
// per thread, threadIdx.x = slice, threadIdx.y = head group, threadIdx.z =
// token.  The heads of a token are its Hq query heads, then Hkv key heads,
// then Hkv value heads; a value head takes the rotation slices' bytes
// unrotated.  The cache row of a token is computed once per token.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace ra {
namespace {

struct AppendKParams {
  void *q, *qo;
  const void *kn, *vn;
  void *kc, *vc;
  int64_t sq_t, sq_h, sqo_t, sqo_h, skn_t, skn_h, svn_t, svn_h, skc_r, skc_h, svc_r, svc_h;
  int64_t T;
  int Hq, Hkv, Htot, half, rot_dim, s_rot, s_tail, q_inplace;
  const int32_t *seq_ids;
  const int64_t *seq_start;
  int64_t n_seqs, cache_rows;
  const void *positions;
  int is64;
  const float *cos_t, *sin_t;
  int64_t table_rows;
  int *status;
};

// Position and cache row of token t; false (and a recorded error) when the
// token has no valid sequence, table row or cache row.
__device__ __forceinline__ bool token_rows(const AppendKParams &p, int64_t t, bool report,
                                           int64_t *pos, int64_t *row) {
  const int64_t sq = p.seq_ids ? (int64_t)p.seq_ids[t] : t;
  *pos = load_position(p.positions, p.is64, t);
  bool ok = sq >= 0 && sq < p.n_seqs && *pos >= 0 && *pos < p.table_rows;
  if (ok) {
    *row = p.seq_start[sq] + *pos;
    ok = *row >= 0 && *row < p.cache_rows;
  }
  if (!ok && report) record_status(p.status, RA_ERR_POSITION_RANGE);
  return ok;
}

// Source and destination of head h (class q / k / v) of token t at cache row `row`.
template <typename T>
__device__ __forceinline__ void head_ptrs(const AppendKParams &p, int h, int64_t t, int64_t row,
                                          const T **src, T **dst, int *cls) {
  if (h < p.Hq) {
    *cls = 0;
    *src = static_cast<const T *>(p.q) + t * p.sq_t + h * p.sq_h;
    *dst = static_cast<T *>(p.qo) + t * p.sqo_t + h * p.sqo_h;
  } else if (h < p.Hq + p.Hkv) {
    const int hh = h - p.Hq;
    *cls = 1;
    *src = static_cast<const T *>(p.kn) + t * p.skn_t + hh * p.skn_h;
    *dst = static_cast<T *>(p.kc) + row * p.skc_r + hh * p.skc_h;
  } else {
    const int hh = h - p.Hq - p.Hkv;
    *cls = 2;
    *src = static_cast<const T *>(p.vn) + t * p.svn_t + hh * p.svn_h;
    *dst = static_cast<T *>(p.vc) + row * p.svc_r + hh * p.svc_h;
  }
}

constexpr int kHeadsPerThread = 4;

template <typename T, int LAYOUT>
__global__ void __launch_bounds__(512) rope_append_vec_kernel(AppendKParams p) {
  constexpr int V = VecN<T>::N;
  constexpr int NP = (LAYOUT == RA_NEOX) ? V : V / 2;
  constexpr int NH = kHeadsPerThread;
  constexpr int LD = (LAYOUT == RA_NEOX) ? 2 : 1;
  const int s = threadIdx.x;
  const int hy = blockDim.y;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.z + threadIdx.z; t < p.T;
       t += (int64_t)gridDim.x * blockDim.z) {
    int64_t pos, row;
    if (!token_rows(p, t, s == 0 && threadIdx.y == 0, &pos, &row)) continue;
    const T *src[NH];
    T *dst[NH];
    int cls[NH];
    bool ok[NH];
#pragma unroll
    for (int k = 0; k < NH; ++k) {
      const int h = threadIdx.y + k * hy;
      ok[k] = h < p.Htot;
      head_ptrs<T>(p, ok[k] ? h : 0, t, row, &src[k], &dst[k], &cls[k]);
    }
    if (s < p.s_rot) {
      const int i0 = s * NP;
      const int off0 = (LAYOUT == RA_NEOX) ? i0 : 2 * i0;
      const int off1 = i0 + p.half;
      uint4 raw[NH][LD];
#pragma unroll
      for (int k = 0; k < NH; ++k) {
        if (!ok[k]) continue;
        raw[k][0] = *reinterpret_cast<const uint4 *>(src[k] + off0);
        if (LD == 2) raw[k][LD - 1] = *reinterpret_cast<const uint4 *>(src[k] + off1);
      }
      float c[NP], sn[NP];
      load_table<NP>(p.cos_t + pos * p.half + i0, c);
      load_table<NP>(p.sin_t + pos * p.half + i0, sn);
#pragma unroll
      for (int k = 0; k < NH; ++k) {
        if (!ok[k]) continue;
        if (cls[k] == 2) {  // V: unrotated
          *reinterpret_cast<uint4 *>(dst[k] + off0) = raw[k][0];
          if (LD == 2) *reinterpret_cast<uint4 *>(dst[k] + off1) = raw[k][LD - 1];
          continue;
        }
        if constexpr (LAYOUT == RA_NEOX) {
          float lo[V], hi[V], olo[V], ohi[V];
          unpack16<T>(raw[k][0], lo);
          unpack16<T>(raw[k][LD - 1], hi);
#pragma unroll
          for (int j = 0; j < V; ++j) {
            olo[j] = lo[j] * c[j] - hi[j] * sn[j];
            ohi[j] = hi[j] * c[j] + lo[j] * sn[j];
          }
          *reinterpret_cast<uint4 *>(dst[k] + off0) = pack16<T>(olo);
          *reinterpret_cast<uint4 *>(dst[k] + off1) = pack16<T>(ohi);
        } else {
          float x[V], y[V];
          unpack16<T>(raw[k][0], x);
#pragma unroll
          for (int j = 0; j < NP; ++j) {
            y[2 * j] = x[2 * j] * c[j] - x[2 * j + 1] * sn[j];
            y[2 * j + 1] = x[2 * j + 1] * c[j] + x[2 * j] * sn[j];
          }
          *reinterpret_cast<uint4 *>(dst[k] + off0) = pack16<T>(y);
        }
      }
    } else if (s < p.s_rot + p.s_tail) {  // dims past rot_dim: copied (not for in-place Q)
      const int e0 = p.rot_dim + (s - p.s_rot) * V;
      uint4 raw[NH];
      bool cp[NH];
#pragma unroll
      for (int k = 0; k < NH; ++k) {
        cp[k] = ok[k] && !(cls[k] == 0 && p.q_inplace);
        if (cp[k]) raw[k] = *reinterpret_cast<const uint4 *>(src[k] + e0);
      }
#pragma unroll
      for (int k = 0; k < NH; ++k)
        if (cp[k]) *reinterpret_cast<uint4 *>(dst[k] + e0) = raw[k];
    }
  }
}

// Any even D / rot_dim, any alignment: one thread per (pair or tail element,
// head) of a token.
template <typename T>
__global__ void __launch_bounds__(256) rope_append_scalar_kernel(AppendKParams p, int layout,
                                                                 int tail) {
  const int per_head = p.half + tail;
  for (int64_t t = blockIdx.x; t < p.T; t += gridDim.x) {
    int64_t pos, row;
    if (!token_rows(p, t, threadIdx.x == 0 && threadIdx.y == 0, &pos, &row)) continue;
    for (int h = threadIdx.y; h < p.Htot; h += blockDim.y) {
      const T *src;
      T *dst;
      int cls;
      head_ptrs<T>(p, h, t, row, &src, &dst, &cls);
      for (int j = threadIdx.x; j < per_head; j += blockDim.x) {
        if (j < p.half) {
          const int lo = layout == RA_NEOX ? j : 2 * j;
          const int hi = layout == RA_NEOX ? j + p.half : 2 * j + 1;
          if (cls == 2) {
            dst[lo] = src[lo];
            dst[hi] = src[hi];
            continue;
          }
          const float c = __ldg(p.cos_t + pos * p.half + j);
          const float sn = __ldg(p.sin_t + pos * p.half + j);
          const float a = Elem<T>::load(src[lo]), b = Elem<T>::load(src[hi]);
          dst[lo] = Elem<T>::store(a * c - b * sn);
          dst[hi] = Elem<T>::store(b * c + a * sn);
        } else if (!(cls == 0 && p.q_inplace)) {
          const int e = p.rot_dim + (j - p.half);
          dst[e] = src[e];
        }
      }
    }
  }
}

template <typename T>
cudaError_t launch_vec(const AppendKParams &kp, ra_layout layout, cudaStream_t s) {
  const int slices = kp.s_rot + kp.s_tail;
  const int hy = (kp.Htot + kHeadsPerThread - 1) / kHeadsPerThread;
  int tz = 256 / (slices * hy);
  if (tz < 1) tz = 1;
  if (tz > 64) tz = 64;
  const dim3 block(slices, hy, tz);
  const int64_t max_grid = (int64_t)sm_count_current() * 64;
  const int64_t need = (kp.T + tz - 1) / tz;
  const unsigned grid = (unsigned)(need < max_grid ? need : max_grid);
  if (layout == RA_NEOX)
    rope_append_vec_kernel<T, RA_NEOX><<<grid, block, 0, s>>>(kp);
  else
    rope_append_vec_kernel<T, RA_GPTJ><<<grid, block, 0, s>>>(kp);
  note_launch("rope_append_vec_kernel");
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_scalar(const AppendKParams &kp, ra_layout layout, int tail, cudaStream_t s) {
  const dim3 block(32, 8);
  const int64_t max_grid = (int64_t)sm_count_current() * 64;
  const unsigned grid = (unsigned)(kp.T < max_grid ? kp.T : max_grid);
  rope_append_scalar_kernel<T><<<grid, block, 0, s>>>(kp, (int)layout, tail);
  note_launch("rope_append_scalar_kernel");
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_typed(const AppendKParams &kp, const AppendArgs &a, bool vectorized,
                         cudaStream_t s) {
  const int tail = a.D - a.rot_dim;
  if (vectorized) {
    const int V = VecN<T>::N;
    AppendKParams v = kp;
    v.s_rot = a.layout == RA_NEOX ? kp.half / V : a.rot_dim / V;
    v.s_tail = tail / V;
    const int hy = (kp.Htot + kHeadsPerThread - 1) / kHeadsPerThread;
    if ((v.s_rot + v.s_tail) * hy <= 512) return launch_vec<T>(v, a.layout, s);
  }
  return launch_scalar<T>(kp, a.layout, tail, s);
}

}  // namespace

cudaError_t launch_rope_append(const AppendArgs &a, bool vectorized, cudaStream_t s) {
  AppendKParams kp{};
  const bool qin = a.q_out == nullptr || a.q_out == a.q;
  kp.q = a.q;
  kp.qo = qin ? a.q : a.q_out;
  kp.kn = a.k_new; kp.vn = a.v_new;
  kp.kc = a.cache.k; kp.vc = a.cache.v;
  kp.sq_t = a.sq[0]; kp.sq_h = a.sq[1];
  kp.sqo_t = qin ? a.sq[0] : a.sqo[0]; kp.sqo_h = qin ? a.sq[1] : a.sqo[1];
  kp.skn_t = a.skn[0]; kp.skn_h = a.skn[1];
  kp.svn_t = a.svn[0]; kp.svn_h = a.svn[1];
  kp.skc_r = a.cache.k_strides[0]; kp.skc_h = a.cache.k_strides[1];
  kp.svc_r = a.cache.v_strides[0]; kp.svc_h = a.cache.v_strides[1];
  kp.T = a.T; kp.Hq = a.Hq; kp.Hkv = a.Hkv; kp.Htot = a.Hq + 2 * a.Hkv;
  kp.half = a.rot_dim / 2; kp.rot_dim = a.rot_dim; kp.q_inplace = qin ? 1 : 0;
  kp.seq_ids = a.seq_ids; kp.seq_start = a.cache.seq_start;
  kp.n_seqs = a.cache.n_seqs; kp.cache_rows = a.cache.rows;
  kp.positions = a.positions; kp.is64 = a.pos_is_int64;
  kp.cos_t = a.cos_t; kp.sin_t = a.sin_t; kp.table_rows = a.table_rows;
  kp.status = a.status;
  if (a.T == 0 || kp.Htot == 0) return cudaSuccess;
  switch (a.dt) {
    case RA_F32: return launch_typed<float>(kp, a, vectorized, s);
    case RA_BF16: return launch_typed<__nv_bfloat16>(kp, a, vectorized, s);
    case RA_F16: return launch_typed<__half>(kp, a, vectorized, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace ra

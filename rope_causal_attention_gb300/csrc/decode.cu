// Decode attention over a KV cache of rotated keys, split along the keys.
//
// What is computed ("RoPE and FlashAttention: relative positions and online
// softmax", sections 2, 4, 5): the new queries of a sequence with L cached
// keys sit at positions L - Sq .. L - 1 and see keys j <= their position
// (the offset mask of section 5); Q and the cached K are already rotated
// (section 2), so the scores are plain dot products times the softmax scale.
//
// Split-KV: a sequence's keys are cut into chunks of `chunk` keys.  Each
// (chunk, kv head, sequence) block runs the online softmax of section 5 over
// its chunk for every query row of the kv head's group and writes the
// normalised partial output O_c and its log-sum-exp LSE_c.  The merge kernel
// then combines the chunks exactly:
//   LSE = M + ln sum_c exp(LSE_c - M),  O = sum_c exp(LSE_c - LSE) O_c,
// M = max_c LSE_c (the same rescaling identity the online softmax applies
// tile by tile).  With one chunk the split kernel writes O and LSE directly.
//
// This file holds the plan, the CUDA-core split kernel (any dtype, even
// D <= 256: fp32 decode, head sizes other than 128, large query groups) and
// the merge; decode_tc.cu holds the tensor-core split kernel.
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace ra {

// Tensor-memory columns a tensor-core decode block allocates (two blocks per SM).
constexpr int kDecodeTmemCols = 256;
// Keys per block on the CUDA-core path (bounds a block's work).
constexpr int64_t kSimtChunkMax = 4096;

bool plan_decode(ra_dtype dt, int B, int Hq, int Hkv, int Sq, int D, int64_t max_kv_len,
                 DecodePlan *plan) {
  if (B < 0 || B > 65535 || Hq < 1 || Hkv < 1 || Hkv > 65535 || Hq % Hkv || Sq < 1 || D < 2 ||
      (D & 1) || D > 256 || max_kv_len < 1)
    return false;
  const int n = (Hq / Hkv) * Sq;  // query rows sharing one kv head
  plan->tc = dt != RA_F32 && D == 128 && n <= 64;
  int64_t chunk_max = kSimtChunkMax;
  if (plan->tc) {
    const int npad = n <= 16 ? 16 : (n <= 32 ? 32 : 64);  // the kernel's column widths
    chunk_max = (int64_t)((kDecodeTmemCols - npad) / npad) * 128;
  }
  const int64_t pairs = (int64_t)(B > 0 ? B : 1) * Hkv;
  const int64_t target = 2 * (int64_t)sm_count_current();
  const int64_t by_len = (max_kv_len + chunk_max - 1) / chunk_max;
  const int64_t max_splits = (max_kv_len + 127) / 128;
  int64_t want = (target + pairs - 1) / pairs;
  if (want > max_splits) want = max_splits;
  int64_t splits = by_len > want ? by_len : want;
  int64_t chunk = (max_kv_len + splits - 1) / splits;
  chunk = (chunk + 127) / 128 * 128;
  splits = (max_kv_len + chunk - 1) / chunk;
  if (splits > 65535) return false;
  plan->splits = (int)splits;
  plan->chunk = chunk;
  plan->ws_bytes = 0;
  plan->ws_lse_offset = 0;
  if (splits > 1) {
    const size_t rows = (size_t)B * Hq * Sq * (size_t)splits;
    const size_t o_bytes = rows * D * sizeof(float);
    plan->ws_lse_offset = (o_bytes + 255) / 256 * 256;
    plan->ws_bytes = plan->ws_lse_offset + rows * sizeof(float);
  }
  return true;
}

namespace {

struct DecodeKParams {
  const void *q;
  void *o;
  float *lse;
  const void *kc, *vc;
  int64_t skc_r, skc_h, svc_r, svc_h;
  const int64_t *seq_start;
  int64_t n_seqs, cache_rows;
  const int32_t *seq_ids, *kv_len;
  int64_t max_kv_len;
  int B, Hq, Hkv, G, Sq, D;
  float scale;
  int64_t sq0, sq1, sq2, so0, so1, so2;
  int splits;
  int64_t chunk;
  float *ws_o, *ws_lse;
  int *status;
};

// Sequence entry b: its key count and first cache row, or false when the
// entry is out of range.
__device__ __forceinline__ bool entry_rows(const DecodeKParams &p, int b, int64_t *L,
                                           int64_t *row0) {
  const int64_t sq = p.seq_ids ? (int64_t)p.seq_ids[b] : (int64_t)b;
  *L = p.kv_len[b];
  if (sq < 0 || sq >= p.n_seqs || *L < p.Sq || *L > p.max_kv_len) return false;
  *row0 = p.seq_start[sq];
  return *row0 >= 0 && *row0 + *L <= p.cache_rows;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

constexpr int kWarps = 8;
constexpr int kTile = 32;  // keys per staged tile (one per lane)
constexpr int kMaxPerLane = 8;

// One block per (chunk, kv head, sequence); warp w handles query rows
// w, w + 8, ... of the kv head's group (row r = group head r / Sq, query r % Sq).
// Lane jj scores key jj of each 32-key tile (K staged as fp32 with a padded
// row so the lanes read distinct banks); lanes split D for the P V update.
template <typename T>
__global__ void __launch_bounds__(kWarps * 32) attn_decode_simt_kernel(DecodeKParams p) {
  extern __shared__ float sm[];
  const int D = p.D, DP = D + 1;
  float *sK = sm;                   // [kTile][D + 1]
  float *sV = sK + kTile * DP;      // [kTile][D]
  float *sQ = sV + kTile * D;       // [kWarps][D]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  int64_t L, row0;
  if (!entry_rows(p, b, &L, &row0)) {
    if (split == 0 && hk == 0 && threadIdx.x == 0) record_status(p.status, RA_ERR_POSITION_RANGE);
    return;
  }
  const int64_t j0 = (int64_t)split * p.chunk;
  if (j0 >= L) return;
  const int64_t j1 = min(L, j0 + p.chunk);
  const T *kb = static_cast<const T *>(p.kc) + hk * p.skc_h;
  const T *vb = static_cast<const T *>(p.vc) + hk * p.svc_h;
  const int R = p.G * p.Sq;

  for (int rbase = 0; rbase < R; rbase += kWarps) {
    const int r = rbase + warp;
    const bool row_ok = r < R;
    const int hg = row_ok ? r / p.Sq : 0, i = row_ok ? r % p.Sq : 0;
    const int h = hk * p.G + hg;
    const int64_t qpos = L - p.Sq + i;
    float *qw = sQ + warp * D;
    __syncwarp();  // every lane is done with the previous row's qw
    if (row_ok) {
      const T *src = static_cast<const T *>(p.q) + b * p.sq0 + h * p.sq1 + i * p.sq2;
      for (int d = lane; d < D; d += 32) qw[d] = Elem<T>::load(src[d]);
    }
    float m = -INFINITY, l = 0.f, acc[kMaxPerLane];
#pragma unroll
    for (int u = 0; u < kMaxPerLane; ++u) acc[u] = 0.f;

    for (int64_t jt = j0; jt < j1; jt += kTile) {
      const int nk = (int)min((int64_t)kTile, j1 - jt);
      __syncthreads();  // previous tile consumed (and sQ written)
      for (int e = threadIdx.x; e < kTile * D; e += blockDim.x) {
        const int jj = e / D, d = e - jj * D;
        float kx = 0.f, vx = 0.f;
        if (jj < nk) {
          const int64_t row = row0 + jt + jj;
          kx = Elem<T>::load(kb[row * p.skc_r + d]);
          vx = Elem<T>::load(vb[row * p.svc_r + d]);
        }
        sK[jj * DP + d] = kx;
        sV[jj * D + d] = vx;
      }
      __syncthreads();
      if (!row_ok) continue;
      float sc = 0.f;
      for (int d = 0; d < D; ++d) sc += qw[d] * sK[lane * DP + d];
      const int64_t j = jt + lane;
      sc = (lane < nk && j <= qpos) ? sc * p.scale : -INFINITY;
      const float tmax = warp_max(sc);
      if (tmax == -INFINITY) continue;  // every key of the tile is masked for this row
      const float m_new = fmaxf(m, tmax);
      const float corr = expf(m - m_new);
      const float pj = expf(sc - m_new);
      l = l * corr + warp_sum(pj);
#pragma unroll
      for (int u = 0; u < kMaxPerLane; ++u) acc[u] *= corr;
      for (int jj = 0; jj < nk; ++jj) {
        const float w = __shfl_sync(0xffffffffu, pj, jj);
#pragma unroll
        for (int u = 0; u < kMaxPerLane; ++u) {
          const int d = lane + 32 * u;
          if (d < D) acc[u] += w * sV[jj * D + d];
        }
      }
      m = m_new;
    }
    if (row_ok) {
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse = l > 0.f ? m + logf(l) : -INFINITY;
      if (p.splits == 1) {
        T *dst = static_cast<T *>(p.o) + b * p.so0 + h * p.so1 + i * p.so2;
#pragma unroll
        for (int u = 0; u < kMaxPerLane; ++u) {
          const int d = lane + 32 * u;
          if (d < D) dst[d] = Elem<T>::store(acc[u] * inv);
        }
        if (p.lse && lane == 0) p.lse[((int64_t)b * p.Hq + h) * p.Sq + i] = lse;
      } else {
        const int64_t wrow = (((int64_t)b * p.Hq + h) * p.Sq + i) * p.splits + split;
        float *dst = p.ws_o + wrow * D;
#pragma unroll
        for (int u = 0; u < kMaxPerLane; ++u) {
          const int d = lane + 32 * u;
          if (d < D) dst[d] = acc[u] * inv;
        }
        if (lane == 0) p.ws_lse[wrow] = lse;
      }
    }
  }
}

// One warp per output row (b, h, i): merges the chunks that hold keys of the
// sequence (chunk c holds keys [c * chunk, (c + 1) * chunk)).
template <typename T>
__global__ void __launch_bounds__(256) attn_decode_merge_kernel(DecodeKParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t rows = (int64_t)p.B * p.Hq * p.Sq;
  if (row >= rows) return;
  const int i = (int)(row % p.Sq);
  const int h = (int)((row / p.Sq) % p.Hq);
  const int b = (int)(row / ((int64_t)p.Sq * p.Hq));
  int64_t L, row0;
  if (!entry_rows(p, b, &L, &row0)) return;  // the split kernel recorded it
  const int n = (int)((L + p.chunk - 1) / p.chunk);
  const float *lse = p.ws_lse + row * p.splits;
  float M = -INFINITY;
  for (int c = lane; c < n; c += 32) M = fmaxf(M, lse[c]);
  M = warp_max(M);
  float wsum = 0.f;
  for (int c = lane; c < n; c += 32) wsum += expf(lse[c] - M);
  wsum = warp_sum(wsum);
  const float total = M + logf(wsum);
  T *dst = static_cast<T *>(p.o) + b * p.so0 + h * p.so1 + i * p.so2;
  const float *src = p.ws_o + row * p.splits * p.D;
  for (int d = lane; d < p.D; d += 32) {
    float acc = 0.f;
    for (int c = 0; c < n; ++c) acc += expf(lse[c] - total) * src[(int64_t)c * p.D + d];
    dst[d] = Elem<T>::store(acc);
  }
  if (p.lse && lane == 0) p.lse[row] = total;
}

DecodeKParams kparams(const DecodeArgs &a) {
  DecodeKParams p{};
  p.q = a.q; p.o = a.o; p.lse = a.lse;
  p.kc = a.cache.k; p.vc = a.cache.v;
  p.skc_r = a.cache.k_strides[0]; p.skc_h = a.cache.k_strides[1];
  p.svc_r = a.cache.v_strides[0]; p.svc_h = a.cache.v_strides[1];
  p.seq_start = a.cache.seq_start; p.n_seqs = a.cache.n_seqs; p.cache_rows = a.cache.rows;
  p.seq_ids = a.seq_ids; p.kv_len = a.kv_len; p.max_kv_len = a.max_kv_len;
  p.B = a.B; p.Hq = a.Hq; p.Hkv = a.Hkv; p.G = a.Hq / a.Hkv; p.Sq = a.Sq; p.D = a.D;
  p.scale = a.scale;
  p.sq0 = a.sq[0]; p.sq1 = a.sq[1]; p.sq2 = a.sq[2];
  p.so0 = a.so[0]; p.so1 = a.so[1]; p.so2 = a.so[2];
  p.splits = a.plan.splits; p.chunk = a.plan.chunk;
  if (a.plan.splits > 1) {
    p.ws_o = static_cast<float *>(a.workspace);
    p.ws_lse = reinterpret_cast<float *>(static_cast<char *>(a.workspace) + a.plan.ws_lse_offset);
  }
  p.status = a.status;
  return p;
}

template <typename T>
cudaError_t launch_simt(const DecodeKParams &p, cudaStream_t s) {
  const size_t smem = ((size_t)kTile * (p.D + 1) + (size_t)kTile * p.D + (size_t)kWarps * p.D) *
                      sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(attn_decode_simt_kernel<T>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)p.splits, (unsigned)p.Hkv, (unsigned)p.B);
  attn_decode_simt_kernel<T><<<grid, kWarps * 32, smem, s>>>(p);
  note_launch("attn_decode_simt_kernel");
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_merge(const DecodeKParams &p, cudaStream_t s) {
  const int64_t rows = (int64_t)p.B * p.Hq * p.Sq;
  const int64_t blocks = (rows + 7) / 8;
  if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
  attn_decode_merge_kernel<T><<<(unsigned)blocks, 256, 0, s>>>(p);
  note_launch("attn_decode_merge_kernel");
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_typed(const DecodeArgs &a, cudaStream_t s) {
  const DecodeKParams p = kparams(a);
  // the tensor-core kernel declines cases it has no variant for (e.g. a cache
  // too tall for a tensor map); the CUDA-core kernel then runs the same plan
  cudaError_t e = a.plan.tc ? launch_attn_decode_tc(a, s) : cudaErrorNotSupported;
  if (e == cudaErrorNotSupported) e = launch_simt<T>(p, s);
  if (e != cudaSuccess) return e;
  return a.plan.splits > 1 ? launch_merge<T>(p, s) : cudaSuccess;
}

}  // namespace

cudaError_t launch_attn_decode(const DecodeArgs &a, cudaStream_t s) {
  if (a.B == 0) return cudaSuccess;
  switch (a.dt) {
    case RA_F32: return launch_typed<float>(a, s);
    case RA_BF16: return launch_typed<__nv_bfloat16>(a, s);
    case RA_F16: return launch_typed<__half>(a, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace ra

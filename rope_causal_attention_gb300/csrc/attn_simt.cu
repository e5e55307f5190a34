// fp32 causal attention with RoPE fused in, on CUDA cores.
//
// Serves fp32 inputs, where rounding rotated Q/K to a 16-bit tensor-core
// operand would break a 1e-4 output tolerance.  Same mathematics as the
// tensor-core kernel ("RoPE and FlashAttention: relative positions and online
// softmax", sections 1, 2, 4, 5): Q rotated once at kv_offset + i, each K tile
// rotated as it is staged in shared memory, online softmax with running max m,
// denominator l and numerator u, output u / l, LSE = m + ln l.
//
// Layout: one warp per query row (lanes split the head dimension for the
// output, D <= 256; the kernel is instantiated for 1, 2, 4 or 8 output
// columns per lane), eight rows per block, key tiles of 32 rows staged and
// rotated in shared memory (rows padded by one float, so 32 lanes reading 32
// different rows at one column hit 32 banks) and shared by the eight warps.
// Lane j of a warp computes the whole score of key j of the tile against the
// warp's rotated query row (shared memory, read as a broadcast), so the
// tile's softmax statistics are warp reductions.  Rotation is by pairs: one
// cos/sin read per pair.
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace ra {
namespace {

constexpr int kRows = 8;    // query rows (warps) per block
constexpr int kTileK = 32;  // keys per staged tile (one per lane)
constexpr int kMaxPerLane = 8;  // D <= 256
constexpr int kStageU = 8;      // loads in flight per thread while staging a tile

struct SimtParams {
  const float *q, *k, *v;
  float *o, *lse;
  int Hq, G, D;
  int64_t Sq, Sk, kv_offset;
  int apply_rope, rot_dim, layout;
  const float *cos_t, *sin_t;
  float scale;
  int64_t sq[3], sk[3], sv[3], so[3];
};

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// Rotates pair i (< rot_dim / 2) of row x (fp32, any memory) in place at
// position pos: NeoX pairs (i, i + rot_dim/2), GPT-J pairs (2i, 2i+1).
__device__ __forceinline__ void rotate_pair(float *x, int i, int64_t pos, const SimtParams &p) {
  const int half = p.rot_dim >> 1;
  const int lo = p.layout == RA_NEOX ? i : 2 * i;
  const int hi = p.layout == RA_NEOX ? i + half : 2 * i + 1;
  const float c = __ldg(p.cos_t + pos * half + i);
  const float s = __ldg(p.sin_t + pos * half + i);
  const float a = x[lo], b = x[hi];
  x[lo] = a * c - b * s;
  x[hi] = b * c + a * s;
}

// The same with cos and sin already loaded.
__device__ __forceinline__ void rotate_pair_cs(float *x, int i, float c, float s,
                                               const SimtParams &p) {
  const int half = p.rot_dim >> 1;
  const int lo = p.layout == RA_NEOX ? i : 2 * i;
  const int hi = p.layout == RA_NEOX ? i + half : 2 * i + 1;
  const float a = x[lo], b = x[hi];
  x[lo] = a * c - b * s;
  x[hi] = b * c + a * s;
}

// NU = output columns per lane (D <= 32 NU)
template <int NU>
__global__ void __launch_bounds__(kRows * 32) attn_simt_kernel(SimtParams p) {
  extern __shared__ float smem[];
  const int D = p.D, DP = D + 1;
  float *sK = smem;                  // [kTileK][D + 1] rotated keys
  float *sV = sK + kTileK * DP;      // [kTileK][D]
  float *sQ = sV + kTileK * D;       // [kRows][D] rotated query rows
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y, b = blockIdx.z, hk = h / p.G;
  const int64_t i = (int64_t)blockIdx.x * kRows + warp;  // this warp's query row
  const bool row_ok = i < p.Sq;
  const int64_t qpos = p.kv_offset + i;
  const int half = p.apply_rope ? p.rot_dim >> 1 : 0;  // rotated pairs per row

  float m = -INFINITY, l = 0.f, acc[NU];
#pragma unroll
  for (int u = 0; u < NU; ++u) acc[u] = 0.f;

  const int64_t last_row = min((int64_t)blockIdx.x * kRows + kRows - 1, p.Sq - 1);
  const int64_t kend = min(p.Sk, p.kv_offset + last_row + 1);
  const float *kb = p.k + b * p.sk[0] + hk * p.sk[1];
  const float *vb = p.v + b * p.sv[0] + hk * p.sv[1];

  // A tile is staged in chunks of kStageU elements (and cos/sin pairs) per
  // thread, each chunk's loads issued together.  The first chunk of the
  // next tile is loaded into registers before this tile's scores and P V,
  // so its latency overlaps them (for D <= 64 that is the whole tile).
  constexpr int CHK = kStageU * kRows * 32;
  float kx[kStageU], vx[kStageU], cv[kStageU], sv[kStageU];
  // element e of a tile is (row e / D, column e % D), pair e is (row
  // e / half, pair e % half): shifts when D and half are powers of two
  const int dsh = (D & (D - 1)) == 0 ? __ffs(D) - 1 : -1;
  const int hsh = half > 0 && (half & (half - 1)) == 0 ? __ffs(half) - 1 : -1;
  auto div_d = [&](int e) { return dsh >= 0 ? e >> dsh : e / D; };
  auto div_h = [&](int e) { return hsh >= 0 ? e >> hsh : (half ? e / half : 0); };
  auto load_chunk = [&](int64_t jt, int nkt, int c0) {
#pragma unroll
    for (int u = 0; u < kStageU; ++u) {
      const int e = c0 + threadIdx.x + u * kRows * 32;
      const int jj = div_d(e), d = e - jj * D;
      const bool in = e < kTileK * D && jj < nkt;
      kx[u] = in ? kb[(jt + jj) * p.sk[2] + d] : 0.f;
      vx[u] = in ? vb[(jt + jj) * p.sv[2] + d] : 0.f;
    }
  };
  auto load_pairs = [&](int64_t jt, int nkt, int c0) {
#pragma unroll
    for (int u = 0; u < kStageU; ++u) {
      const int e = c0 + threadIdx.x + u * kRows * 32;
      const int jj = div_h(e), pi = e - jj * half;
      const bool in = e < kTileK * half && jj < nkt;
      cv[u] = in ? __ldg(p.cos_t + (jt + jj) * half + pi) : 1.f;
      sv[u] = in ? __ldg(p.sin_t + (jt + jj) * half + pi) : 0.f;
    }
  };
  if (kend > 0) {
    const int nk0 = (int)min((int64_t)kTileK, kend);
    load_chunk(0, nk0, 0);
    load_pairs(0, nk0, 0);
  }

  // ---- this warp's query row, rotated once (while the first tile's loads
  // are in flight)
  float *qs = sQ + warp * D;
  {
    const float *src = p.q + b * p.sq[0] + h * p.sq[1] + (row_ok ? i : 0) * p.sq[2];
    for (int d = lane; d < D; d += 32) qs[d] = row_ok ? src[d] : 0.f;
    __syncwarp();
    if (row_ok)
      for (int e = lane; e < half; e += 32) rotate_pair(qs, e, qpos, p);
    __syncwarp();
  }
  for (int64_t j0 = 0; j0 < kend; j0 += kTileK) {
    const int nk = (int)min((int64_t)kTileK, kend - j0);
    // stage raw K (padded rows) and V
    for (int c0 = 0; c0 < kTileK * D; c0 += CHK) {
      if (c0 > 0) load_chunk(j0, nk, c0);
#pragma unroll
      for (int u = 0; u < kStageU; ++u) {
        const int e = c0 + threadIdx.x + u * kRows * 32;
        if (e < kTileK * D) {
          const int jj = div_d(e), d = e - jj * D;
          sK[jj * DP + d] = kx[u];
          sV[e] = vx[u];
        }
      }
    }
    __syncthreads();
    // rotate K at positions j, pair by pair
    for (int c0 = 0; c0 < kTileK * half; c0 += CHK) {
      if (c0 > 0) load_pairs(j0, nk, c0);
#pragma unroll
      for (int u = 0; u < kStageU; ++u) {
        const int e = c0 + threadIdx.x + u * kRows * 32;
        const int jj = div_h(e), pi = e - jj * half;
        if (e < kTileK * half && jj < nk) rotate_pair_cs(sK + jj * DP, pi, cv[u], sv[u], p);
      }
    }
    __syncthreads();
    if (j0 + kTileK < kend) {  // the next tile's first chunk, in flight meanwhile
      const int nkn = (int)min((int64_t)kTileK, kend - j0 - kTileK);
      load_chunk(j0 + kTileK, nkn, 0);
      load_pairs(j0 + kTileK, nkn, 0);
    }

    if (row_ok) {
      // lane jj scores key j0 + jj (four partial sums to shorten the chain)
      const float *kr = sK + lane * DP;
      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
      int d = 0;
      for (; d + 4 <= D; d += 4) {
        s0 = fmaf(qs[d], kr[d], s0);
        s1 = fmaf(qs[d + 1], kr[d + 1], s1);
        s2 = fmaf(qs[d + 2], kr[d + 2], s2);
        s3 = fmaf(qs[d + 3], kr[d + 3], s3);
      }
      for (; d < D; ++d) s0 = fmaf(qs[d], kr[d], s0);
      const int64_t j = j0 + lane;
      const float my_s = (lane < nk && j <= qpos) ? ((s0 + s1) + (s2 + s3)) * p.scale : -INFINITY;
      const float tmax = warp_max(my_s);
      if (tmax != -INFINITY) {
        const float m_new = fmaxf(m, tmax);
        const float corr = expf(m - m_new);
        const float pj = expf(my_s - m_new);
        l = l * corr + warp_sum(pj);
#pragma unroll
        for (int u = 0; u < NU; ++u) acc[u] *= corr;
        for (int jj = 0; jj < nk; ++jj) {
          const float w = __shfl_sync(0xffffffffu, pj, jj);
#pragma unroll
          for (int u = 0; u < NU; ++u) {
            const int d = lane + 32 * u;
            if (d < D) acc[u] += w * sV[jj * D + d];
          }
        }
        m = m_new;
      }
    }
    __syncthreads();
  }

  if (row_ok) {
    const float inv = 1.f / l;
    float *dst = p.o + b * p.so[0] + h * p.so[1] + i * p.so[2];
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      const int d = lane + 32 * u;
      if (d < D) dst[d] = acc[u] * inv;
    }
    if (p.lse && lane == 0) p.lse[((int64_t)b * p.Hq + h) * p.Sq + i] = m + logf(l);
  }
}

template <int NU>
cudaError_t launch_nu(const SimtParams &p, dim3 grid, size_t smem, cudaStream_t s) {
  const cudaError_t e = cudaFuncSetAttribute(attn_simt_kernel<NU>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  attn_simt_kernel<NU><<<grid, kRows * 32, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_simt(const AttnArgs &a, cudaStream_t s) {
  SimtParams p{};
  p.q = static_cast<const float *>(a.q);
  p.k = static_cast<const float *>(a.k);
  p.v = static_cast<const float *>(a.v);
  p.o = static_cast<float *>(a.o);
  p.lse = a.lse;
  p.Hq = a.Hq; p.G = a.Hq / a.Hkv; p.D = a.D;
  p.Sq = a.Sq; p.Sk = a.Sk; p.kv_offset = a.kv_offset;
  p.apply_rope = a.apply_rope; p.rot_dim = a.rot_dim; p.layout = a.layout;
  p.cos_t = a.cos_t; p.sin_t = a.sin_t; p.scale = a.scale;
  for (int j = 0; j < 3; ++j) {
    p.sq[j] = a.sq[j]; p.sk[j] = a.sk[j]; p.sv[j] = a.sv[j]; p.so[j] = a.so[j];
  }
  const size_t smem = ((size_t)kTileK * (a.D + 1) + (size_t)kTileK * a.D + (size_t)kRows * a.D) * sizeof(float);
  const dim3 grid((unsigned)((a.Sq + kRows - 1) / kRows), (unsigned)a.Hq, (unsigned)a.B);
  if (a.D <= 32) return launch_nu<1>(p, grid, smem, s);
  if (a.D <= 64) return launch_nu<2>(p, grid, smem, s);
  if (a.D <= 128) return launch_nu<4>(p, grid, smem, s);
  return launch_nu<kMaxPerLane>(p, grid, smem, s);
}

}  // namespace ra

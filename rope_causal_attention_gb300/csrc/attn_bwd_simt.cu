// Backward of causal attention with RoPE fused in: the row-term kernel shared
// by both backward paths, and the CUDA-core (fp32) gradient kernels.
//
// Mathematics ("RoPE and FlashAttention: relative positions and online
// softmax", section 5: probabilities are rebuilt from Q, K and the forward's
// row normaliser LSE; sections 1-2: the rotation):
//   P_ij = exp(s_ij - LSE_i) for admissible j (s as in the forward),
//   D_i = <dO_i, O_i>  (= sum_j P_ij dP_ij),
//   dS_ij = P_ij (dP_ij - D_i),  dP_ij = <dO_i, v_j>,
//   dV_j = sum_i P_ij dO_i,  dq~_i = scale sum_j dS_ij k~_j,
//   dk~_j = scale sum_i dS_ij q~_i,  dq = R^T dq~,  dk = R^T dk~.
//
// CUDA-core layout (fp32 inputs, D <= 256): the dq kernel gives each warp one
// query row and stages 32 rotated keys (and their values) per step in
// shared memory, lane jj scoring key jj; the dk/dv kernel gives each warp one
// key row and stages 32 rotated queries (with dO, LSE and D) per step, over
// every q-head of the kv head's group.  Rows are padded by one float so that
// lanes reading different rows hit different banks.
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace ra {
namespace {

constexpr int kRows = 8;   // warps (rows) per block
constexpr int kTile = 32;  // staged rows per step (one per lane)
constexpr int kMaxPerLane = 8;

struct BwdSimtParams {
  const void *q, *k, *v, *dout;
  const float *lse, *dsum;
  void *dq, *dk, *dv;
  int Hq, Hkv, G, D;
  int64_t Sq, Sk, off;
  int apply_rope, rot_dim, layout;
  const float *cos_t, *sin_t;
  float scale;
  int64_t sq[3], sk[3], sv[3], sdo[3], sdq[3], sdk[3], sdv[3];
};

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Dim d of row x (fp32, length D) rotated at position pos: dir = +1 applies
// R(pos), dir = -1 applies R(pos)^T (the rotation by the negated angle).
__device__ __forceinline__ float rot_at(const float *x, int d, int64_t pos, float dir,
                                        const BwdSimtParams &p) {
  if (!p.apply_rope || d >= p.rot_dim) return x[d];
  const int half = p.rot_dim >> 1;
  bool low;
  int i, partner;
  if (p.layout == RA_NEOX) {
    low = d < half;
    i = low ? d : d - half;
    partner = low ? d + half : d - half;
  } else {
    low = (d & 1) == 0;
    i = d >> 1;
    partner = d ^ 1;
  }
  const float c = __ldg(p.cos_t + pos * half + i);
  const float s = dir * __ldg(p.sin_t + pos * half + i);
  return low ? x[d] * c - x[partner] * s : x[d] * c + x[partner] * s;
}

// D_i = <dO_i, O_i> with 16-byte loads: CH = D / (16 / sizeof(T)) lanes per
// row (a power of two <= 32), 32 / CH rows per warp; O and dO are read once,
// so they take the streaming cache hint.
template <typename T>
__global__ void __launch_bounds__(256) bwd_rowterm_vec_kernel(const T *o, const T *dout,
                                                              float *dsum, int Hq, int64_t Sq,
                                                              int CH, int64_t so0, int64_t so1,
                                                              int64_t so2, int64_t sd0,
                                                              int64_t sd1, int64_t sd2,
                                                              int64_t rows) {
  constexpr int V = VecN<T>::N;
  const int lane = threadIdx.x & 31;
  const int c = lane & (CH - 1);
  const int64_t r = ((int64_t)blockIdx.x * 8 + (threadIdx.x >> 5)) * (32 / CH) + lane / CH;
  float acc = 0.f;
  if (r < rows) {
    const int64_t i = r % Sq, bh = r / Sq;
    const int64_t h = bh % Hq, b = bh / Hq;
    const uint4 uo = __ldcs(reinterpret_cast<const uint4 *>(o + b * so0 + h * so1 + i * so2) + c);
    const uint4 ud = __ldcs(reinterpret_cast<const uint4 *>(dout + b * sd0 + h * sd1 + i * sd2) + c);
    float fo[V], fd[V];
    unpack16<T>(uo, fo);
    unpack16<T>(ud, fd);
#pragma unroll
    for (int e = 0; e < V; ++e) acc = fmaf(fo[e], fd[e], acc);
  }
  for (int off = CH >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (c == 0 && r < rows) dsum[r] = acc;
}

template <typename T>
__global__ void __launch_bounds__(256) bwd_rowterm_kernel(const T *o, const T *dout, float *dsum,
                                                          int Hq, int64_t Sq, int D, int64_t so0,
                                                          int64_t so1, int64_t so2, int64_t sd0,
                                                          int64_t sd1, int64_t sd2, int64_t rows) {
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= rows) return;
  const int64_t i = r % Sq, bh = r / Sq;
  const int64_t h = bh % Hq, b = bh / Hq;
  const T *po = o + b * so0 + h * so1 + i * so2;
  const T *pd = dout + b * sd0 + h * sd1 + i * sd2;
  float acc = 0.f;
  for (int d = lane; d < D; d += 32) acc += Elem<T>::load(po[d]) * Elem<T>::load(pd[d]);
  acc = warp_sum(acc);
  if (lane == 0) dsum[r] = acc;
}

template <typename T>
__global__ void __launch_bounds__(kRows * 32) bwd_dq_simt_kernel(BwdSimtParams p) {
  extern __shared__ float sm[];
  const int D = p.D, DP = D + 1;
  float *sK = sm;                   // [kTile][D+1] rotated keys
  float *sV = sK + kTile * DP;      // [kTile][D+1] values
  float *sRaw = sV + kTile * DP;    // [kTile][D] raw keys
  float *sRow = sRaw + kTile * D;   // [kRows][3][D]: q~, dO, dq~ of each warp
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y, b = blockIdx.z, hk = h / p.G;
  const int64_t i = (int64_t)blockIdx.x * kRows + warp;
  const bool row_ok = i < p.Sq;
  const int64_t qpos = p.off + i;
  float *qr = sRow + warp * 3 * D, *dor = qr + D, *dqr = dor + D;
  float lse = 0.f, dsum = 0.f;
  if (row_ok) {
    const T *qs = static_cast<const T *>(p.q) + b * p.sq[0] + h * p.sq[1] + i * p.sq[2];
    const T *ds = static_cast<const T *>(p.dout) + b * p.sdo[0] + h * p.sdo[1] + i * p.sdo[2];
    for (int d = lane; d < D; d += 32) {
      dqr[d] = Elem<T>::load(qs[d]);  // raw q, rotated below
      dor[d] = Elem<T>::load(ds[d]);
    }
    const int64_t r = ((int64_t)b * p.Hq + h) * p.Sq + i;
    lse = p.lse[r];
    dsum = p.dsum[r];
  }
  __syncwarp();
  if (row_ok)
    for (int d = lane; d < D; d += 32) qr[d] = rot_at(dqr, d, qpos, 1.f, p);
  __syncwarp();

  float acc[kMaxPerLane];
#pragma unroll
  for (int u = 0; u < kMaxPerLane; ++u) acc[u] = 0.f;
  const int64_t last = min((int64_t)blockIdx.x * kRows + kRows - 1, p.Sq - 1);
  const int64_t kend = min(p.Sk, p.off + last + 1);
  const T *kb = static_cast<const T *>(p.k) + b * p.sk[0] + hk * p.sk[1];
  const T *vb = static_cast<const T *>(p.v) + b * p.sv[0] + hk * p.sv[1];
  for (int64_t j0 = 0; j0 < kend; j0 += kTile) {
    const int nk = (int)min((int64_t)kTile, kend - j0);
    __syncthreads();
    for (int e = threadIdx.x; e < kTile * D; e += blockDim.x) {
      const int jj = e / D, d = e - jj * D;
      const bool ok = jj < nk;
      sRaw[e] = ok ? Elem<T>::load(kb[(j0 + jj) * p.sk[2] + d]) : 0.f;
      sV[jj * DP + d] = ok ? Elem<T>::load(vb[(j0 + jj) * p.sv[2] + d]) : 0.f;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < kTile * D; e += blockDim.x) {
      const int jj = e / D, d = e - jj * D;
      sK[jj * DP + d] = jj < nk ? rot_at(sRaw + jj * D, d, j0 + jj, 1.f, p) : 0.f;
    }
    __syncthreads();
    if (!row_ok) continue;
    float s = 0.f, dp = 0.f;
    for (int d = 0; d < D; ++d) {
      s += qr[d] * sK[lane * DP + d];
      dp += dor[d] * sV[lane * DP + d];
    }
    const bool vis = lane < nk && j0 + lane <= qpos;
    const float pr = vis ? expf(s * p.scale - lse) : 0.f;
    const float dsv = pr * (dp - dsum);
    for (int jj = 0; jj < nk; ++jj) {
      const float w = __shfl_sync(0xffffffffu, dsv, jj);
#pragma unroll
      for (int u = 0; u < kMaxPerLane; ++u) {
        const int d = lane + 32 * u;
        if (d < D) acc[u] += w * sK[jj * DP + d];
      }
    }
  }
  if (!row_ok) return;
#pragma unroll
  for (int u = 0; u < kMaxPerLane; ++u) {
    const int d = lane + 32 * u;
    if (d < D) dqr[d] = acc[u] * p.scale;
  }
  __syncwarp();
  T *dst = static_cast<T *>(p.dq) + b * p.sdq[0] + h * p.sdq[1] + i * p.sdq[2];
  for (int d = lane; d < D; d += 32) dst[d] = Elem<T>::store(rot_at(dqr, d, qpos, -1.f, p));
}

template <typename T>
__global__ void __launch_bounds__(kRows * 32) bwd_dkdv_simt_kernel(BwdSimtParams p) {
  extern __shared__ float sm[];
  const int D = p.D, DP = D + 1;
  float *sQ = sm;                   // [kTile][D+1] rotated queries
  float *sO = sQ + kTile * DP;      // [kTile][D+1] dO rows
  float *sRaw = sO + kTile * DP;    // [kTile][D] raw queries
  float *sL = sRaw + kTile * D;     // [kTile] LSE, then [kTile] D terms
  float *sRow = sL + 2 * kTile;     // [kRows][3][D]: k~, v, dk~ of each warp
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hk = blockIdx.y, b = blockIdx.z;
  const int64_t j = (int64_t)blockIdx.x * kRows + warp;
  const bool row_ok = j < p.Sk;
  float *kr = sRow + warp * 3 * D, *vr = kr + D, *dkr = vr + D;
  if (row_ok) {
    const T *ks = static_cast<const T *>(p.k) + b * p.sk[0] + hk * p.sk[1] + j * p.sk[2];
    const T *vs = static_cast<const T *>(p.v) + b * p.sv[0] + hk * p.sv[1] + j * p.sv[2];
    for (int d = lane; d < D; d += 32) {
      dkr[d] = Elem<T>::load(ks[d]);
      vr[d] = Elem<T>::load(vs[d]);
    }
  }
  __syncwarp();
  if (row_ok)
    for (int d = lane; d < D; d += 32) kr[d] = rot_at(dkr, d, j, 1.f, p);
  __syncwarp();

  float dv[kMaxPerLane], dk[kMaxPerLane];
#pragma unroll
  for (int u = 0; u < kMaxPerLane; ++u) dv[u] = dk[u] = 0.f;
  // queries that see the block's first key: off + i >= j_first
  const int64_t jfirst = (int64_t)blockIdx.x * kRows;
  int64_t istart = jfirst - p.off;
  istart = istart < 0 ? 0 : (istart / kTile) * kTile;
  for (int g = 0; g < p.G; ++g) {
    const int h = hk * p.G + g;
    const T *qb = static_cast<const T *>(p.q) + b * p.sq[0] + h * p.sq[1];
    const T *db = static_cast<const T *>(p.dout) + b * p.sdo[0] + h * p.sdo[1];
    const int64_t rbase = ((int64_t)b * p.Hq + h) * p.Sq;
    for (int64_t i0 = istart; i0 < p.Sq; i0 += kTile) {
      const int ni = (int)min((int64_t)kTile, p.Sq - i0);
      __syncthreads();
      for (int e = threadIdx.x; e < kTile * D; e += blockDim.x) {
        const int ii = e / D, d = e - ii * D;
        const bool ok = ii < ni;
        sRaw[e] = ok ? Elem<T>::load(qb[(i0 + ii) * p.sq[2] + d]) : 0.f;
        sO[ii * DP + d] = ok ? Elem<T>::load(db[(i0 + ii) * p.sdo[2] + d]) : 0.f;
      }
      if (threadIdx.x < kTile) {
        const bool ok = (int)threadIdx.x < ni;
        sL[threadIdx.x] = ok ? p.lse[rbase + i0 + threadIdx.x] : 0.f;
        sL[kTile + threadIdx.x] = ok ? p.dsum[rbase + i0 + threadIdx.x] : 0.f;
      }
      __syncthreads();
      for (int e = threadIdx.x; e < kTile * D; e += blockDim.x) {
        const int ii = e / D, d = e - ii * D;
        sQ[ii * DP + d] = ii < ni ? rot_at(sRaw + ii * D, d, p.off + i0 + ii, 1.f, p) : 0.f;
      }
      __syncthreads();
      if (!row_ok) continue;
      float s = 0.f, dp = 0.f;
      for (int d = 0; d < D; ++d) {
        s += kr[d] * sQ[lane * DP + d];
        dp += vr[d] * sO[lane * DP + d];
      }
      const bool vis = lane < ni && j <= p.off + i0 + lane;
      const float pr = vis ? expf(s * p.scale - sL[lane]) : 0.f;
      const float dsv = pr * (dp - sL[kTile + lane]);
      for (int ii = 0; ii < ni; ++ii) {
        const float wp = __shfl_sync(0xffffffffu, pr, ii);
        const float ws = __shfl_sync(0xffffffffu, dsv, ii);
#pragma unroll
        for (int u = 0; u < kMaxPerLane; ++u) {
          const int d = lane + 32 * u;
          if (d < D) {
            dv[u] += wp * sO[ii * DP + d];
            dk[u] += ws * sQ[ii * DP + d];
          }
        }
      }
    }
  }
  if (!row_ok) return;
#pragma unroll
  for (int u = 0; u < kMaxPerLane; ++u) {
    const int d = lane + 32 * u;
    if (d < D) dkr[d] = dk[u] * p.scale;
  }
  __syncwarp();
  T *dks = static_cast<T *>(p.dk) + b * p.sdk[0] + hk * p.sdk[1] + j * p.sdk[2];
  T *dvs = static_cast<T *>(p.dv) + b * p.sdv[0] + hk * p.sdv[1] + j * p.sdv[2];
  for (int d = lane; d < D; d += 32) dks[d] = Elem<T>::store(rot_at(dkr, d, j, -1.f, p));
#pragma unroll
  for (int u = 0; u < kMaxPerLane; ++u) {
    const int d = lane + 32 * u;
    if (d < D) dvs[d] = Elem<T>::store(dv[u]);
  }
}

BwdSimtParams simt_params(const BwdArgs &a) {
  BwdSimtParams p{};
  p.q = a.f.q; p.k = a.f.k; p.v = a.f.v; p.dout = a.dout;
  p.lse = a.lse; p.dsum = a.dsum;
  p.dq = a.dq; p.dk = a.dk; p.dv = a.dv;
  p.Hq = a.f.Hq; p.Hkv = a.f.Hkv; p.G = a.f.Hq / a.f.Hkv; p.D = a.f.D;
  p.Sq = a.f.Sq; p.Sk = a.f.Sk; p.off = a.f.kv_offset;
  p.apply_rope = a.f.apply_rope; p.rot_dim = a.f.rot_dim; p.layout = a.f.layout;
  p.cos_t = a.f.cos_t; p.sin_t = a.f.sin_t; p.scale = a.f.scale;
  for (int j = 0; j < 3; ++j) {
    p.sq[j] = a.f.sq[j]; p.sk[j] = a.f.sk[j]; p.sv[j] = a.f.sv[j];
    p.sdo[j] = a.sdo[j]; p.sdq[j] = a.sdq[j]; p.sdk[j] = a.sdk[j]; p.sdv[j] = a.sdv[j];
  }
  return p;
}

template <typename T>
cudaError_t rowterm_typed(const BwdArgs &a, cudaStream_t s) {
  const int64_t rows = (int64_t)a.f.B * a.f.Hq * a.f.Sq;
  constexpr int V = VecN<T>::N;
  const int CH = a.f.D / V;  // lanes per row in the vector kernel
  // the vector kernel serves the 16-bit inputs of the tensor-core backward
  bool vec = sizeof(T) == 2 && a.f.D % V == 0 && CH >= 1 && CH <= 32 && (CH & (CH - 1)) == 0 &&
             reinterpret_cast<uintptr_t>(a.o) % 16 == 0 &&
             reinterpret_cast<uintptr_t>(a.dout) % 16 == 0;
  for (int j = 0; j < 3; ++j) vec = vec && a.sod[j] % V == 0 && a.sdo[j] % V == 0;
  if (vec) {
    const int64_t rows_per_block = 8 * (32 / CH);
    const int64_t blocks = (rows + rows_per_block - 1) / rows_per_block;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    bwd_rowterm_vec_kernel<T><<<(unsigned)blocks, 256, 0, s>>>(
        static_cast<const T *>(a.o), static_cast<const T *>(a.dout), a.dsum, a.f.Hq, a.f.Sq,
        CH, a.sod[0], a.sod[1], a.sod[2], a.sdo[0], a.sdo[1], a.sdo[2], rows);
    note_launch("bwd_rowterm_vec_kernel");
    return cudaGetLastError();
  }
  const int64_t blocks = (rows + 7) / 8;
  if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
  bwd_rowterm_kernel<T><<<(unsigned)blocks, 256, 0, s>>>(
      static_cast<const T *>(a.o), static_cast<const T *>(a.dout), a.dsum, a.f.Hq, a.f.Sq, a.f.D,
      a.sod[0], a.sod[1], a.sod[2], a.sdo[0], a.sdo[1], a.sdo[2], rows);
  note_launch("bwd_rowterm_kernel");
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_rowterm(const BwdArgs &a, cudaStream_t s) {
  switch (a.f.dt) {
    case RA_F32: return rowterm_typed<float>(a, s);
    case RA_BF16: return rowterm_typed<__nv_bfloat16>(a, s);
    case RA_F16: return rowterm_typed<__half>(a, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_attn_bwd_simt(const BwdArgs &a, cudaStream_t s) {
  if (a.f.dt != RA_F32) return cudaErrorNotSupported;
  const BwdSimtParams p = simt_params(a);
  const int D = a.f.D;
  const size_t smem = ((size_t)2 * kTile * (D + 1) + (size_t)kTile * D + 2 * kTile +
                       (size_t)kRows * 3 * D) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(bwd_dq_simt_kernel<float>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bwd_dkdv_simt_kernel<float>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (a.f.Sq > 0) {
    const dim3 gq((unsigned)((a.f.Sq + kRows - 1) / kRows), (unsigned)a.f.Hq, (unsigned)a.f.B);
    bwd_dq_simt_kernel<float><<<gq, kRows * 32, smem, s>>>(p);
    note_launch("bwd_dq_simt_kernel");
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const dim3 gk((unsigned)((a.f.Sk + kRows - 1) / kRows), (unsigned)a.f.Hkv, (unsigned)a.f.B);
  bwd_dkdv_simt_kernel<float><<<gk, kRows * 32, smem, s>>>(p);
  note_launch("bwd_dkdv_simt_kernel");
  return cudaGetLastError();
}

}  // namespace ra

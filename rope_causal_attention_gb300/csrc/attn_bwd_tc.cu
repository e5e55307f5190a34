// Backward of causal attention with RoPE fused in, on the sm_103a tensor
// cores (tcgen05 + tensor memory + TMA), bf16/fp16, head dims 64 and 128.
//
// Mathematics ("RoPE and FlashAttention: relative positions and online
// softmax", section 5: the probabilities are rebuilt from Q, K and the
// forward's LSE instead of being stored; sections 1-2: the rotation):
//   q~_i = R(kv_offset + i) q_i,  k~_j = R(j) k_j  (fp16 operands, as in the
//   forward, so the rebuilt scores are the forward's);
//   P_ij = 2^(s_ij log2e - LSE_i log2e) on admissible pairs, 0 elsewhere;
//   dP = dO V^T,  dS = P o (dP - D),  D_i = <dO_i, O_i> (row-term kernel);
//   dV = P^T dO,  dk~ = scale dS^T q~,  dq~ = scale dS k~;
//   dk_j = R(j)^T dk~_j,  dq_i = R(kv_offset + i)^T dq~_i.
//
// GB300 design.  A memory-bound pass first rotates Q and K once into fp16
// workspace tensors (every query and key row is used by many tiles, and
// rotating them tile by tile inside the kernels cost more issue slots than
// the products), so both kernels load all four operands with TMA.  Then two
// kernels, neither using atomics:
//   bwd_dkdv_tc_kernel: one CTA per (key tile of 128 rows, kv head, batch);
//     K~ and V stay in shared memory, and the CTA walks every (q-head of the
//     kv group, query tile) that sees its keys, in halves of 64 queries.
//     Half v uses TMEM buffer b = v & 1:
//       S^T  = K~ Q~^T   (TMEM cols 256 + 128 b ..; M = 128 keys, N = 64 queries)
//       dP^T = V  dO^T   (the next 64 columns)
//       threads: P^T (input dtype) over S^T, dS^T (fp16) over dP^T
//       dV  += P^T  dO   (TS: A = P^T in TMEM, B = dO read MN-major, K = 64)
//       dK~ += dS^T Q~   (TS: A = dS^T in TMEM, B = Q~ read MN-major)
//     Two warps issue the products, one per buffer, so the next half's
//     S^T and dP^T overlap this half's thread work and one warp's waits are
//     covered by the other's products.  dV and dK~ accumulate in TMEM
//     cols 0..2D-1 over the whole walk, so the group's q-heads are summed
//     inside the CTA.
//   bwd_dq_tc_kernel: one CTA per (query tile, q-head, batch); Q~ and dO stay
//     in shared memory, key tiles stream.  S alternates between two TMEM
//     slots (cols 0..127, 128..255), dP has one (256..383) that the threads
//     release as soon as they have read it, dQ~ accumulates in 384..: the
//     two MMA-issuing warps (even and odd key tiles, one S slot each) let
//     the tensor core compute the next tile's S and dP while the threads
//     turn this tile's into dS.
//   The epilogues scale, rotate back with R^T (the table's sine negated) and
//   store in the input dtype.  A shared-memory tile in the 128-byte swizzled
//   K-major layout doubles as the MN-major operand of the transposed product,
//   so each operand tile is loaded once.
// Roles.  dQ (352 threads): warps 0-7 compute P and dS, two warps per TMEM
// lane quadrant, each on half of the 128 columns (they pack their 16-bit
// results into columns they have already read: +0 for the first half, +64
// for the second, and the TS products address the two halves per k-step);
// warp 8 issues the TMA loads; warp 9 allocates TMEM; warps 9 and 10 issue
// the MMAs of the even and the odd key tiles.
// dK/dV (352 threads): warps 0-7 compute P^T and dS^T, two warps per lane
// quadrant, each on 32 of a half's 64 query columns, i.e. two 16-query
// k-blocks (each block's P^T and dS^T packed over the first 8 of its own 16
// S^T and dP^T columns); warp 8 issues the TMA loads and stages the row
// statistics (one unit ahead); warp 9 allocates TMEM; warps 9 and 10 issue
// the MMAs of the even and the odd halves.  (With 16 compute warps on 16
// columns each the kernel was ~2 % slower: the issuers then shared their
// sub-partitions with four busy warps instead of two.)  The MMA warps issue warp-wide (one elected lane per
// instruction).  Every mbarrier wait is bounded (RA_ERR_DEVICE_TIMEOUT,
// abort flag, drain).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>

#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace ra {
namespace {

using namespace ptx;

constexpr int kThreads = 352;  // dQ: 8 compute warps, TMA, two MMA issuers
constexpr int kWarpTma = 8, kWarpMma = 9;  // and kWarpMma + 1
// dK/dV: 8 compute warps (2 per SM sub-partition: each owns 32 of a half's
// 64 query columns), then the TMA and MMA warps
constexpr int kThreadsK = 352;
constexpr int kWarpTmaK = 8, kWarpMmaK = 9;  // and kWarpMmaK + 1: the second MMA issuer
constexpr uint32_t kTmemCols = 512;
constexpr long long kTimeoutCycles = 1LL << 32;  // about two seconds
constexpr int kBandKv = 4;                       // kv heads per band of the launch orders
constexpr float kLog2e = 1.4426950408889634f;

template <typename T> struct Pack16;
template <> struct Pack16<__nv_bfloat16> {
  static __device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
  }
};
template <> struct Pack16<__half> {
  static __device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
  }
};
__device__ __forceinline__ uint32_t f16x2(float lo, float hi) { return Pack16<__half>::pack2(lo, hi); }

template <int D> struct BCfg {
  static constexpr int TILE = 128 * D * 2;  // 128 rows of 16-bit values
  static constexpr int SUBT = 16384;        // one 64-column sub-tile
  static constexpr int NS = D == 128 ? 2 : 3;
  // dk/dv kernel: K~ | V | (Q~, dO) ring | row stats ring (LSE log2, D)
  static constexpr int K_OFF_K = 0, K_OFF_V = TILE, K_OFF_Q = 2 * TILE;
  static constexpr int K_OFF_DO = K_OFF_Q + NS * TILE;
  static constexpr int K_OFF_ST = K_OFF_DO + NS * TILE;
  static constexpr int K_OFF_BAR = K_OFF_ST + NS * 1024;
  // S^T, dP^T and P^T/dS^T per 64-query half-unit, two TMEM buffers: one
  // barrier of each per buffer
  static constexpr int KB_KVFULL = 0, KB_QFULL = 1, KB_QEMPTY = 1 + NS, KB_SFULL = 1 + 2 * NS,
                       KB_DPFULL = 3 + 2 * NS, KB_PFULL = 5 + 2 * NS, KB_ACC = 7 + 2 * NS,
                       KB_DONE = 8 + 2 * NS, KB_DVDK = 9 + 2 * NS, KB_N = 10 + 2 * NS;
  static constexpr int K_OFF_MISC = K_OFF_BAR + KB_N * 8;
  static constexpr int K_SMEM = K_OFF_MISC + 16 + 1024;
  // dq kernel: Q~ | dO | K~ ring (NSK) | V ring (NSV)
  static constexpr int NSK = 3, NSV = D == 128 ? 2 : 3;
  static constexpr int Q_OFF_Q = 0, Q_OFF_DO = TILE, Q_OFF_K = 2 * TILE;
  static constexpr int Q_OFF_V = Q_OFF_K + NSK * TILE;
  static constexpr int Q_OFF_BAR = Q_OFF_V + NSV * TILE;
  static constexpr int QB_QFULL = 0, QB_KFULL = 1, QB_KEMPTY = 1 + NSK,
                       QB_VFULL = 1 + 2 * NSK, QB_VEMPTY = 1 + 2 * NSK + NSV,
                       QB_SFULL = 1 + 2 * NSK + 2 * NSV,  // two S slots
                       QB_DPFULL = 3 + 2 * NSK + 2 * NSV, QB_DPFREE = 4 + 2 * NSK + 2 * NSV,
                       QB_PFULL = 5 + 2 * NSK + 2 * NSV,  // two S slots
                       QB_ACC = 7 + 2 * NSK + 2 * NSV, QB_DONE = 8 + 2 * NSK + 2 * NSV,
                       QB_DQ = 9 + 2 * NSK + 2 * NSV, QB_N = 10 + 2 * NSK + 2 * NSV;
  static constexpr int Q_OFF_MISC = Q_OFF_BAR + QB_N * 8;
  static constexpr int Q_SMEM = Q_OFF_MISC + 16 + 1024;
  static_assert(K_SMEM <= 232448 && Q_SMEM <= 232448, "shared memory");
  // the epilogues stage 128 padded fp32 rows over the rings
  static_assert(128 * (D + 1) * 4 <= 2 * NS * TILE && 128 * (D + 1) * 4 <= NSK * TILE,
                "epilogue scratch");
};

struct BwdTcParams {
  const float *lse, *dsum;
  void *dq, *dk, *dv;
  int64_t sdq0, sdq1, sdq2, sdk0, sdk1, sdk2, sdv0, sdv1, sdv2;
  int64_t Sq, Sk, off;
  int B, Hq, Hkv, G, n_qt, n_kt;
  // launch order: (batch, kv head) units per band of the dK/dV grid and
  // (batch, q-head) units per band of the dQ grid (all units: no bands)
  int kv_band, q_band;
  int apply_rope, rot_dim, layout;
  const float *cos_t, *sin_t;
  float scale, scale_log2;
  // tensor-map dims 1..3 -> logical coordinate (0 row, 1 head, 2 batch)
  int qperm[3], kperm[3], vperm[3], operm[3];
  int *status;
};

struct Ctl {
  volatile int *abort;
  int *status;
};

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctl &c) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*c.abort) return false;
    if (clock64() - t0 > kTimeoutCycles) {
      *c.abort = 1;
      record_status(c.status, RA_ERR_DEVICE_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ void wait_bar_drain(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > kTimeoutCycles) return;
}

// Bounded wait taken by a whole warp (the MMA issuers run warp-wide).
__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity, const Ctl &c) {
  return __all_sync(0xffffffffu, wait_bar(bar, parity, c));
}

__device__ __forceinline__ int map_coord(const int perm, int row, int head, int b) {
  return perm == 0 ? row : (perm == 1 ? head : b);
}

// One 128-row tile (D/64 boxes of 64 columns) of a [B][H][S][D] tensor map.
template <int D>
__device__ __forceinline__ void tma_tile(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                         const int perm[3], int row, int head, int b) {
#pragma unroll
  for (int sub = 0; sub < D / 64; ++sub)
    tma_load_4d(dst + sub * 16384, map, bar, sub * 64, map_coord(perm[0], row, head, b),
                map_coord(perm[1], row, head, b), map_coord(perm[2], row, head, b));
}

// Dim e of a padded fp32 row rotated back with R(pos)^T.
__device__ __forceinline__ float rot_back(const float *row, int e, int64_t pos,
                                          const BwdTcParams &p) {
  if (!p.apply_rope || e >= p.rot_dim) return row[e];
  const int half = p.rot_dim >> 1;
  bool low;
  int i, partner;
  if (p.layout == RA_NEOX) {
    low = e < half;
    i = low ? e : e - half;
    partner = low ? e + half : e - half;
  } else {
    low = (e & 1) == 0;
    i = e >> 1;
    partner = e ^ 1;
  }
  const float c = __ldg(p.cos_t + pos * half + i);
  const float s = __ldg(p.sin_t + pos * half + i);
  return low ? row[e] * c + row[partner] * s : row[e] * c - row[partner] * s;
}

// Stores 8-dim groups [g0, g1) of a padded fp32 row as dtype, rotated back
// at pos when `rotate` (16-byte stores).
template <int D, typename TIn>
__device__ __forceinline__ void store_row(const float *row, bool rotate, int64_t pos, TIn *dst,
                                          int g0, int g1, const BwdTcParams &p) {
#pragma unroll 1
  for (int g = g0; g < g1; ++g) {
    float v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = rotate ? rot_back(row, 8 * g + e, pos, p) : row[8 * g + e];
    reinterpret_cast<uint4 *>(dst)[g] =
        make_uint4(Pack16<TIn>::pack2(v[0], v[1]), Pack16<TIn>::pack2(v[2], v[3]),
                   Pack16<TIn>::pack2(v[4], v[5]), Pack16<TIn>::pack2(v[6], v[7]));
  }
}

// ================================================================ rotation
// Rotated fp16 copy of a [B][H][S][D] tensor (row s at position pos0 + s),
// written contiguous.  A row's work items are its rotation units (NeoX: a
// 16-byte chunk of the low half with its high-half partner; GPT-J: a 16-byte
// chunk of whole pairs), then the 16-byte chunks of the unrotated tail;
// without rotation every chunk is a tail chunk.  One thread per item: fp32
// arithmetic with the fp32 table (float4 loads: the host passes 16-byte
// aligned tables and whole 8-element units), one rounding to fp16.  The
// input is read once, with the streaming cache hint.  A value that does not
// round to a finite fp16 records RA_ERR_RANGE.
__host__ __device__ inline int rotate_units(int D, int apply_rope, int rot_dim, int layout) {
  if (!apply_rope) return D >> 3;
  return (layout == RA_NEOX ? rot_dim >> 4 : rot_dim >> 3) + ((D - rot_dim) >> 3);
}

__device__ __forceinline__ void ld_f4x2(const float *p, float *f) {
  const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
  const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

template <typename TIn>
__global__ void __launch_bounds__(256) bwd_rotate_f16_kernel(const TIn *__restrict__ x, int H,
                                                             int64_t S, int D, int64_t s0,
                                                             int64_t s1, int64_t s2,
                                                             int64_t pos0, __half *__restrict__ out,
                                                             int apply_rope, int rot_dim,
                                                             int layout, const float *cos_t,
                                                             const float *sin_t, int64_t n,
                                                             int *status) {
  const int half = rot_dim >> 1;
  uint32_t bad = 0;
  const int per_row = rotate_units(D, apply_rope, rot_dim, layout);
  const int nr = apply_rope ? (layout == RA_NEOX ? rot_dim >> 4 : rot_dim >> 3) : 0;
  const int tail0 = apply_rope ? rot_dim >> 3 : 0;  // first tail chunk
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = idx / per_row;
    const int u = (int)(idx - r * per_row);
    const int64_t s = r % S, h = (r / S) % H, b = r / (S * H);
    const TIn *src = x + b * s0 + h * s1 + s * s2;
    __half *dst = out + r * D;
    if (u >= nr) {  // a chunk of the unrotated tail
      const int c = tail0 + (u - nr);
      float a[8];
      unpack16<TIn>(__ldcs(reinterpret_cast<const uint4 *>(src + 8 * c)), a);
      const uint4 w = pack16<__half>(a);
      bad |= f16x2_nonfinite(w.x) | f16x2_nonfinite(w.y) | f16x2_nonfinite(w.z) |
             f16x2_nonfinite(w.w);
      *reinterpret_cast<uint4 *>(dst + 8 * c) = w;
      continue;
    }
    const float *cr = cos_t + (pos0 + s) * half, *sr = sin_t + (pos0 + s) * half;
    if (layout == RA_NEOX) {
      float lo[8], hi[8], cs[8], sn[8], a[8], bb[8];
      unpack16<TIn>(__ldcs(reinterpret_cast<const uint4 *>(src + 8 * u)), lo);
      unpack16<TIn>(__ldcs(reinterpret_cast<const uint4 *>(src + 8 * u + half)), hi);
      ld_f4x2(cr + 8 * u, cs);
      ld_f4x2(sr + 8 * u, sn);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        a[e] = lo[e] * cs[e] - hi[e] * sn[e];
        bb[e] = hi[e] * cs[e] + lo[e] * sn[e];
      }
      const uint4 wa = pack16<__half>(a), wb = pack16<__half>(bb);
      bad |= f16x2_nonfinite(wa.x) | f16x2_nonfinite(wa.y) | f16x2_nonfinite(wa.z) |
             f16x2_nonfinite(wa.w) | f16x2_nonfinite(wb.x) | f16x2_nonfinite(wb.y) |
             f16x2_nonfinite(wb.z) | f16x2_nonfinite(wb.w);
      *reinterpret_cast<uint4 *>(dst + 8 * u) = wa;
      *reinterpret_cast<uint4 *>(dst + 8 * u + half) = wb;
    } else {
      float xv[8], y[8];
      unpack16<TIn>(__ldcs(reinterpret_cast<const uint4 *>(src + 8 * u)), xv);
      const float4 cs = __ldg(reinterpret_cast<const float4 *>(cr + 4 * u));
      const float4 sn = __ldg(reinterpret_cast<const float4 *>(sr + 4 * u));
      const float c4[4] = {cs.x, cs.y, cs.z, cs.w}, s4[4] = {sn.x, sn.y, sn.z, sn.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        y[2 * e] = xv[2 * e] * c4[e] - xv[2 * e + 1] * s4[e];
        y[2 * e + 1] = xv[2 * e + 1] * c4[e] + xv[2 * e] * s4[e];
      }
      const uint4 w = pack16<__half>(y);
      bad |= f16x2_nonfinite(w.x) | f16x2_nonfinite(w.y) | f16x2_nonfinite(w.z) |
             f16x2_nonfinite(w.w);
      *reinterpret_cast<uint4 *>(dst + 8 * u) = w;
    }
  }
  record_range_flag(status, bad);
}

// ===================================================================== dK, dV
template <int D, typename TIn>
__global__ void __launch_bounds__(kThreadsK, 1)
    bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tmap_q,
                       const __grid_constant__ CUtensorMap tmap_k,
                       const __grid_constant__ CUtensorMap tmap_v,
                       const __grid_constant__ CUtensorMap tmap_do, const BwdTcParams p) {
  using C = BCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  auto bar = [&](int i) { return sbase + C::K_OFF_BAR + 8u * (uint32_t)i; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::K_OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::K_OFF_MISC + 4);
  const Ctl ctl{abort_flag, p.status};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work: key tile kt (low tiles, seen by the most queries, first),
  // band by band of (batch, kv head) units so that the Q~ and dO of the
  // heads in flight stay in L2
  const int n_u = p.B * p.Hkv;
  const int per_band = p.n_kt * p.kv_band;
  const int band = blockIdx.x / per_band;
  const int rb = blockIdx.x - band * per_band;
  const int ub = min(p.kv_band, n_u - band * p.kv_band);
  const int kt = rb / ub;
  const int unit = band * p.kv_band + rb % ub;
  const int b = unit / p.Hkv, hk = unit % p.Hkv;
  const int64_t j0 = (int64_t)kt * 128;
  const int64_t mf = j0 - p.off < 0 ? 0 : (j0 - p.off) / 128;  // first query tile that sees it
  const int m_first = (int)min(mf, (int64_t)p.n_qt);
  const int per_g = p.n_qt - m_first;
  const int NU = p.G * per_g;  // (q-head, query tile) units

  if (threadIdx.x == 0) {
    mbar_init(bar(C::KB_KVFULL), 1);
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(bar(C::KB_QFULL + i), 33);  // TMA arrive + 32 lanes of row statistics
      mbar_init(bar(C::KB_QEMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::KB_SFULL + i), 1);
      mbar_init(bar(C::KB_DPFULL + i), 1);
      mbar_init(bar(C::KB_PFULL + i), 8);  // one arrive per compute warp
    }
    mbar_init(bar(C::KB_ACC), 1);
    mbar_init(bar(C::KB_DONE), 2);  // both MMA issuers
    mbar_init(bar(C::KB_DVDK), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMmaK) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kWarpTmaK && lane == 0) {
    prefetch_tmap(&tmap_q);
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
    prefetch_tmap(&tmap_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 8) {
    // ========================================================= P^T and dS^T
    // A unit (q-head, 128-query tile) is processed as two halves of 64
    // queries; half v uses TMEM buffer v & 1 (S^T at 256 + 128 (v & 1), dP^T
    // 64 columns further), so the tensor core computes the next half's S^T
    // and dP^T while the threads turn this half's into P^T and dS^T.
    const int qd = warp & 3, cq = warp >> 2;  // TMEM lane quarter, query-column half
    const int t = qd * 32 + lane;  // key row of the tile = TMEM lane
    const uint32_t lanes = tmem + ((uint32_t)(qd * 32) << 16);
    const int64_t j = j0 + t;
    const float sl2 = p.scale_log2;
    const int c0 = 32 * cq;  // query columns [c0, c0 + 32) of every half
    bool ok = true;
    for (int v = 0; v < 2 * NU; ++v) {
      const int u = v >> 1, hh = v & 1, bf = v & 1;
      const int st = u % C::NS;
      const int m = m_first + u % per_g;
      if (hh == 0)
        ok = ok && __all_sync(0xffffffffu, wait_bar(bar(C::KB_QFULL + st), (uint32_t)((u / C::NS) & 1), ctl));
      ok = ok && __all_sync(0xffffffffu, wait_bar(bar(C::KB_SFULL + bf), (uint32_t)((v >> 1) & 1), ctl));
      if (!ok) break;
      tc_fence_after();
      const float4 *lse4 = reinterpret_cast<const float4 *>(smem + C::K_OFF_ST + st * 1024);
      const float4 *dsm4 = lse4 + 32;
      const int q0 = 64 * hh + c0;  // first query row (of the 128-row tile) of this warp
      const int64_t i0 = (int64_t)m * 128 + 64 * hh;
      const bool straddle = j0 + 127 > p.off + i0;
      const int64_t lim = j - p.off - i0;  // half column c sees key j iff c >= lim
      const uint32_t sbuf = lanes + 256u + 128u * (uint32_t)bf;
      // P^T from S^T first: the exponentials overlap the dP^T product, which
      // is only waited for before dS^T
      uint32_t sr[32], dr[32];
      tmem_ld32(sbuf + (uint32_t)c0, sr);
      {
        uint32_t pp[2][8];
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const float4 l4 = lse4[(q0 >> 2) + e4];
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
          for (int k = 0; k < 4; k += 2) {
            const int e = 4 * e4 + k;
            const float2 xa = __ffma2_rn(make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])),
                                         make_float2(sl2, sl2), make_float2(-lv[k], -lv[k + 1]));
            float p0 = ex2(xa.x);
            float p1 = ex2(xa.y);
            if (straddle) {
              if (c0 + e < lim) p0 = 0.f;
              if (c0 + e + 1 < lim) p1 = 0.f;
            }
            pp[e >> 4][(e >> 1) & 7] = Pack16<TIn>::pack2(p0, p1);
            sr[e] = __float_as_uint(p0);
            sr[e + 1] = __float_as_uint(p1);
          }
        }
        // P^T of query blocks 2 cq and 2 cq + 1, each packed over the first
        // 8 of its 16 columns
        tmem_st8(sbuf + (uint32_t)c0, pp[0]);
        tmem_st8(sbuf + (uint32_t)c0 + 16u, pp[1]);
      }
      if (!__all_sync(0xffffffffu, wait_bar(bar(C::KB_DPFULL + bf), (uint32_t)((v >> 1) & 1), ctl))) {
        ok = false;
        break;
      }
      tc_fence_after();
      tmem_ld32(sbuf + 64u + (uint32_t)c0, dr);
      uint32_t pd[2][8];
#pragma unroll
      for (int e4 = 0; e4 < 8; ++e4) {
        const float4 d4 = dsm4[(q0 >> 2) + e4];
        const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
        for (int k = 0; k < 4; k += 2) {
          const int e = 4 * e4 + k;
          const float2 ds = __fmul2_rn(
              make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])),
              __fadd2_rn(make_float2(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])),
                         make_float2(-dv[k], -dv[k + 1])));
          pd[e >> 4][(e >> 1) & 7] = f16x2(ds.x, ds.y);
        }
      }
      tmem_st8(sbuf + 64u + (uint32_t)c0, pd[0]);
      tmem_st8(sbuf + 64u + (uint32_t)c0 + 16u, pd[1]);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::KB_PFULL + bf));
    }
    // ---- epilogue: dV straight from TMEM; dK = R(j)^T (scale dK~) through a
    // padded fp32 row per key (the rotation pairs dims across the two halves).
    // A non-finite accumulator value (a dS^T term past the fp16 range reaches
    // every dK~ dim of its key) records RA_ERR_RANGE.
    const bool acc = ok && NU > 0 &&
                     __all_sync(0xffffffffu, wait_bar(bar(C::KB_ACC), 0u, ctl));
    const bool write = ok && (NU == 0 || acc);
    tc_fence_after();
    float *row = reinterpret_cast<float *>(smem + C::K_OFF_Q) + t * (D + 1);
    TIn *dvd = static_cast<TIn *>(p.dv) + b * p.sdv0 + hk * p.sdv1 + j * p.sdv2;
    TIn *dkd = static_cast<TIn *>(p.dk) + b * p.sdk0 + hk * p.sdk1 + j * p.sdk2;
    const bool row_ok = j < p.Sk;
    constexpr int QD = D / 2;  // dims per column half
    uint32_t bad = 0;
#pragma unroll 1
    for (int c = 0; c < QD / 16; ++c) {
      const int col = QD * cq + 16 * c;
      uint32_t r[16];
      if (acc) tmem_ld16(lanes + (uint32_t)col, r);
      if (acc)
#pragma unroll
        for (int e = 0; e < 16; ++e) bad |= (r[e] & 0x7f800000u) == 0x7f800000u;
      if (write && row_ok) {
        uint4 *d4 = reinterpret_cast<uint4 *>(dvd + col);
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          float v[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) v[e] = acc ? __uint_as_float(r[8 * g + e]) : 0.f;
          d4[g] = make_uint4(Pack16<TIn>::pack2(v[0], v[1]), Pack16<TIn>::pack2(v[2], v[3]),
                             Pack16<TIn>::pack2(v[4], v[5]), Pack16<TIn>::pack2(v[6], v[7]));
        }
      }
      if (acc) tmem_ld16(lanes + (uint32_t)(D + col), r);
      if (acc)
#pragma unroll
        for (int e = 0; e < 16; ++e) bad |= (r[e] & 0x7f800000u) == 0x7f800000u;
#pragma unroll
      for (int e = 0; e < 16; ++e) row[col + e] = acc ? __uint_as_float(r[e]) * p.scale : 0.f;
    }
    record_range_flag(p.status, bad);
    named_bar_sync(1, 256);  // both halves of every row are in shared memory
    if (write && row_ok) store_row<D, TIn>(row, true, j, dkd, cq * (D / 16), (cq + 1) * (D / 16), p);
  } else if (warp == kWarpTmaK) {
    // ============================================= TMA and row statistics
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(C::KB_KVFULL), (uint32_t)(2 * C::TILE));
      tma_tile<D>(sbase + C::K_OFF_K, &tmap_k, bar(C::KB_KVFULL), p.kperm, (int)j0, hk, b);
      tma_tile<D>(sbase + C::K_OFF_V, &tmap_v, bar(C::KB_KVFULL), p.vperm, (int)j0, hk, b);
    }
    // LSE (log2 units) and D of a unit's 128 rows, 4 rows per lane; rows past
    // Sq get P = 0.  They are loaded one unit ahead, so their latency
    // overlaps the wait for the ring instead of holding back the unit's QFULL.
    float nl[4], nd[4];
    auto load_stats = [&](int u) {
      const int g = u / per_g, m = m_first + u % per_g, h = hk * p.G + g;
      const int64_t rb = ((int64_t)b * p.Hq + h) * p.Sq + (int64_t)m * 128;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int t = lane + 32 * k;
        const bool in = (int64_t)m * 128 + t < p.Sq;
        nl[k] = in ? p.lse[rb + t] * kLog2e : INFINITY;
        nd[k] = in ? p.dsum[rb + t] : 0.f;
      }
    };
    if (NU > 0) load_stats(0);
    int issued = 0;
    for (int u = 0; u < NU; ++u) {
      const int st = u % C::NS;
      if (u >= C::NS &&
          !__all_sync(0xffffffffu, wait_bar(bar(C::KB_QEMPTY + st), (uint32_t)((u / C::NS - 1) & 1), ctl)))
        break;
      const int g = u / per_g, m = m_first + u % per_g, h = hk * p.G + g;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(C::KB_QFULL + st), (uint32_t)(2 * C::TILE));
        tma_tile<D>(sbase + C::K_OFF_Q + st * C::TILE, &tmap_q, bar(C::KB_QFULL + st), p.qperm,
                    m * 128, h, b);
        tma_tile<D>(sbase + C::K_OFF_DO + st * C::TILE, &tmap_do, bar(C::KB_QFULL + st), p.operm,
                    m * 128, h, b);
      }
      float *sv = reinterpret_cast<float *>(smem + C::K_OFF_ST + st * 1024);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        sv[lane + 32 * k] = nl[k];
        sv[128 + lane + 32 * k] = nd[k];
      }
      mbar_arrive(bar(C::KB_QFULL + st));
      if (u + 1 < NU) load_stats(u + 1);
      issued = u + 1;
    }
    if (lane == 0) {  // copies in flight land before the block exits
      wait_bar_drain(bar(C::KB_KVFULL), 0u);
      if (*abort_flag)
        for (int u = max(0, issued - C::NS); u < issued; ++u)
          wait_bar_drain(bar(C::KB_QFULL + u % C::NS), (uint32_t)((u / C::NS) & 1));
    }
  } else {  // MMA issuers: two whole warps, one elected lane of each issues
    // =================================================================== MMA
    // Warp kWarpMmaK issues every product of the even halves (TMEM buffer 0),
    // warp kWarpMmaK + 1 those of the odd halves (buffer 1).  One issuing
    // warp alone cannot keep the tensor core busy: its queue holds only a
    // few products, and its waits and bookkeeping between groups outlast
    // them; with two, one issues while the other waits.  Each warp keeps
    // the in-order rule on its own buffer (S^T of half v + 2 after dV/dK of
    // half v).  The dV/dK accumulations alternate between the warps; each
    // waits for the previous half's dV/dK to complete first, so they run in
    // half order (the first one initialises the accumulators, and the
    // result does not depend on timing).
    const int hb = warp - kWarpMmaK;  // halves v with v % 2 == hb
    constexpr uint32_t ab = std::is_same<TIn, __nv_bfloat16>::value ? 1u : 0u;
    constexpr uint32_t IDESC_S = idesc_f16(0u, 0u, 64);    // fp16 K~ x Q~^T, 64 queries
    constexpr uint32_t IDESC_DP = idesc_f16(ab, 0u, 64);   // V x dO^T, 64 queries
    constexpr uint32_t IDESC_DV = idesc_f16(ab, 1u, D);    // P^T x dO (dO MN-major)
    constexpr uint32_t IDESC_DK = idesc_f16(0u, 1u, D);    // dS^T x Q~ (Q~ MN-major)
    constexpr uint32_t HI = sdesc_hi_sw128(1024);
    const uint32_t k_lo = sdesc_lo(sbase + C::K_OFF_K, 16);
    const uint32_t v_lo = sdesc_lo(sbase + C::K_OFF_V, 16);
    const uint32_t q_lo0 = sdesc_lo(sbase + C::K_OFF_Q, 16);
    const uint32_t do_lo0 = sdesc_lo(sbase + C::K_OFF_DO, 16);
    const uint32_t qmn_lo0 = sdesc_lo(sbase + C::K_OFF_Q, C::SUBT);
    const uint32_t domn_lo0 = sdesc_lo(sbase + C::K_OFF_DO, C::SUBT);
    const uint32_t sb = tmem + 256u + 128u * (uint32_t)hb;  // this warp's S^T | dP^T buffer
    bool ok = NU == 0 || wait_all(bar(C::KB_KVFULL), 0u, ctl);
    for (int v = hb; ok && v < 2 * NU; v += 2) {
      const int u = v >> 1, st = u % C::NS;
      const uint32_t so = (uint32_t)((st * C::TILE + hb * 8192) >> 4);
      if (!wait_all(bar(C::KB_QFULL + st), (uint32_t)((u / C::NS) & 1), ctl)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (uint32_t)(((kk >> 2) * C::SUBT + (kk & 3) * 32) >> 4);
        mma_ss_w(sb, sdesc_join(k_lo + off, HI), sdesc_join(q_lo0 + so + off, HI), IDESC_S,
                 kk > 0 ? 1u : 0u);
      }
      tc_commit_w(bar(C::KB_SFULL + hb));
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (uint32_t)(((kk >> 2) * C::SUBT + (kk & 3) * 32) >> 4);
        mma_ss_w(sb + 64u, sdesc_join(v_lo + off, HI), sdesc_join(do_lo0 + so + off, HI),
                 IDESC_DP, kk > 0 ? 1u : 0u);
      }
      tc_commit_w(bar(C::KB_DPFULL + hb));
      // P^T and dS^T of half v in the buffer, and the previous half's
      // accumulation complete
      if (!wait_all(bar(C::KB_PFULL + hb), (uint32_t)((v >> 1) & 1), ctl) ||
          (v >= 1 && !wait_all(bar(C::KB_DVDK), (uint32_t)((v - 1) & 1), ctl))) {
        ok = false;
        break;
      }
      tc_fence_after();
      // dV += P^T dO and dK~ += dS^T Q~ (K = 64 queries; query block kk of
      // 16 is packed over columns [16 kk, 16 kk + 8) of the buffer)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_ts_w(tmem, sb + (uint32_t)(16 * kk),
                 sdesc_join(domn_lo0 + so + (uint32_t)(kk * 2048 >> 4), HI), IDESC_DV,
                 (v > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_ts_w(tmem + (uint32_t)D, sb + 64u + (uint32_t)(16 * kk),
                 sdesc_join(qmn_lo0 + so + (uint32_t)(kk * 2048 >> 4), HI), IDESC_DK,
                 (v > 0 || kk > 0) ? 1u : 0u);
      tc_commit_w(bar(C::KB_DVDK));
      // the odd half closes its unit: every product that read the ring slot
      // has completed (its own in issue order, the even half's before its
      // dV/dK started)
      if (hb == 1) tc_commit_w(bar(C::KB_QEMPTY + st));
      if (v == 2 * NU - 1) tc_commit_w(bar(C::KB_ACC));
    }
    tc_commit_w(bar(C::KB_DONE));
    wait_bar_drain(bar(C::KB_DONE), 0u);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMmaK) tmem_dealloc(tmem, kTmemCols);
}


// 2^x for x <= ~0 on the FMA pipe: Cody-Waite split x = j + f (j the nearest
// integer, found by adding 1.5 * 2^23), 2^f on [-0.5, 0.5] by a degree-3
// minimax polynomial (relative error below 7.5e-5), 2^j added to the
// exponent field.  Inputs below -125 are clamped (the result is then a
// tiny normal number, not 0).
__device__ __forceinline__ float2 ex2_fma2(float2 x) {
  x.x = fmaxf(x.x, -125.f);
  x.y = fmaxf(x.y, -125.f);
  const float2 y = __fadd2_rn(x, make_float2(12582912.f, 12582912.f));
  const float2 jf = __fadd2_rn(y, make_float2(-12582912.f, -12582912.f));
  const float2 f = __ffma2_rn(jf, make_float2(-1.f, -1.f), x);
  float2 p = __ffma2_rn(make_float2(0.0551716685295105f, 0.0551716685295105f), f,
                        make_float2(0.2426111251115799f, 0.2426111251115799f));
  p = __ffma2_rn(p, f, make_float2(0.6932609677314758f, 0.6932609677314758f));
  p = __ffma2_rn(p, f, make_float2(0.9999280571937561f, 0.9999280571937561f));
  return make_float2(__int_as_float(__float_as_int(p.x) + (__float_as_int(y.x) << 23)),
                     __int_as_float(__float_as_int(p.y) + (__float_as_int(y.y) << 23)));
}

// ========================================================================= dQ
template <int D, typename TIn>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tmap_q,
                     const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v,
                     const __grid_constant__ CUtensorMap tmap_do, const BwdTcParams p) {
  using C = BCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  auto bar = [&](int i) { return sbase + C::Q_OFF_BAR + 8u * (uint32_t)i; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::Q_OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::Q_OFF_MISC + 4);
  const Ctl ctl{abort_flag, p.status};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work: query tile m (last tiles, which see the most keys, first),
  // band by band of (batch, q-head) units so that the K~ and V of the kv
  // heads in flight stay in L2
  const int n_u = p.B * p.Hq;
  const int per_band = p.n_qt * p.q_band;
  const int band = blockIdx.x / per_band;
  const int rb = blockIdx.x - band * per_band;
  const int ub = min(p.q_band, n_u - band * p.q_band);
  const int m = p.n_qt - 1 - rb / ub;
  const int unit = band * p.q_band + rb % ub;
  const int b = unit / p.Hq, h = unit % p.Hq;
  const int hk = h / p.G;
  const int64_t i0 = (int64_t)m * 128;
  const int64_t last_pos = p.off + min(i0 + 127, p.Sq - 1);
  const int N = (int)min((int64_t)p.n_kt, last_pos / 128 + 1);  // key tiles seen (>= 1)

  if (threadIdx.x == 0) {
    mbar_init(bar(C::QB_QFULL), 1);
    for (int i = 0; i < C::NSK; ++i) {
      mbar_init(bar(C::QB_KFULL + i), 1);
      mbar_init(bar(C::QB_KEMPTY + i), 1);
    }
    for (int i = 0; i < C::NSV; ++i) {
      mbar_init(bar(C::QB_VFULL + i), 1);
      mbar_init(bar(C::QB_VEMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::QB_SFULL + i), 1);
      mbar_init(bar(C::QB_PFULL + i), 8);  // one arrive per compute warp
    }
    mbar_init(bar(C::QB_DPFULL), 1);
    mbar_init(bar(C::QB_DPFREE), 8);
    mbar_init(bar(C::QB_ACC), 1);
    mbar_init(bar(C::QB_DONE), 2);  // both MMA issuers
    mbar_init(bar(C::QB_DQ), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kWarpTma && lane == 0) {
    prefetch_tmap(&tmap_q);
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
    prefetch_tmap(&tmap_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 8) {
    // ================================================================== dS
    const int qd = warp & 3, hf = warp >> 2;
    const int t = qd * 32 + lane;  // query row of the tile = TMEM lane
    const uint32_t lanes = tmem + ((uint32_t)(qd * 32) << 16);
    const int64_t i = i0 + t;
    const bool row_ok = i < p.Sq;
    const int64_t r = ((int64_t)b * p.Hq + h) * p.Sq + i;
    const float lse2 = row_ok ? p.lse[r] * kLog2e : INFINITY;  // rows past Sq: P = 0
    const float dsum = row_ok ? p.dsum[r] : 0.f;
    const float sl2 = p.scale_log2;
    const int64_t qpos = p.off + i;
    bool ok = true;
    for (int n = 0; n < N; ++n) {
      const int sl = n & 1;  // S slot of this key tile (TMEM cols 128 sl ..)
      ok = ok && __all_sync(0xffffffffu, wait_bar(bar(C::QB_SFULL + sl), (uint32_t)((n >> 1) & 1), ctl));
      if (!ok) break;
      tc_fence_after();
      const int64_t jt = (int64_t)n * 128;
      const bool straddle = (jt + 127 > p.off + i0) || (jt + 127 >= p.Sk);
      // key column c is admissible iff c <= lim
      const int64_t lim = min(qpos, p.Sk - 1) - jt;
      const uint32_t sbase_t = lanes + (uint32_t)(128 * sl);
      // P from S first (kept in the S registers): the exponentials overlap
      // the dP product, which is only waited for before dS
      uint32_t sr[64];
      tmem_ld64(sbase_t + (uint32_t)(64 * hf), sr);
#pragma unroll
      for (int x = 0; x < 64; x += 2) {
        const int c = 64 * hf + x;
        const float2 xa = __ffma2_rn(make_float2(__uint_as_float(sr[x]), __uint_as_float(sr[x + 1])),
                                     make_float2(sl2, sl2), make_float2(-lse2, -lse2));
        float p0, p1;
        if (x < 8) {  // an eighth of the exponentials on the FMA pipe
          const float2 pe = ex2_fma2(xa);
          p0 = pe.x;
          p1 = pe.y;
        } else {
          p0 = ex2(xa.x);
          p1 = ex2(xa.y);
        }
        if (straddle) {
          if (c > lim) p0 = 0.f;
          if (c + 1 > lim) p1 = 0.f;
        }
        sr[x] = __float_as_uint(p0);
        sr[x + 1] = __float_as_uint(p1);
      }
      ok = __all_sync(0xffffffffu, wait_bar(bar(C::QB_DPFULL), (uint32_t)(n & 1), ctl));
      if (!ok) break;
      tc_fence_after();
      // dP, then release its columns so the next tile's dP can start
      uint32_t dr[64];
      tmem_ld64(lanes + 256u + (uint32_t)(64 * hf), dr);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::QB_DPFREE));
#pragma unroll
      for (int bt = 0; bt < 2; ++bt) {
        uint32_t pd[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int x = 32 * bt + e;
          const float2 ds = __fmul2_rn(
              make_float2(__uint_as_float(sr[x]), __uint_as_float(sr[x + 1])),
              __fadd2_rn(make_float2(__uint_as_float(dr[x]), __uint_as_float(dr[x + 1])),
                         make_float2(-dsum, -dsum)));
          pd[e >> 1] = f16x2(ds.x, ds.y);
        }
        // packed into columns this warp has already read: [64 hf + 16 bt, +16)
        tmem_st16(sbase_t + (uint32_t)(64 * hf + 16 * bt), pd);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::QB_PFULL + sl));
    }
    // ---- epilogue: dq = R(kv_offset + i)^T (scale dQ~) through a padded row
    const bool acc = ok && __all_sync(0xffffffffu, wait_bar(bar(C::QB_ACC), 0u, ctl));
    tc_fence_after();
    float *row = reinterpret_cast<float *>(smem + C::Q_OFF_K) + t * (D + 1);
    constexpr int HD = D / 2;
    uint32_t bad = 0;  // a non-finite dQ~ value: a dS term past the fp16 range
#pragma unroll 1
    for (int c = 0; c < HD / 32; ++c) {
      const int col = HD * hf + 32 * c;
      uint32_t rr[32];
      if (acc) tmem_ld32(lanes + 384u + (uint32_t)col, rr);
      if (acc)
#pragma unroll
        for (int e = 0; e < 32; ++e) bad |= (rr[e] & 0x7f800000u) == 0x7f800000u;
#pragma unroll
      for (int e = 0; e < 32; ++e) row[col + e] = acc ? __uint_as_float(rr[e]) * p.scale : 0.f;
    }
    record_range_flag(p.status, bad);
    named_bar_sync(1, 256);  // both halves of every row are in shared memory
    if (acc && row_ok)
      store_row<D, TIn>(row, true, qpos,
                        static_cast<TIn *>(p.dq) + b * p.sdq0 + h * p.sdq1 + i * p.sdq2,
                        hf * (D / 16), (hf + 1) * (D / 16), p);
  } else if (warp == kWarpTma) {
    // =================================================================== TMA
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(C::QB_QFULL), (uint32_t)(2 * C::TILE));
      tma_tile<D>(sbase + C::Q_OFF_Q, &tmap_q, bar(C::QB_QFULL), p.qperm, (int)i0, h, b);
      tma_tile<D>(sbase + C::Q_OFF_DO, &tmap_do, bar(C::QB_QFULL), p.operm, (int)i0, h, b);
      // K~ and V tiles of key tile n; K~(n) is released after dQ~(n), V(n) after dP(n)
      int nk = 0, nv = 0;
      bool live = true;
      while (live && (nk < N || nv < N)) {
        bool progressed = false;
        if (nk < N && (nk < C::NSK || mbar_try_wait(bar(C::QB_KEMPTY + nk % C::NSK),
                                                    (uint32_t)((nk / C::NSK - 1) & 1)))) {
          const int st = nk % C::NSK;
          mbar_arrive_expect_tx(bar(C::QB_KFULL + st), (uint32_t)C::TILE);
          tma_tile<D>(sbase + C::Q_OFF_K + st * C::TILE, &tmap_k, bar(C::QB_KFULL + st), p.kperm,
                      nk * 128, hk, b);
          ++nk;
          progressed = true;
        }
        if (nv < N && (nv < C::NSV || mbar_try_wait(bar(C::QB_VEMPTY + nv % C::NSV),
                                                    (uint32_t)((nv / C::NSV - 1) & 1)))) {
          const int st = nv % C::NSV;
          mbar_arrive_expect_tx(bar(C::QB_VFULL + st), (uint32_t)C::TILE);
          tma_tile<D>(sbase + C::Q_OFF_V + st * C::TILE, &tmap_v, bar(C::QB_VFULL + st), p.vperm,
                      nv * 128, hk, b);
          ++nv;
          progressed = true;
        }
        if (!progressed) {
          // both rings full: wait (bounded) for the release the MMA needs first
          const bool k_next = nk < N && (nv >= N || nk <= nv);
          const uint32_t eb = k_next ? bar(C::QB_KEMPTY + nk % C::NSK) : bar(C::QB_VEMPTY + nv % C::NSV);
          const uint32_t ep = k_next ? (uint32_t)((nk / C::NSK - 1) & 1) : (uint32_t)((nv / C::NSV - 1) & 1);
          live = wait_bar(eb, ep, ctl);
        }
      }
      wait_bar_drain(bar(C::QB_QFULL), 0u);
      if (*abort_flag) {
        for (int n = max(0, nk - C::NSK); n < nk; ++n)
          wait_bar_drain(bar(C::QB_KFULL + n % C::NSK), (uint32_t)((n / C::NSK) & 1));
        for (int n = max(0, nv - C::NSV); n < nv; ++n)
          wait_bar_drain(bar(C::QB_VFULL + n % C::NSV), (uint32_t)((n / C::NSV) & 1));
      }
    }
  } else {  // MMA issuers: two whole warps, one elected lane of each issues
    // =================================================================== MMA
    // Warp kWarpMma issues the products of the even key tiles (S slot 0),
    // warp kWarpMma + 1 those of the odd ones (S slot 1), so that one warp's
    // waits are covered by the other's products.  Each keeps S(n + 2) after
    // dQ~(n) on its own slot (issue order); the shared dP columns are handed
    // over by the threads (dP of tile n + 1 only after they have read tile
    // n's); the dQ~ accumulations run in tile order (each waits for the
    // previous one to complete, so the first initialises the accumulator and
    // the result does not depend on timing).
    const int hb = warp - kWarpMma;  // key tiles n with n % 2 == hb
    constexpr uint32_t ab = std::is_same<TIn, __nv_bfloat16>::value ? 1u : 0u;
    constexpr uint32_t IDESC_S = idesc_f16(0u, 0u, 128);   // fp16 Q~ x K~^T
    constexpr uint32_t IDESC_DP = idesc_f16(ab, 0u, 128);  // dO x V^T
    constexpr uint32_t IDESC_DQ = idesc_f16(0u, 1u, D);    // dS x K~ (K~ MN-major)
    constexpr uint32_t HI = sdesc_hi_sw128(1024);
    const uint32_t q_lo = sdesc_lo(sbase + C::Q_OFF_Q, 16);
    const uint32_t do_lo = sdesc_lo(sbase + C::Q_OFF_DO, 16);
    const uint32_t k_lo0 = sdesc_lo(sbase + C::Q_OFF_K, 16);
    const uint32_t v_lo0 = sdesc_lo(sbase + C::Q_OFF_V, 16);
    const uint32_t kmn_lo0 = sdesc_lo(sbase + C::Q_OFF_K, C::SUBT);
    const uint32_t s_col = tmem + (uint32_t)(128 * hb);  // this warp's S slot
    bool ok = wait_all(bar(C::QB_QFULL), 0u, ctl);
    for (int n = hb; ok && n < N; n += 2) {
      const int stk = n % C::NSK, stv = n % C::NSV;
      if (!wait_all(bar(C::QB_KFULL + stk), (uint32_t)((n / C::NSK) & 1), ctl)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sok = (uint32_t)(stk * C::TILE >> 4), sov = (uint32_t)(stv * C::TILE >> 4);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (uint32_t)(((kk >> 2) * C::SUBT + (kk & 3) * 32) >> 4);
        mma_ss_w(s_col, sdesc_join(q_lo + off, HI), sdesc_join(k_lo0 + sok + off, HI), IDESC_S,
                 kk > 0 ? 1u : 0u);
      }
      tc_commit_w(bar(C::QB_SFULL + hb));
      if (!wait_all(bar(C::QB_VFULL + stv), (uint32_t)((n / C::NSV) & 1), ctl) ||
          (n >= 1 && !wait_all(bar(C::QB_DPFREE), (uint32_t)((n - 1) & 1), ctl))) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (uint32_t)(((kk >> 2) * C::SUBT + (kk & 3) * 32) >> 4);
        mma_ss_w(tmem + 256u, sdesc_join(do_lo + off, HI), sdesc_join(v_lo0 + sov + off, HI),
                 IDESC_DP, kk > 0 ? 1u : 0u);
      }
      tc_commit_w(bar(C::QB_DPFULL));
      tc_commit_w(bar(C::QB_VEMPTY + stv));
      // dS of tile n in the slot, and the previous tile's dQ~ complete
      if (!wait_all(bar(C::QB_PFULL + hb), (uint32_t)((n >> 1) & 1), ctl) ||
          (n >= 1 && !wait_all(bar(C::QB_DQ), (uint32_t)((n - 1) & 1), ctl))) {
        ok = false;
        break;
      }
      tc_fence_after();
      // dQ~ += dS(n) K~(n), A = dS packed in the slot (keys 64..127 at +64)
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ts_w(tmem + 384u, s_col + (uint32_t)((kk >> 2) * 64 + (kk & 3) * 8),
                 sdesc_join(kmn_lo0 + sok + (uint32_t)(kk * 2048 >> 4), HI), IDESC_DQ,
                 (n > 0 || kk > 0) ? 1u : 0u);
      tc_commit_w(bar(C::QB_DQ));
      tc_commit_w(bar(C::QB_KEMPTY + stk));
      if (n == N - 1) tc_commit_w(bar(C::QB_ACC));
    }
    tc_commit_w(bar(C::QB_DONE));
    wait_bar_drain(bar(C::QB_DONE), 0u);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------- host
// A [B][H][S][D] tensor as a tensor map over (row, head, batch): box 64
// head-dim elements x 128 rows, 128-byte swizzle; rows past S read as zero.
cudaError_t make_rows_map(const void *base, int B, int H, int64_t S, int D, const int64_t st[3],
                          bool bf16, CUtensorMap *map, int perm[3]) {
  const int64_t size[3] = {S, H, B}, stride[3] = {st[2], st[1], st[0]};
  return make_row_tile_map(base, bf16, D, 3, size, stride, map, perm);
}

template <typename TIn>
cudaError_t rotate_f16(const void *x, int B, int H, int64_t S, int D, const int64_t st[3],
                       int64_t pos0, __half *out, const AttnArgs &f, cudaStream_t s) {
  const int64_t n = (int64_t)B * H * S * rotate_units(D, f.apply_rope, f.rot_dim, f.layout);
  if (n == 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = (int64_t)sm_count_current() * 16;
  if (blocks > cap) blocks = cap;
  bwd_rotate_f16_kernel<TIn><<<(unsigned)blocks, 256, 0, s>>>(
      static_cast<const TIn *>(x), H, S, D, st[0], st[1], st[2], pos0, out, f.apply_rope,
      f.rot_dim, f.layout, f.cos_t, f.sin_t, n, f.status);
  note_launch("bwd_rotate_f16_kernel");
  return cudaGetLastError();
}

template <int D, typename TIn>
cudaError_t launch_typed(const CUtensorMap (&maps)[4], const BwdTcParams &p, cudaStream_t s) {
  using C = BCfg<D>;
  static PerDeviceOnce once;
  const cudaError_t attr_err = once.run([] {
    cudaError_t e = cudaFuncSetAttribute(bwd_dkdv_tc_kernel<D, TIn>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::K_SMEM);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(bwd_dq_tc_kernel<D, TIn>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, C::Q_SMEM);
    return e;
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int64_t gk = (int64_t)p.n_kt * p.B * p.Hkv;
  const int64_t gq = (int64_t)p.n_qt * p.B * p.Hq;
  if (gk > 0x7fffffff || gq > 0x7fffffff) return cudaErrorInvalidConfiguration;
  bwd_dkdv_tc_kernel<D, TIn><<<(unsigned)gk, kThreadsK, C::K_SMEM, s>>>(maps[0], maps[1], maps[2],
                                                                       maps[3], p);
  note_launch("bwd_dkdv_tc_kernel");
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || gq == 0) return e;
  bwd_dq_tc_kernel<D, TIn><<<(unsigned)gq, kThreads, C::Q_SMEM, s>>>(maps[0], maps[1], maps[2],
                                                                     maps[3], p);
  note_launch("bwd_dq_tc_kernel");
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bwd_tc(const BwdArgs &a, cudaStream_t s) {
  const AttnArgs &f = a.f;
  if (f.D != 64 && f.D != 128) return cudaErrorNotSupported;
  const bool bf = f.dt == RA_BF16;
  // rotated fp16 copies of Q and K (contiguous [B][H][S][D]) in the workspace
  const int64_t cq[3] = {(int64_t)f.Hq * f.Sq * f.D, f.Sq * f.D, f.D};
  const int64_t ck[3] = {(int64_t)f.Hkv * f.Sk * f.D, f.Sk * f.D, f.D};
  cudaError_t e = bf ? rotate_f16<__nv_bfloat16>(f.q, f.B, f.Hq, f.Sq, f.D, f.sq, f.kv_offset,
                                                 static_cast<__half *>(a.qrot), f, s)
                     : rotate_f16<__half>(f.q, f.B, f.Hq, f.Sq, f.D, f.sq, f.kv_offset,
                                          static_cast<__half *>(a.qrot), f, s);
  if (e == cudaSuccess)
    e = bf ? rotate_f16<__nv_bfloat16>(f.k, f.B, f.Hkv, f.Sk, f.D, f.sk, 0,
                                       static_cast<__half *>(a.krot), f, s)
           : rotate_f16<__half>(f.k, f.B, f.Hkv, f.Sk, f.D, f.sk, 0,
                                static_cast<__half *>(a.krot), f, s);
  if (e != cudaSuccess) return e;

  BwdTcParams p{};
  CUtensorMap maps[4];  // q~, k~, v, dO
  e = make_rows_map(a.krot, f.B, f.Hkv, f.Sk, f.D, ck, false, &maps[1], p.kperm);
  if (e == cudaSuccess) e = make_rows_map(f.v, f.B, f.Hkv, f.Sk, f.D, f.sv, bf, &maps[2], p.vperm);
  if (e != cudaSuccess) return e;
  if (f.Sq > 0) {
    e = make_rows_map(a.qrot, f.B, f.Hq, f.Sq, f.D, cq, false, &maps[0], p.qperm);
    if (e == cudaSuccess)
      e = make_rows_map(a.dout, f.B, f.Hq, f.Sq, f.D, a.sdo, bf, &maps[3], p.operm);
    if (e != cudaSuccess) return e;
  } else {  // no query tiles: the maps are never read
    maps[0] = maps[1];
    maps[3] = maps[2];
    for (int i = 0; i < 3; ++i) {
      p.qperm[i] = p.kperm[i];
      p.operm[i] = p.vperm[i];
    }
  }
  p.lse = a.lse; p.dsum = a.dsum;
  p.dq = a.dq; p.dk = a.dk; p.dv = a.dv;
  p.sdq0 = a.sdq[0]; p.sdq1 = a.sdq[1]; p.sdq2 = a.sdq[2];
  p.sdk0 = a.sdk[0]; p.sdk1 = a.sdk[1]; p.sdk2 = a.sdk[2];
  p.sdv0 = a.sdv[0]; p.sdv1 = a.sdv[1]; p.sdv2 = a.sdv[2];
  p.Sq = f.Sq; p.Sk = f.Sk; p.off = f.kv_offset;
  p.B = f.B; p.Hq = f.Hq; p.Hkv = f.Hkv; p.G = f.Hq / f.Hkv;
  p.n_qt = (int)((f.Sq + 127) / 128);
  p.n_kt = (int)((f.Sk + 127) / 128);
  p.apply_rope = f.apply_rope; p.rot_dim = f.rot_dim; p.layout = f.layout;
  p.cos_t = f.cos_t; p.sin_t = f.sin_t;
  p.scale = f.scale;
  p.scale_log2 = (float)((double)f.scale * 1.4426950408889634);
  p.status = f.status;
  {
    // Past one wave of blocks, the dQ grid runs in bands of four kv heads'
    // q-heads, heaviest query tile first within a band, so that the K~/V of
    // the heads in flight stay in L2 (long-context GQA workload: dQ DRAM
    // 1.22 -> 0.50 GB per call, same time).  The dK/dV grid keeps one band:
    // its blocks' work is very uneven (the first key tiles see every query
    // tile, the last ones a few), and in bands the last band's heaviest
    // blocks start late (2-3 % slower at 2048-4096 queries).
    const int sms = sm_count_current();
    const int64_t gq = (int64_t)p.n_qt * p.B * p.Hq;
    p.kv_band = p.B * p.Hkv;
    p.q_band = gq > sms ? std::min(p.B * p.Hq, kBandKv * p.G) : p.B * p.Hq;
  }
  if (f.D == 64)
    return bf ? launch_typed<64, __nv_bfloat16>(maps, p, s) : launch_typed<64, __half>(maps, p, s);
  return bf ? launch_typed<128, __nv_bfloat16>(maps, p, s) : launch_typed<128, __half>(maps, p, s);
}

}  // namespace ra

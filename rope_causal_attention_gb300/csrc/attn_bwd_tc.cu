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
// GB300 design.  Two kernels, neither using atomics:
//   bwd_dkdv_tc_kernel: one CTA per (key tile of 128 rows, kv head, batch);
//     K~ and V stay in shared memory, and the CTA walks every (q-head of the
//     kv group, query tile) that sees its keys.  Per query tile:
//       S^T  = K~ Q~^T   (TMEM cols 256..383; M = 128 keys, N = 128 queries)
//       dP^T = V  dO^T   (TMEM cols 384..511)
//       threads: P^T (input dtype) over S^T, dS^T (fp16) over dP^T
//       dV  += P^T  dO   (TS: A = P^T in TMEM, B = dO read MN-major)
//       dK~ += dS^T Q~   (TS: A = dS^T in TMEM, B = Q~ read MN-major)
//     dV and dK~ accumulate in TMEM cols 0..2D-1 over the whole walk, so the
//     group's q-heads are summed inside the CTA.
//   bwd_dq_tc_kernel: one CTA per (query tile, q-head, batch); Q~ and dO stay
//     in shared memory, key tiles stream:
//       S = Q~ K~^T (cols 0..127),  dP = dO V^T (cols 128..255),
//       threads: dS (fp16) over S,  dQ~ += dS K~ (TS: B = K~ read MN-major,
//       TMEM cols 256..256+D-1).
//   The epilogues scale, rotate back with R^T (the table's sine negated) and
//   store in the input dtype.  A shared-memory tile written in the 128-byte
//   swizzled K-major layout doubles as the MN-major operand of the
//   transposed product, so Q~, dO and K~ are staged once.
// Roles (320 threads): warps 0-3 own TMEM lanes 0-127 (probabilities, dS,
// epilogue), warps 4-7 rotate Q/K rows into fp16 operand tiles, warp 8 issues
// TMA loads (V, dO), warp 9 allocates TMEM and issues the MMAs.  Every
// mbarrier wait is bounded (RA_ERR_DEVICE_TIMEOUT, abort flag, drain).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "rot_tile.cuh"
#include "tc_ptx.cuh"

namespace ra {
namespace {

using namespace ptx;
using rot::f16x2;
using rot::In16;

constexpr int kThreads = 320;
constexpr int kWarpRot = 4, kWarpTma = 8, kWarpMma = 9;
constexpr uint32_t kTmemCols = 512;
constexpr long long kTimeoutCycles = 1LL << 32;  // about two seconds
constexpr float kLog2e = 1.4426950408889634f;

template <int D> struct BCfg {
  static constexpr int TILE = 128 * D * 2;  // 128 rows of 16-bit values
  static constexpr int SUBT = 16384;        // one 64-column sub-tile
  static constexpr int NS = D == 128 ? 2 : 3;
  // dk/dv kernel: K~ | V | Q~ ring | dO ring | row stats ring (LSE log2, D)
  static constexpr int K_OFF_K = 0, K_OFF_V = TILE, K_OFF_Q = 2 * TILE;
  static constexpr int K_OFF_DO = K_OFF_Q + NS * TILE;
  static constexpr int K_OFF_ST = K_OFF_DO + NS * TILE;
  static constexpr int K_OFF_BAR = K_OFF_ST + NS * 1024;
  // barriers of the dk/dv kernel
  static constexpr int KB_KFULL = 0, KB_VFULL = 1, KB_QFULL = 2, KB_QEMPTY = 2 + NS,
                       KB_DOFULL = 2 + 2 * NS, KB_DOEMPTY = 2 + 3 * NS, KB_SFULL = 2 + 4 * NS,
                       KB_DPFULL = 3 + 4 * NS, KB_PFULL = 4 + 4 * NS, KB_ACC = 5 + 4 * NS,
                       KB_DONE = 6 + 4 * NS, KB_N = 7 + 4 * NS;
  static constexpr int K_OFF_MISC = K_OFF_BAR + KB_N * 8;
  static constexpr int K_SMEM = K_OFF_MISC + 16 + 1024;
  // dq kernel: Q~ | dO | K~ ring | V ring
  static constexpr int Q_OFF_Q = 0, Q_OFF_DO = TILE, Q_OFF_K = 2 * TILE;
  static constexpr int Q_OFF_V = Q_OFF_K + NS * TILE;
  static constexpr int Q_OFF_BAR = Q_OFF_V + NS * TILE;
  static constexpr int QB_QFULL = 0, QB_DOFULL = 1, QB_KFULL = 2, QB_KEMPTY = 2 + NS,
                       QB_VFULL = 2 + 2 * NS, QB_VEMPTY = 2 + 3 * NS, QB_SFULL = 2 + 4 * NS,
                       QB_DPFULL = 3 + 4 * NS, QB_PFULL = 4 + 4 * NS, QB_ACC = 5 + 4 * NS,
                       QB_DONE = 6 + 4 * NS, QB_N = 7 + 4 * NS;
  static constexpr int Q_OFF_MISC = Q_OFF_BAR + QB_N * 8;
  static constexpr int Q_SMEM = Q_OFF_MISC + 16 + 1024;
  static_assert(K_SMEM <= 232448 && Q_SMEM <= 232448, "shared memory");
  // the epilogue stages 128 padded fp32 rows over the rings
  static_assert(128 * (D + 1) * 4 <= 2 * NS * TILE, "epilogue scratch");
};

struct BwdTcParams {
  const void *q, *k;
  const float *lse, *dsum;
  void *dq, *dk, *dv;
  int64_t sq0, sq1, sq2, sk0, sk1, sk2;
  int64_t sdq0, sdq1, sdq2, sdk0, sdk1, sdk2, sdv0, sdv1, sdv2;
  int64_t Sq, Sk, off;
  int B, Hq, Hkv, G, n_qt, n_kt;
  int apply_rope, rot_dim, layout;
  const float *cos_t, *sin_t;
  int64_t table_rows;
  float scale, scale_log2;
  int vperm[3], operm[3];  // tensor-map dims 1..3 -> logical (0 row, 1 head, 2 batch)
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

__device__ __forceinline__ int map_coord(const int perm, int row, int head, int b) {
  return perm == 0 ? row : (perm == 1 ? head : b);
}

// One 128-row tile of rows (positions pos0 + r) rotated into a fp16 operand
// tile by the 128 rotation threads (thread t).
template <int D, typename TIn>
__device__ __forceinline__ void rotate_tile(const TIn *rows, int64_t stride, int64_t nvalid,
                                            int64_t pos0, uint8_t *tile, int t,
                                            const BwdTcParams &p) {
  if (p.apply_rope && p.rot_dim == D) {
    if (p.layout == RA_NEOX)
      rot::rotate_tile_full<D, TIn, RA_NEOX>(rows, stride, nvalid, pos0, tile, t, p);
    else
      rot::rotate_tile_full<D, TIn, RA_GPTJ>(rows, stride, nvalid, pos0, tile, t, p);
  } else {
    const bool valid = t < nvalid;
    rot::rotate_row<D, TIn>(rows + (valid ? t : 0) * stride, valid, pos0 + t, tile, t, p);
  }
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

// Stores a D-wide fp32 row (scratch, padded) as dtype, rotated back at pos
// when `rotate` (16-byte stores).
template <int D, typename TIn>
__device__ __forceinline__ void store_row(const float *row, bool rotate, int64_t pos, TIn *dst,
                                          const BwdTcParams &p) {
#pragma unroll 1
  for (int g = 0; g < D / 8; ++g) {
    float v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = rotate ? rot_back(row, 8 * g + e, pos, p) : row[8 * g + e];
    uint4 u;
    u.x = In16<TIn>::pack2(v[0], v[1]);
    u.y = In16<TIn>::pack2(v[2], v[3]);
    u.z = In16<TIn>::pack2(v[4], v[5]);
    u.w = In16<TIn>::pack2(v[6], v[7]);
    reinterpret_cast<uint4 *>(dst)[g] = u;
  }
}

// ===================================================================== dK, dV
template <int D, typename TIn>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tmap_v,
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

  // ---- work: key tile kt (low tiles, seen by the most queries, first)
  const int per_kt = p.B * p.Hkv;
  const int kt = blockIdx.x / per_kt;
  const int b = (blockIdx.x % per_kt) / p.Hkv, hk = blockIdx.x % p.Hkv;
  const int64_t j0 = (int64_t)kt * 128;
  const int64_t mf = j0 - p.off < 0 ? 0 : (j0 - p.off) / 128;  // first query tile that sees it
  const int m_first = (int)min(mf, (int64_t)p.n_qt);
  const int per_g = p.n_qt - m_first;
  const int NU = p.G * per_g;  // (q-head, query tile) units

  if (threadIdx.x == 0) {
    mbar_init(bar(C::KB_KFULL), 128);
    mbar_init(bar(C::KB_VFULL), 1);
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(bar(C::KB_QFULL + i), 128);
      mbar_init(bar(C::KB_QEMPTY + i), 1);
      mbar_init(bar(C::KB_DOFULL + i), 1);
      mbar_init(bar(C::KB_DOEMPTY + i), 1);
    }
    mbar_init(bar(C::KB_SFULL), 1);
    mbar_init(bar(C::KB_DPFULL), 1);
    mbar_init(bar(C::KB_PFULL), 128);
    mbar_init(bar(C::KB_ACC), 1);
    mbar_init(bar(C::KB_DONE), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kWarpTma && lane == 0) {
    prefetch_tmap(&tmap_v);
    prefetch_tmap(&tmap_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    // ========================================================= P^T and dS^T
    const int t = threadIdx.x;
    const uint32_t lanes = tmem + ((uint32_t)(warp * 32) << 16);
    const int64_t j = j0 + t;
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int u = 0; u < NU; ++u) {
      const int st = u % C::NS;
      const int m = m_first + u % per_g;
      ok = ok && __all_sync(0xffffffffu, wait_bar(bar(C::KB_QFULL + st), (uint32_t)((u / C::NS) & 1), ctl));
      ok = ok && __all_sync(0xffffffffu, wait_bar(bar(C::KB_SFULL), (uint32_t)(u & 1), ctl));
      ok = ok && __all_sync(0xffffffffu, wait_bar(bar(C::KB_DPFULL), (uint32_t)(u & 1), ctl));
      if (!ok) break;
      tc_fence_after();
      const float *lse2 = reinterpret_cast<const float *>(smem + C::K_OFF_ST + st * 1024);
      const float *dsm = lse2 + 128;
      const int64_t i0 = (int64_t)m * 128;
      const bool straddle = j0 + 127 > p.off + i0;
      const int64_t lim = j - p.off - i0;  // query column c sees key j iff c >= lim
#pragma unroll 1
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t sr[32], dr[32];
        tmem_ld32_pair(lanes + 256u + (uint32_t)c0, lanes + 384u + (uint32_t)c0, sr, dr);
        uint32_t pp[16], pd[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float p0 = ex2(fmaf(__uint_as_float(sr[e]), sl2, -lse2[c0 + e]));
          float p1 = ex2(fmaf(__uint_as_float(sr[e + 1]), sl2, -lse2[c0 + e + 1]));
          if (straddle) {
            if (c0 + e < lim) p0 = 0.f;
            if (c0 + e + 1 < lim) p1 = 0.f;
          }
          const float d0 = p0 * (__uint_as_float(dr[e]) - dsm[c0 + e]);
          const float d1 = p1 * (__uint_as_float(dr[e + 1]) - dsm[c0 + e + 1]);
          pp[e >> 1] = In16<TIn>::pack2(p0, p1);
          pd[e >> 1] = f16x2(d0, d1);
        }
        tmem_st16(lanes + 256u + (uint32_t)(c0 >> 1), pp);
        tmem_st16(lanes + 384u + (uint32_t)(c0 >> 1), pd);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::KB_PFULL));
    }
    // ---- epilogue: dV, dK = R(j)^T (scale dK~) for key row j
    const bool acc = ok && NU > 0 &&
                     __all_sync(0xffffffffu, wait_bar(bar(C::KB_ACC), 0u, ctl));
    if (!ok || (NU > 0 && !acc)) goto teardown_k;
    tc_fence_after();
    {
      float *row = reinterpret_cast<float *>(smem + C::K_OFF_Q) + t * (D + 1);
      TIn *dvd = static_cast<TIn *>(p.dv) + b * p.sdv0 + hk * p.sdv1 + j * p.sdv2;
      TIn *dkd = static_cast<TIn *>(p.dk) + b * p.sdk0 + hk * p.sdk1 + j * p.sdk2;
      const bool row_ok = j < p.Sk;
#pragma unroll 1
      for (int pass = 0; pass < 2; ++pass) {  // 0: dV (cols 0..D-1), 1: dK~ (cols D..2D-1)
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          if (acc) tmem_ld32(lanes + (uint32_t)(pass * D + 32 * c), r);
#pragma unroll
          for (int e = 0; e < 32; ++e)
            row[32 * c + e] = acc ? __uint_as_float(r[e]) * (pass ? p.scale : 1.f) : 0.f;
        }
        if (row_ok) store_row<D, TIn>(row, pass == 1, j, pass ? dkd : dvd, p);
      }
    }
  teardown_k:;
  } else if (warp < 8) {
    // ============================================================== rotation
    const int t = threadIdx.x - kWarpRot * 32;
    const TIn *kb = static_cast<const TIn *>(p.k) + b * p.sk0 + hk * p.sk1 + j0 * p.sk2;
    rotate_tile<D, TIn>(kb, p.sk2, p.Sk - j0, j0, smem + C::K_OFF_K, t, p);
    fence_proxy_async_smem();
    mbar_arrive(bar(C::KB_KFULL));
    for (int u = 0; u < NU; ++u) {
      const int st = u % C::NS;
      if (u >= C::NS &&
          !wait_bar(bar(C::KB_QEMPTY + st), (uint32_t)((u / C::NS - 1) & 1), ctl))
        break;
      const int g = u / per_g, m = m_first + u % per_g, h = hk * p.G + g;
      const int64_t i0 = (int64_t)m * 128;
      const TIn *qb = static_cast<const TIn *>(p.q) + b * p.sq0 + h * p.sq1 + i0 * p.sq2;
      rotate_tile<D, TIn>(qb, p.sq2, p.Sq - i0, p.off + i0, smem + C::K_OFF_Q + st * C::TILE, t, p);
      float *stats = reinterpret_cast<float *>(smem + C::K_OFF_ST + st * 1024);
      const int64_t i = i0 + t;
      const int64_t r = ((int64_t)b * p.Hq + h) * p.Sq + i;
      stats[t] = i < p.Sq ? p.lse[r] * kLog2e : INFINITY;  // rows past Sq: P = 0
      stats[128 + t] = i < p.Sq ? p.dsum[r] : 0.f;
      fence_proxy_async_smem();
      mbar_arrive(bar(C::KB_QFULL + st));
    }
  } else if (warp == kWarpTma) {
    // =================================================================== TMA
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(C::KB_VFULL), (uint32_t)C::TILE);
#pragma unroll
      for (int sub = 0; sub < D / 64; ++sub)
        tma_load_4d(sbase + C::K_OFF_V + sub * C::SUBT, &tmap_v, bar(C::KB_VFULL), sub * 64,
                    map_coord(p.vperm[0], (int)j0, hk, b), map_coord(p.vperm[1], (int)j0, hk, b),
                    map_coord(p.vperm[2], (int)j0, hk, b));
      int issued = 0;
      for (int u = 0; u < NU; ++u) {
        const int st = u % C::NS;
        if (u >= C::NS &&
            !wait_bar(bar(C::KB_DOEMPTY + st), (uint32_t)((u / C::NS - 1) & 1), ctl))
          break;
        const int g = u / per_g, m = m_first + u % per_g, h = hk * p.G + g;
        const int row = m * 128;
        mbar_arrive_expect_tx(bar(C::KB_DOFULL + st), (uint32_t)C::TILE);
#pragma unroll
        for (int sub = 0; sub < D / 64; ++sub)
          tma_load_4d(sbase + C::K_OFF_DO + st * C::TILE + sub * C::SUBT, &tmap_do,
                      bar(C::KB_DOFULL + st), sub * 64, map_coord(p.operm[0], row, h, b),
                      map_coord(p.operm[1], row, h, b), map_coord(p.operm[2], row, h, b));
        issued = u + 1;
      }
      // copies in flight land before the block exits
      wait_bar_drain(bar(C::KB_VFULL), 0u);
      if (*abort_flag)
        for (int u = max(0, issued - C::NS); u < issued; ++u)
          wait_bar_drain(bar(C::KB_DOFULL + u % C::NS), (uint32_t)((u / C::NS) & 1));
    }
  } else {
    // =================================================================== MMA
    if (lane == 0) {
      constexpr uint32_t ab = std::is_same<TIn, __nv_bfloat16>::value ? 1u : 0u;
      constexpr uint32_t IDESC_S = idesc_f16(0u, 0u, 128);   // fp16 K~ x Q~^T
      constexpr uint32_t IDESC_DP = idesc_f16(ab, 0u, 128);  // V x dO^T
      constexpr uint32_t IDESC_DV = idesc_f16(ab, 1u, D);    // P^T x dO (dO MN-major)
      constexpr uint32_t IDESC_DK = idesc_f16(0u, 1u, D);    // dS^T x Q~ (Q~ MN-major)
      constexpr uint32_t HI = sdesc_hi_sw128(1024);
      const uint32_t k_lo = sdesc_lo(sbase + C::K_OFF_K, 16);
      const uint32_t v_lo = sdesc_lo(sbase + C::K_OFF_V, 16);
      const uint32_t q_lo0 = sdesc_lo(sbase + C::K_OFF_Q, 16);
      const uint32_t do_lo0 = sdesc_lo(sbase + C::K_OFF_DO, 16);
      const uint32_t qmn_lo0 = sdesc_lo(sbase + C::K_OFF_Q, C::SUBT);
      const uint32_t domn_lo0 = sdesc_lo(sbase + C::K_OFF_DO, C::SUBT);
      bool ok = NU == 0 || (wait_bar(bar(C::KB_KFULL), 0u, ctl) && wait_bar(bar(C::KB_VFULL), 0u, ctl));
      for (int u = 0; ok && u < NU; ++u) {
        const int st = u % C::NS;
        if (!wait_bar(bar(C::KB_QFULL + st), (uint32_t)((u / C::NS) & 1), ctl) ||
            !wait_bar(bar(C::KB_DOFULL + st), (uint32_t)((u / C::NS) & 1), ctl)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t so = (uint32_t)(st * C::TILE >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (uint32_t)(((kk >> 2) * C::SUBT + (kk & 3) * 32) >> 4);
          mma_ss(tmem + 256u, sdesc_join(k_lo + off, HI), sdesc_join(q_lo0 + so + off, HI),
                 IDESC_S, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar(C::KB_SFULL));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (uint32_t)(((kk >> 2) * C::SUBT + (kk & 3) * 32) >> 4);
          mma_ss(tmem + 384u, sdesc_join(v_lo + off, HI), sdesc_join(do_lo0 + so + off, HI),
                 IDESC_DP, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar(C::KB_DPFULL));
        if (!wait_bar(bar(C::KB_PFULL), (uint32_t)(u & 1), ctl)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // 16 queries per step
          mma_ts(tmem, tmem + 256u + (uint32_t)(kk * 8),
                 sdesc_join(domn_lo0 + so + (uint32_t)(kk * 2048 >> 4), HI), IDESC_DV,
                 (u > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + (uint32_t)D, tmem + 384u + (uint32_t)(kk * 8),
                 sdesc_join(qmn_lo0 + so + (uint32_t)(kk * 2048 >> 4), HI), IDESC_DK,
                 (u > 0 || kk > 0) ? 1u : 0u);
        tc_commit(bar(C::KB_QEMPTY + st));
        tc_commit(bar(C::KB_DOEMPTY + st));
      }
      if (ok && NU > 0) tc_commit(bar(C::KB_ACC));
      tc_commit(bar(C::KB_DONE));
      wait_bar_drain(bar(C::KB_DONE), 0u);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, kTmemCols);
}

// ========================================================================= dQ
template <int D, typename TIn>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tmap_v,
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

  // ---- work: query tile m (last tiles, which see the most keys, first)
  const int per_m = p.B * p.Hq;
  const int m = p.n_qt - 1 - (int)(blockIdx.x / per_m);
  const int b = (blockIdx.x % per_m) / p.Hq, h = blockIdx.x % p.Hq;
  const int hk = h / p.G;
  const int64_t i0 = (int64_t)m * 128;
  const int64_t last_pos = p.off + min(i0 + 127, p.Sq - 1);
  const int N = (int)min((int64_t)p.n_kt, last_pos / 128 + 1);  // key tiles seen (>= 1)

  if (threadIdx.x == 0) {
    mbar_init(bar(C::QB_QFULL), 128);
    mbar_init(bar(C::QB_DOFULL), 1);
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(bar(C::QB_KFULL + i), 128);
      mbar_init(bar(C::QB_KEMPTY + i), 1);
      mbar_init(bar(C::QB_VFULL + i), 1);
      mbar_init(bar(C::QB_VEMPTY + i), 1);
    }
    mbar_init(bar(C::QB_SFULL), 1);
    mbar_init(bar(C::QB_DPFULL), 1);
    mbar_init(bar(C::QB_PFULL), 128);
    mbar_init(bar(C::QB_ACC), 1);
    mbar_init(bar(C::QB_DONE), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kWarpTma && lane == 0) {
    prefetch_tmap(&tmap_v);
    prefetch_tmap(&tmap_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    // ================================================================== dS
    const int t = threadIdx.x;
    const uint32_t lanes = tmem + ((uint32_t)(warp * 32) << 16);
    const int64_t i = i0 + t;
    const bool row_ok = i < p.Sq;
    const int64_t r = ((int64_t)b * p.Hq + h) * p.Sq + i;
    const float lse2 = row_ok ? p.lse[r] * kLog2e : INFINITY;  // rows past Sq: P = 0
    const float dsum = row_ok ? p.dsum[r] : 0.f;
    const float sl2 = p.scale_log2;
    const int64_t qpos = p.off + i;
    bool ok = true;
    for (int n = 0; n < N; ++n) {
      ok = ok && __all_sync(0xffffffffu, wait_bar(bar(C::QB_SFULL), (uint32_t)(n & 1), ctl));
      ok = ok && __all_sync(0xffffffffu, wait_bar(bar(C::QB_DPFULL), (uint32_t)(n & 1), ctl));
      if (!ok) break;
      tc_fence_after();
      const int64_t jt = (int64_t)n * 128;
      const bool straddle = (jt + 127 > p.off + i0) || (jt + 127 >= p.Sk);
      // key column c is admissible iff c <= lim
      const int64_t lim = min(qpos, p.Sk - 1) - jt;
#pragma unroll 1
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t sr[32], dr[32];
        tmem_ld32_pair(lanes + (uint32_t)c0, lanes + 128u + (uint32_t)c0, sr, dr);
        uint32_t pd[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float p0 = ex2(fmaf(__uint_as_float(sr[e]), sl2, -lse2));
          float p1 = ex2(fmaf(__uint_as_float(sr[e + 1]), sl2, -lse2));
          if (straddle) {
            if (c0 + e > lim) p0 = 0.f;
            if (c0 + e + 1 > lim) p1 = 0.f;
          }
          pd[e >> 1] = f16x2(p0 * (__uint_as_float(dr[e]) - dsum),
                             p1 * (__uint_as_float(dr[e + 1]) - dsum));
        }
        tmem_st16(lanes + (uint32_t)(c0 >> 1), pd);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::QB_PFULL));
    }
    // ---- epilogue: dq = R(kv_offset + i)^T (scale dQ~)
    const bool acc = ok && __all_sync(0xffffffffu, wait_bar(bar(C::QB_ACC), 0u, ctl));
    if (acc) {
      tc_fence_after();
      float *row = reinterpret_cast<float *>(smem + C::Q_OFF_K) + t * (D + 1);
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(lanes + 256u + (uint32_t)(32 * c), rr);
#pragma unroll
        for (int e = 0; e < 32; ++e) row[32 * c + e] = __uint_as_float(rr[e]) * p.scale;
      }
      if (row_ok)
        store_row<D, TIn>(row, true, qpos,
                          static_cast<TIn *>(p.dq) + b * p.sdq0 + h * p.sdq1 + i * p.sdq2, p);
    }
  } else if (warp < 8) {
    // ============================================================== rotation
    const int t = threadIdx.x - kWarpRot * 32;
    const TIn *qb = static_cast<const TIn *>(p.q) + b * p.sq0 + h * p.sq1 + i0 * p.sq2;
    rotate_tile<D, TIn>(qb, p.sq2, p.Sq - i0, p.off + i0, smem + C::Q_OFF_Q, t, p);
    fence_proxy_async_smem();
    mbar_arrive(bar(C::QB_QFULL));
    const TIn *kb = static_cast<const TIn *>(p.k) + b * p.sk0 + hk * p.sk1;
    for (int n = 0; n < N; ++n) {
      const int st = n % C::NS;
      if (n >= C::NS &&
          !wait_bar(bar(C::QB_KEMPTY + st), (uint32_t)((n / C::NS - 1) & 1), ctl))
        break;
      const int64_t jt = (int64_t)n * 128;
      rotate_tile<D, TIn>(kb + jt * p.sk2, p.sk2, p.Sk - jt, jt, smem + C::Q_OFF_K + st * C::TILE,
                          t, p);
      fence_proxy_async_smem();
      mbar_arrive(bar(C::QB_KFULL + st));
    }
  } else if (warp == kWarpTma) {
    // =================================================================== TMA
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(C::QB_DOFULL), (uint32_t)C::TILE);
#pragma unroll
      for (int sub = 0; sub < D / 64; ++sub)
        tma_load_4d(sbase + C::Q_OFF_DO + sub * C::SUBT, &tmap_do, bar(C::QB_DOFULL), sub * 64,
                    map_coord(p.operm[0], (int)i0, h, b), map_coord(p.operm[1], (int)i0, h, b),
                    map_coord(p.operm[2], (int)i0, h, b));
      int issued = 0;
      for (int n = 0; n < N; ++n) {
        const int st = n % C::NS;
        if (n >= C::NS &&
            !wait_bar(bar(C::QB_VEMPTY + st), (uint32_t)((n / C::NS - 1) & 1), ctl))
          break;
        const int row = n * 128;
        mbar_arrive_expect_tx(bar(C::QB_VFULL + st), (uint32_t)C::TILE);
#pragma unroll
        for (int sub = 0; sub < D / 64; ++sub)
          tma_load_4d(sbase + C::Q_OFF_V + st * C::TILE + sub * C::SUBT, &tmap_v,
                      bar(C::QB_VFULL + st), sub * 64, map_coord(p.vperm[0], row, hk, b),
                      map_coord(p.vperm[1], row, hk, b), map_coord(p.vperm[2], row, hk, b));
        issued = n + 1;
      }
      wait_bar_drain(bar(C::QB_DOFULL), 0u);
      if (*abort_flag)
        for (int n = max(0, issued - C::NS); n < issued; ++n)
          wait_bar_drain(bar(C::QB_VFULL + n % C::NS), (uint32_t)((n / C::NS) & 1));
    }
  } else {
    // =================================================================== MMA
    if (lane == 0) {
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
      bool ok = wait_bar(bar(C::QB_QFULL), 0u, ctl) && wait_bar(bar(C::QB_DOFULL), 0u, ctl);
      for (int n = 0; ok && n < N; ++n) {
        const int st = n % C::NS;
        if (!wait_bar(bar(C::QB_KFULL + st), (uint32_t)((n / C::NS) & 1), ctl) ||
            !wait_bar(bar(C::QB_VFULL + st), (uint32_t)((n / C::NS) & 1), ctl)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t so = (uint32_t)(st * C::TILE >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (uint32_t)(((kk >> 2) * C::SUBT + (kk & 3) * 32) >> 4);
          mma_ss(tmem, sdesc_join(q_lo + off, HI), sdesc_join(k_lo0 + so + off, HI), IDESC_S,
                 kk > 0 ? 1u : 0u);
        }
        tc_commit(bar(C::QB_SFULL));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (uint32_t)(((kk >> 2) * C::SUBT + (kk & 3) * 32) >> 4);
          mma_ss(tmem + 128u, sdesc_join(do_lo + off, HI), sdesc_join(v_lo0 + so + off, HI),
                 IDESC_DP, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar(C::QB_DPFULL));
        if (!wait_bar(bar(C::QB_PFULL), (uint32_t)(n & 1), ctl)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // 16 keys per step
          mma_ts(tmem + 256u, tmem + (uint32_t)(kk * 8),
                 sdesc_join(kmn_lo0 + so + (uint32_t)(kk * 2048 >> 4), HI), IDESC_DQ,
                 (n > 0 || kk > 0) ? 1u : 0u);
        tc_commit(bar(C::QB_KEMPTY + st));
        tc_commit(bar(C::QB_VEMPTY + st));
      }
      if (ok) tc_commit(bar(C::QB_ACC));
      tc_commit(bar(C::QB_DONE));
      wait_bar_drain(bar(C::QB_DONE), 0u);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------- host
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

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

// A [B][H][S][D] tensor as a 4-D tensor map: dim 0 = head dim (contiguous),
// dims 1..3 = row, head and batch ordered by increasing stride (size-1 dims
// last); box 64 head-dim elements x 128 rows, 128-byte swizzle; rows past S
// read as zero.
cudaError_t make_rows_map(const void *base, int B, int H, int64_t S, int D, const int64_t st[3],
                          ra_dtype dt, CUtensorMap *map, int perm[3]) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  struct Dim { uint64_t size, stride; int logical; };
  Dim d[3] = {{(uint64_t)S, (uint64_t)st[2] * 2, 0},
              {(uint64_t)H, (uint64_t)st[1] * 2, 1},
              {(uint64_t)B, (uint64_t)st[0] * 2, 2}};
  std::stable_sort(d, d + 3, [](const Dim &x, const Dim &y) {
    if ((x.size == 1) != (y.size == 1)) return y.size == 1;
    return x.stride < y.stride;
  });
  uint64_t prev_extent = (uint64_t)D * 2;
  for (int i = 0; i < 3; ++i) {
    if (d[i].size == 1 || d[i].stride == 0) d[i].stride = (prev_extent + 15) & ~uint64_t(15);
    prev_extent = d[i].stride * d[i].size;
    perm[i] = d[i].logical;
  }
  const cuuint64_t gdim[4] = {(cuuint64_t)D, d[0].size, d[1].size, d[2].size};
  const cuuint64_t gstride[3] = {d[0].stride, d[1].stride, d[2].stride};
  cuuint32_t box[4] = {64, 1, 1, 1};
  for (int i = 0; i < 3; ++i)
    if (d[i].logical == 0) box[1 + i] = 128;
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType t =
      dt == RA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUresult r = enc(map, t, 4, const_cast<void *>(base), gdim, gstride, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D, typename TIn>
cudaError_t launch_typed(const CUtensorMap &mv, const CUtensorMap &mdo, const BwdTcParams &p,
                         cudaStream_t s) {
  using C = BCfg<D>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(bwd_dkdv_tc_kernel<D, TIn>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, C::K_SMEM);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(bwd_dq_tc_kernel<D, TIn>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, C::Q_SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int64_t gk = (int64_t)p.n_kt * p.B * p.Hkv;
  const int64_t gq = (int64_t)p.n_qt * p.B * p.Hq;
  if (gk > 0x7fffffff || gq > 0x7fffffff) return cudaErrorInvalidConfiguration;
  bwd_dkdv_tc_kernel<D, TIn><<<(unsigned)gk, kThreads, C::K_SMEM, s>>>(mv, mdo, p);
  note_launch("bwd_dkdv_tc_kernel");
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || gq == 0) return e;
  bwd_dq_tc_kernel<D, TIn><<<(unsigned)gq, kThreads, C::Q_SMEM, s>>>(mv, mdo, p);
  note_launch("bwd_dq_tc_kernel");
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bwd_tc(const BwdArgs &a, cudaStream_t s) {
  const AttnArgs &f = a.f;
  if (f.D != 64 && f.D != 128) return cudaErrorNotSupported;
  BwdTcParams p{};
  CUtensorMap mv, mdo;
  cudaError_t e = make_rows_map(f.v, f.B, f.Hkv, f.Sk, f.D, f.sv, f.dt, &mv, p.vperm);
  if (e != cudaSuccess) return e;
  if (f.Sq > 0) {
    e = make_rows_map(a.dout, f.B, f.Hq, f.Sq, f.D, a.sdo, f.dt, &mdo, p.operm);
    if (e != cudaSuccess) return e;
  } else {
    mdo = mv;  // never read: no query tiles
    p.operm[0] = p.vperm[0]; p.operm[1] = p.vperm[1]; p.operm[2] = p.vperm[2];
  }
  p.q = f.q; p.k = f.k; p.lse = a.lse; p.dsum = a.dsum;
  p.dq = a.dq; p.dk = a.dk; p.dv = a.dv;
  p.sq0 = f.sq[0]; p.sq1 = f.sq[1]; p.sq2 = f.sq[2];
  p.sk0 = f.sk[0]; p.sk1 = f.sk[1]; p.sk2 = f.sk[2];
  p.sdq0 = a.sdq[0]; p.sdq1 = a.sdq[1]; p.sdq2 = a.sdq[2];
  p.sdk0 = a.sdk[0]; p.sdk1 = a.sdk[1]; p.sdk2 = a.sdk[2];
  p.sdv0 = a.sdv[0]; p.sdv1 = a.sdv[1]; p.sdv2 = a.sdv[2];
  p.Sq = f.Sq; p.Sk = f.Sk; p.off = f.kv_offset;
  p.B = f.B; p.Hq = f.Hq; p.Hkv = f.Hkv; p.G = f.Hq / f.Hkv;
  p.n_qt = (int)((f.Sq + 127) / 128);
  p.n_kt = (int)((f.Sk + 127) / 128);
  p.apply_rope = f.apply_rope; p.rot_dim = f.rot_dim; p.layout = f.layout;
  p.cos_t = f.cos_t; p.sin_t = f.sin_t; p.table_rows = f.table_rows;
  p.scale = f.scale;
  p.scale_log2 = (float)((double)f.scale * 1.4426950408889634);
  p.status = f.status;
  const bool bf = f.dt == RA_BF16;
  if (f.D == 64)
    return bf ? launch_typed<64, __nv_bfloat16>(mv, mdo, p, s) : launch_typed<64, __half>(mv, mdo, p, s);
  return bf ? launch_typed<128, __nv_bfloat16>(mv, mdo, p, s) : launch_typed<128, __half>(mv, mdo, p, s);
}

}  // namespace ra

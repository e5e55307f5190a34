// Causal attention forward with RoPE fused in, on the sm_103a tensor cores
// (tcgen05 + tensor memory), for bf16/fp16 inputs and head dims 64 and 128.
//
// Mathematics ("RoPE and FlashAttention: relative positions and online
// softmax", sections 1, 2, 4 and 5; "RoPE + PoPE Attention Kernels", which
// moves the rotation inside the attention kernel):
//   q~_i = R(kv_offset + i) q_i,  k~_j = R(j) k_j,  V never rotated;
//   s_ij = scale * <q~_i, k~_j> for j <= kv_offset + i, j < Sk;
//   online softmax per row: running max m, denominator l, numerator u;
//   O_i = u_i / l_i,  LSE_i = m_i + ln l_i.
//
// GB300 design
// ------------
// One CTA owns two 128-row query "slots" that share every K/V tile: two
// q-heads of one kv group at the same rows (grouped-query attention), or two
// consecutive 128-row tiles of one head.  Warp roles (448 threads):
//   warps 0-3   softmax for slot 0 (thread = query row = TMEM lane)
//   warps 4-7   softmax for slot 1
//   warps 8-11  rotation: Q tiles once, then each K tile as it is staged:
//               global bf16/fp16 -> fp32 rotation with the fp32 cos/sin table
//               -> fp16 operand in 128B-swizzled shared memory
//   warp 12     TMA producer for V tiles (raw, never rotated)
//   warp 13     tcgen05 MMA issuer; owns the tensor-memory allocation
// Tensor memory (512 columns): S0 | S1 | O0 | O1.  P is written as 16-bit
// pairs over the first 64 columns of its S block and fed to the PV product
// straight from tensor memory.  The issue order S0(n+1) after PV0(n) and
// S1(n+1) after PV1(n) lets one slot's softmax run while the tensor core
// works on the other slot.  K tiles fully in the future of every row of a
// slot are never visited (causal tile skipping); the mask is evaluated only
// on tiles that straddle the diagonal or the end of K.  No rotated tensor
// ever reaches global memory.
//
// Every mbarrier wait is bounded: on expiry the kernel records
// RA_ERR_DEVICE_TIMEOUT, raises a block-wide abort flag, drains the copies
// and MMAs it has in flight, frees tensor memory and returns.
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
#include "tc_ptx.cuh"

namespace ra {
namespace {

using namespace ptx;

constexpr int kThreads = 448;
constexpr int kWarpRot = 8;
constexpr int kWarpTma = 12;
constexpr int kWarpMma = 13;
constexpr uint32_t kTmemCols = 512;
constexpr long long kTimeoutCycles = 1LL << 32;  // about two seconds

template <int D>
struct TcCfg {
  static constexpr int NS = (D == 128) ? 2 : 3;  // K~ and V pipeline stages
  static constexpr int TILE = 128 * D * 2;       // one 128-row tile of 16-bit values
  static constexpr int SUBT = 128 * 128;         // one 64-column (128-byte-row) sub-tile
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = 2 * TILE;
  static constexpr int OFF_V = OFF_K + NS * TILE;
  static constexpr int OFF_BAR = OFF_V + NS * TILE;
  static constexpr int B_QFULL = 0;
  static constexpr int B_KFULL = 2;
  static constexpr int B_KEMPTY = 2 + NS;
  static constexpr int B_VFULL = 2 + 2 * NS;
  static constexpr int B_VEMPTY = 2 + 3 * NS;
  static constexpr int B_SFULL = 2 + 4 * NS;
  static constexpr int B_PFULL = 4 + 4 * NS;
  static constexpr int B_OFULL = 6 + 4 * NS;
  static constexpr int B_DONE = 8 + 4 * NS;
  static constexpr int NBAR = 9 + 4 * NS;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;  // slack to align the base to 1024
  // tensor-memory columns: S0 | S1 | O0 | O1
  static __device__ __forceinline__ uint32_t s_col(int slot) { return slot ? 128u : 0u; }
  static __device__ __forceinline__ uint32_t o_col(int slot) { return 256u + (slot ? D : 0); }
};

struct TcParams {
  const void *q, *k;
  void *o;
  float *lse;
  int64_t sq0, sq1, sq2, sk0, sk1, sk2, so0, so1, so2;
  int64_t Sq, Sk, kv_off;
  int Hq, G, n_units, units_per_b, n_qt, pack_heads;
  int apply_rope, rot_dim, layout;
  const float *cos_t, *sin_t;
  float scale_log2;
  int vperm[3];  // tensor-map dims 1..3 -> logical coordinate (0 key row, 1 kv head, 2 batch)
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

// Wait used while draining after an abort: ignores the abort flag, still bounded.
__device__ __forceinline__ void wait_bar_drain(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > kTimeoutCycles) return;
}

template <typename T> struct In16;
template <> struct In16<__nv_bfloat16> {
  static __device__ __forceinline__ void unpack(const uint4 &u, float *f) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t = __bfloat1622float2(h[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
  static __device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
  }
};
template <> struct In16<__half> {
  static __device__ __forceinline__ void unpack(const uint4 &u, float *f) {
    const __half2 *h = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t = __half22float2(h[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
  static __device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
  }
};

__device__ __forceinline__ uint32_t f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&h);
}

// Stores 8 values as fp16 into 16-byte chunk c of row `row` of a 128-row tile
// laid out as 64-column sub-tiles with the 128-byte swizzle (chunk index XOR
// row mod 8), the layout the tcgen05 K-major descriptor expects.
__device__ __forceinline__ void st_chunk(uint8_t *tile, int row, int c, const float *f) {
  const int sub = c >> 3, cc = c & 7;
  uint4 u;
  u.x = f16x2(f[0], f[1]);
  u.y = f16x2(f[2], f[3]);
  u.z = f16x2(f[4], f[5]);
  u.w = f16x2(f[6], f[7]);
  *reinterpret_cast<uint4 *>(tile + sub * 16384 + row * 128 + ((cc ^ (row & 7)) << 4)) = u;
}

__device__ __forceinline__ void ld_table4(const float *p, float *f) {
  const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
}

// Rotates one D-wide row (position pos) into fp16 row `row` of a swizzled
// operand tile.  Rows outside the tensor (valid == false) become zeros.
// NeoX pairs (i, i + r/2), GPT-J pairs (2i, 2i+1); dims past rot_dim copied.
template <int D, typename TIn>
__device__ __forceinline__ void rotate_row(const TIn *src, bool valid, int64_t pos, uint8_t *tile,
                                           int row, const TcParams &p) {
  constexpr int NC = D / 8;
  if (!valid) {
    const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < NC; ++c) st_chunk(tile, row, c, z);
    return;
  }
  const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
  int done = 0;  // chunks written by the rotation
  if (p.apply_rope) {
    const int half = p.rot_dim >> 1;
    const float *cr = p.cos_t + pos * half;
    const float *sr = p.sin_t + pos * half;
    if (p.layout == RA_NEOX) {
      const int hc = half >> 3;  // chunks per half
#pragma unroll 2
      for (int c = 0; c < hc; ++c) {
        float lo[8], hi[8], cs[8], sn[8], a[8], b[8];
        In16<TIn>::unpack(__ldg(s4 + c), lo);
        In16<TIn>::unpack(__ldg(s4 + c + hc), hi);
        ld_table4(cr + 8 * c, cs);
        ld_table4(cr + 8 * c + 4, cs + 4);
        ld_table4(sr + 8 * c, sn);
        ld_table4(sr + 8 * c + 4, sn + 4);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          a[e] = lo[e] * cs[e] - hi[e] * sn[e];
          b[e] = hi[e] * cs[e] + lo[e] * sn[e];
        }
        st_chunk(tile, row, c, a);
        st_chunk(tile, row, c + hc, b);
      }
    } else {
      const int rc = p.rot_dim >> 3;  // chunks of 4 pairs
#pragma unroll 2
      for (int c = 0; c < rc; ++c) {
        float x[8], cs[4], sn[4], y[8];
        In16<TIn>::unpack(__ldg(s4 + c), x);
        ld_table4(cr + 4 * c, cs);
        ld_table4(sr + 4 * c, sn);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          y[2 * e] = x[2 * e] * cs[e] - x[2 * e + 1] * sn[e];
          y[2 * e + 1] = x[2 * e + 1] * cs[e] + x[2 * e] * sn[e];
        }
        st_chunk(tile, row, c, y);
      }
    }
    done = p.rot_dim >> 3;
  }
  for (int c = done; c < NC; ++c) {
    float x[8];
    In16<TIn>::unpack(__ldg(s4 + c), x);
    st_chunk(tile, row, c, x);
  }
}

template <int D, typename TIn>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmap_v, const TcParams p) {
  using C = TcCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
  const Ctl ctl{abort_flag, p.status};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work item: (batch, head unit, query tile), heaviest (last) tiles first
  const int bid = blockIdx.x;
  const int qt = p.n_qt - 1 - bid / p.n_units;
  const int unit = bid % p.n_units;
  const int b = unit / p.units_per_b, hu = unit % p.units_per_b;
  int h[2];
  int64_t m0[2];
  if (p.pack_heads) {
    h[0] = 2 * hu;
    h[1] = 2 * hu + 1;
    m0[0] = m0[1] = (int64_t)qt * 128;
  } else {
    h[0] = h[1] = hu;
    m0[0] = (int64_t)qt * 256;
    m0[1] = m0[0] + 128;
  }
  const int hk = h[0] / p.G;
  const int nkt = (int)((p.Sk + 127) / 128);
  bool act[2];
  int nend[2];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    act[s] = m0[s] < p.Sq;
    const int64_t last = min(m0[s] + 127, p.Sq - 1);
    nend[s] = act[s] ? (int)min((int64_t)nkt, (last + p.kv_off) / 128 + 1) : 0;
  }
  const int N = max(nend[0], nend[1]);

  // ---- set-up: barriers, tensor memory
  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_QFULL + 0), 128);
    mbar_init(bar(C::B_QFULL + 1), 128);
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(bar(C::B_KFULL + i), 128);
      mbar_init(bar(C::B_KEMPTY + i), 1);
      mbar_init(bar(C::B_VFULL + i), 1);
      mbar_init(bar(C::B_VEMPTY + i), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::B_SFULL + s), 1);
      mbar_init(bar(C::B_PFULL + s), 128);
      mbar_init(bar(C::B_OFULL + s), 1);
    }
    mbar_init(bar(C::B_DONE), 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kWarpTma && lane == 0) prefetch_tmap(&tmap_v);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 8) {
    // ================================================================ softmax
    const int slot = warp >> 2;
    const int wq = warp & 3;
    const int t = wq * 32 + lane;
    const uint32_t lane_bits = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_bits + C::s_col(slot);
    const uint32_t tO = tmem + lane_bits + C::o_col(slot);
    if (act[slot]) {
      const int64_t i = m0[slot] + t;
      const int64_t qpos = p.kv_off + i;
      const float sl2 = p.scale_log2;
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int n = 0; n < nend[slot]; ++n) {
        if (!wait_bar(bar(C::B_SFULL + slot), (uint32_t)(n & 1), ctl)) { ok = false; break; }
        tc_fence_after();
        const int64_t j0 = (int64_t)n * 128;
        const bool need_mask = (j0 + 127 > m0[slot] + p.kv_off) || (j0 + 127 >= p.Sk);
        const int64_t jlim = min(qpos, p.Sk - 1);  // last admissible key of this row
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld32(tS + 32 * c, r);
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            float x = __uint_as_float(r[e]);
            if (need_mask && j0 + 32 * c + e > jlim) x = -INFINITY;
            mx = fmaxf(mx, x);
          }
        }
        const float m_new = fmaxf(m, mx * sl2);
        const float alpha = ex2(m - m_new);
        float rs = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32], pk[16];
          tmem_ld32(tS + 32 * c, r);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float x0 = __uint_as_float(r[e]), x1 = __uint_as_float(r[e + 1]);
            if (need_mask) {
              if (j0 + 32 * c + e > jlim) x0 = -INFINITY;
              if (j0 + 32 * c + e + 1 > jlim) x1 = -INFINITY;
            }
            const float p0 = ex2(fmaf(x0, sl2, -m_new));
            const float p1 = ex2(fmaf(x1, sl2, -m_new));
            rs += p0 + p1;
            pk[e >> 1] = In16<TIn>::pack2(p0, p1);
          }
          tmem_st16(tS + 16 * c, pk);  // P over the first 64 columns of S
        }
        tmem_st_wait();
        l = l * alpha + rs;
        if (n > 0 && __any_sync(0xffffffffu, alpha < 1.f)) {
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(tO + 32 * c, r);
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
            tmem_st32(tO + 32 * c, r);
          }
          tmem_st_wait();
        }
        m = m_new;
        tc_fence_before();
        mbar_arrive(bar(C::B_PFULL + slot));
      }
      // ---- epilogue: O = u / l, LSE = ln 2 * (m + log2 l)
      if (ok && wait_bar(bar(C::B_OFULL + slot), 0u, ctl)) {
        tc_fence_after();
        const float inv_l = 1.f / l;
        const bool row_ok = i < p.Sq;
        TIn *dst = static_cast<TIn *>(p.o) + b * p.so0 + h[slot] * p.so1 + i * p.so2;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tO + 32 * c, r);
          if (row_ok) {
            uint4 *d4 = reinterpret_cast<uint4 *>(dst + 32 * c);
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              uint4 u;
              u.x = In16<TIn>::pack2(__uint_as_float(r[8 * g + 0]) * inv_l,
                                     __uint_as_float(r[8 * g + 1]) * inv_l);
              u.y = In16<TIn>::pack2(__uint_as_float(r[8 * g + 2]) * inv_l,
                                     __uint_as_float(r[8 * g + 3]) * inv_l);
              u.z = In16<TIn>::pack2(__uint_as_float(r[8 * g + 4]) * inv_l,
                                     __uint_as_float(r[8 * g + 5]) * inv_l);
              u.w = In16<TIn>::pack2(__uint_as_float(r[8 * g + 6]) * inv_l,
                                     __uint_as_float(r[8 * g + 7]) * inv_l);
              d4[g] = u;
            }
          }
        }
        if (row_ok && p.lse)
          p.lse[((int64_t)b * p.Hq + h[slot]) * p.Sq + i] = (m + log2f(l)) * 0.69314718055994531f;
      }
    }
  } else if (warp < 12) {
    // =============================================================== rotation
    const int t = threadIdx.x - kWarpRot * 32;
    const TIn *qbase = static_cast<const TIn *>(p.q);
    const TIn *kbase = static_cast<const TIn *>(p.k) + b * p.sk0 + hk * p.sk1;
    for (int s = 0; s < 2; ++s) {
      if (!act[s]) continue;
      const int64_t i = m0[s] + t;
      const bool valid = i < p.Sq;
      const TIn *src = qbase + b * p.sq0 + h[s] * p.sq1 + (valid ? i : 0) * p.sq2;
      rotate_row<D, TIn>(src, valid, p.kv_off + i, smem + C::OFF_Q + s * C::TILE, t, p);
      fence_proxy_async_smem();
      mbar_arrive(bar(C::B_QFULL + s));
    }
    for (int n = 0; n < N; ++n) {
      const int st = n % C::NS;
      if (n >= C::NS && !wait_bar(bar(C::B_KEMPTY + st), (uint32_t)((n / C::NS - 1) & 1), ctl))
        break;
      const int64_t j = (int64_t)n * 128 + t;
      const bool valid = j < p.Sk;
      rotate_row<D, TIn>(kbase + (valid ? j : 0) * p.sk2, valid, j, smem + C::OFF_K + st * C::TILE,
                         t, p);
      fence_proxy_async_smem();
      mbar_arrive(bar(C::B_KFULL + st));
    }
  } else if (warp == kWarpTma) {
    // ==================================================================== TMA
    if (lane == 0) {
      int issued = 0;
      for (int n = 0; n < N; ++n) {
        const int st = n % C::NS;
        if (n >= C::NS && !wait_bar(bar(C::B_VEMPTY + st), (uint32_t)((n / C::NS - 1) & 1), ctl))
          break;
        mbar_arrive_expect_tx(bar(C::B_VFULL + st), (uint32_t)C::TILE);
        const int logical[3] = {n * 128, hk, b};
        const int c1 = logical[p.vperm[0]], c2 = logical[p.vperm[1]], c3 = logical[p.vperm[2]];
#pragma unroll
        for (int sub = 0; sub < D / 64; ++sub)
          tma_load_4d(sbase + C::OFF_V + st * C::TILE + sub * C::SUBT, &tmap_v,
                      bar(C::B_VFULL + st), sub * 64, c1, c2, c3);
        issued = n + 1;
      }
      if (*abort_flag) {  // let copies already in flight land before the block exits
        for (int n = max(0, issued - C::NS); n < issued; ++n)
          wait_bar_drain(bar(C::B_VFULL + n % C::NS), (uint32_t)((n / C::NS) & 1));
      }
    }
  } else {
    // ==================================================================== MMA
    if (lane == 0) {
      constexpr uint32_t tin_bf16 = std::is_same<TIn, __nv_bfloat16>::value ? 1u : 0u;
      constexpr uint32_t IDESC_S = idesc_f16(0u, 0u, 128);      // fp16 x fp16, K-major B
      constexpr uint32_t IDESC_PV = idesc_f16(tin_bf16, 1u, D);  // P x V, V N-major
      const uint32_t q_addr[2] = {sbase + C::OFF_Q, sbase + C::OFF_Q + C::TILE};
      auto mma_s = [&](int s, int st) {
        const uint32_t kaddr = sbase + C::OFF_K + st * C::TILE;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::SUBT + (kk & 3) * 32;
          mma_ss(tmem + C::s_col(s), sdesc_sw128(q_addr[s] + off, 16, 1024),
                 sdesc_sw128(kaddr + off, 16, 1024), IDESC_S, kk > 0 ? 1u : 0u);
        }
      };
      auto mma_pv = [&](int s, int st, bool acc) {
        const uint32_t vaddr = sbase + C::OFF_V + st * C::TILE;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + C::o_col(s), tmem + C::s_col(s) + kk * 8,
                 sdesc_sw128(vaddr + kk * 2048, C::SUBT, 1024), IDESC_PV,
                 (acc || kk > 0) ? 1u : 0u);
      };
      auto part = [&](int s, int n) { return n < nend[s]; };
      bool ok = true;
      for (int s = 0; s < 2 && ok; ++s)
        if (act[s]) ok = wait_bar(bar(C::B_QFULL + s), 0u, ctl);
      if (ok && N > 0) ok = wait_bar(bar(C::B_KFULL + 0), 0u, ctl);
      if (ok && N > 0) {
        for (int s = 0; s < 2; ++s)
          if (part(s, 0)) {
            mma_s(s, 0);
            tc_commit(bar(C::B_SFULL + s));
          }
        tc_commit(bar(C::B_KEMPTY + 0));
      }
      for (int n = 0; ok && n < N; ++n) {
        const int st = n % C::NS, nst = (n + 1) % C::NS;
        if (!wait_bar(bar(C::B_VFULL + st), (uint32_t)((n / C::NS) & 1), ctl)) { ok = false; break; }
        bool k_next = false;
        for (int s = 0; s < 2; ++s) {
          if (!part(s, n)) continue;
          if (!wait_bar(bar(C::B_PFULL + s), (uint32_t)(n & 1), ctl)) { ok = false; break; }
          tc_fence_after();
          mma_pv(s, st, n > 0);
          if (n == nend[s] - 1) tc_commit(bar(C::B_OFULL + s));
          if (part(s, n + 1)) {
            if (!k_next) {
              if (!wait_bar(bar(C::B_KFULL + nst), (uint32_t)(((n + 1) / C::NS) & 1), ctl)) {
                ok = false;
                break;
              }
              k_next = true;
            }
            mma_s(s, nst);
            tc_commit(bar(C::B_SFULL + s));
          }
        }
        if (!ok) break;
        tc_commit(bar(C::B_VEMPTY + st));
        if (k_next) tc_commit(bar(C::B_KEMPTY + nst));
      }
      // all issued MMAs complete before tensor memory is released
      tc_commit(bar(C::B_DONE));
      wait_bar_drain(bar(C::B_DONE), 0u);
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

// V as a 4-D tensor map: dim 0 = head dim (contiguous), dims 1..3 = key row,
// kv head and batch ordered by increasing stride (size-1 dims last); the box
// is 64 head-dim elements x 128 key rows (1 along the other dims), with the
// 128-byte swizzle.
cudaError_t make_v_map(const AttnArgs &a, CUtensorMap *map, int vperm[3]) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  struct Dim { uint64_t size, stride; int logical; };
  Dim d[3] = {{(uint64_t)a.Sk, (uint64_t)a.sv[2] * 2, 0},
              {(uint64_t)a.Hkv, (uint64_t)a.sv[1] * 2, 1},
              {(uint64_t)a.B, (uint64_t)a.sv[0] * 2, 2}};
  std::stable_sort(d, d + 3, [](const Dim &x, const Dim &y) {
    if ((x.size == 1) != (y.size == 1)) return y.size == 1;
    return x.stride < y.stride;
  });
  uint64_t prev_extent = (uint64_t)a.D * 2;
  for (int i = 0; i < 3; ++i) {
    if (d[i].size == 1 || d[i].stride == 0) d[i].stride = (prev_extent + 15) & ~uint64_t(15);
    prev_extent = d[i].stride * d[i].size;
    vperm[i] = d[i].logical;
  }
  const cuuint64_t gdim[4] = {(cuuint64_t)a.D, d[0].size, d[1].size, d[2].size};
  const cuuint64_t gstride[3] = {d[0].stride, d[1].stride, d[2].stride};
  cuuint32_t box[4] = {64, 1, 1, 1};
  for (int i = 0; i < 3; ++i)
    if (d[i].logical == 0) box[1 + i] = 128;  // 128 key rows, whichever map dim holds them
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType dt =
      a.dt == RA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUresult r = enc(map, dt, 4, const_cast<void *>(a.v), gdim, gstride, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D, typename TIn>
cudaError_t launch_typed(const AttnArgs &a, const CUtensorMap &map, const TcParams &p,
                         unsigned grid, cudaStream_t s) {
  using C = TcCfg<D>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(attn_tc_kernel<D, TIn>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;
  attn_tc_kernel<D, TIn><<<grid, kThreads, C::SMEM, s>>>(map, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_tc(const AttnArgs &a, cudaStream_t s) {
  if (a.D != 64 && a.D != 128) return cudaErrorNotSupported;
  CUtensorMap map;
  TcParams p{};
  cudaError_t e = make_v_map(a, &map, p.vperm);
  if (e != cudaSuccess) return e;
  p.q = a.q; p.k = a.k; p.o = a.o; p.lse = a.lse;
  p.sq0 = a.sq[0]; p.sq1 = a.sq[1]; p.sq2 = a.sq[2];
  p.sk0 = a.sk[0]; p.sk1 = a.sk[1]; p.sk2 = a.sk[2];
  p.so0 = a.so[0]; p.so1 = a.so[1]; p.so2 = a.so[2];
  p.Sq = a.Sq; p.Sk = a.Sk; p.kv_off = a.kv_offset;
  p.Hq = a.Hq; p.G = a.Hq / a.Hkv;
  p.pack_heads = (p.G % 2 == 0) ? 1 : 0;
  p.units_per_b = p.pack_heads ? a.Hq / 2 : a.Hq;
  p.n_units = a.B * p.units_per_b;
  p.n_qt = (int)(p.pack_heads ? (a.Sq + 127) / 128 : (a.Sq + 255) / 256);
  p.apply_rope = a.apply_rope; p.rot_dim = a.rot_dim; p.layout = a.layout;
  p.cos_t = a.cos_t; p.sin_t = a.sin_t;
  p.scale_log2 = (float)((double)a.scale * 1.4426950408889634);
  p.status = a.status;
  const int64_t grid = (int64_t)p.n_qt * p.n_units;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffff) return cudaErrorInvalidConfiguration;
  const bool bf = a.dt == RA_BF16;
  if (a.D == 64)
    return bf ? launch_typed<64, __nv_bfloat16>(a, map, p, (unsigned)grid, s)
              : launch_typed<64, __half>(a, map, p, (unsigned)grid, s);
  return bf ? launch_typed<128, __nv_bfloat16>(a, map, p, (unsigned)grid, s)
            : launch_typed<128, __half>(a, map, p, (unsigned)grid, s);
}

}  // namespace ra

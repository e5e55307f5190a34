// Tensor-core split kernel of the decode attention (tcgen05 + TMEM + TMA),
// bf16/fp16, head size 128, up to 64 query rows per kv head.
//
// What is computed: the chunk part of decode.cu's split-KV scheme ("RoPE and
// FlashAttention: relative positions and online softmax", sections 4-5):
// for one (chunk, kv head, sequence), the scores of every query row of the
// kv head's group against the chunk's keys (already rotated, section 2), the
// softmax over the chunk, P V, and the chunk's log-sum-exp.
//
// GB300 design.  A decode step has few query rows per kv head (GQA group x
// new tokens: 1..64) and many keys, so the products are computed transposed:
//   S^T = K Q^T   (M = 128 keys, N = query columns padded to 16/32/64,
//                  K = 128 head dims; A = the K tile, B = Q, both K-major),
//   O^T = V^T P^T (M = 128 head dims, N = query columns, K = 128 keys; A =
//                  the V tile read MN-major, B = P^T, K-major),
// which keeps the 128-row MMA shape busy with keys instead of padding a
// handful of query rows to 128.  A chunk has at most (256 - N) / N tiles of
// 128 keys, so every score tile of the chunk stays in tensor memory (256
// columns: O^T at columns [0, N), S^T tile t at [N (1 + t), N (2 + t))) and
// the softmax is exact in two passes over TMEM -- column maxima, then
// exponentials -- with no rescaling of O.  K tiles then V tiles stream
// through a ring of 32 KB TMA stages; two blocks share an SM so that one's
// set-up and epilogue overlap the other's streaming.
//
// Roles (192 threads): warps 0-3 own TMEM lanes 0-127 (softmax over keys,
// P^T to shared memory, epilogue over head dims); warp 4 issues the TMA
// loads; warp 5 allocates TMEM and issues the MMAs.  Every mbarrier wait is
// bounded: on expiry the block records RA_ERR_DEVICE_TIMEOUT, raises an abort
// flag, lets copies and MMAs already issued finish, frees TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>

#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace ra {
namespace {

using namespace ptx;

constexpr int kThreads = 192;
constexpr int kWarpTma = 4, kWarpMma = 5;
constexpr int kTmemCols = 256;
constexpr int kTileBytes = 128 * 128 * 2;  // one K or V tile: 128 keys x 128 dims
constexpr int kHalfBytes = kTileBytes / 2;  // 64 head dims (one 128-byte swizzle column)
constexpr long long kTimeoutCycles = 1LL << 32;  // about two seconds

template <int NPAD> struct DCfg {
  static constexpr int TILES = (kTmemCols - NPAD) / NPAD;  // score tiles per chunk
  static constexpr int NS = NPAD == 16 ? 3 : 2;            // ring stages
  static constexpr int QB = NPAD * 256;                    // Q operand: two 64-dim atoms
  static constexpr int PB = NPAD * 256;                    // one P^T buffer: two 64-key atoms
  static constexpr int OFF_KV = 0;
  static constexpr int OFF_Q = NS * kTileBytes;
  static constexpr int OFF_P = OFF_Q + QB;
  static constexpr int OFF_RED = OFF_P + 2 * PB;        // float [4][NPAD]
  static constexpr int OFF_M = OFF_RED + 4 * NPAD * 4;  // float [NPAD]: column max, log2 units
  static constexpr int OFF_L = OFF_M + NPAD * 4;        // float [NPAD]: column sum
  static constexpr int OFF_BAR = OFF_L + NPAD * 4;
  static constexpr int B_FULL = 0, B_EMPTY = NS, B_QFULL = 2 * NS, B_SFULL = 2 * NS + 1,
                       B_PFULL = 2 * NS + 2, B_PEMPTY = 2 * NS + 4, B_OFULL = 2 * NS + 6,
                       B_DONE = 2 * NS + 7, NBAR = 2 * NS + 8;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;   // TMEM base, abort flag
  static constexpr int SMEM = OFF_MISC + 16 + 1024;     // + slack for 1024-byte alignment
  static_assert(TILES >= 1 && OFF_BAR % 8 == 0 && QB % 1024 == 0, "layout");
};

struct DTcParams {
  const void *q;
  void *o;
  float *lse;
  int64_t sq0, sq1, sq2, so0, so1, so2;
  const int64_t *seq_start;
  int64_t n_seqs, cache_rows;
  const int32_t *seq_ids, *kv_len;
  int64_t max_kv_len;
  int Hq, G, Sq, n_cols;
  float scale_log2;
  int splits;
  int64_t chunk;
  float *ws_o, *ws_lse;
  int kperm[2], vperm[2];  // tensor-map dims 1..2 -> logical coordinate (0 row, 1 kv head)
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

// Visibility of key j to query column c: every key j <= L - Sq is seen by
// all columns; of the last Sq keys, column c (query i = c % Sq at position
// L - Sq + i) sees those with j - (L - Sq) <= i; padding columns see every
// key of the sequence.
__device__ __forceinline__ bool visible(int64_t over, int c, int n_cols, int Sq) {
  if (over <= 0) return true;
  if (c >= n_cols) return over < Sq;  // j < L
  return over <= c % Sq;
}

template <typename TIn, int NPAD>
__global__ void __launch_bounds__(kThreads, 2)
    attn_decode_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                          const __grid_constant__ CUtensorMap tmap_v, const DTcParams p) {
  using C = DCfg<NPAD>;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;

  // ---- the block's keys [j0, j1) of entry b (uniform over the block)
  const int64_t sq = p.seq_ids ? (int64_t)p.seq_ids[b] : (int64_t)b;
  const int64_t L = p.kv_len[b];
  bool valid = sq >= 0 && sq < p.n_seqs && L >= p.Sq && L <= p.max_kv_len;
  int64_t row0 = 0;
  if (valid) {
    row0 = p.seq_start[sq];
    valid = row0 >= 0 && row0 + L <= p.cache_rows;
  }
  if (!valid) {
    if (split == 0 && hk == 0 && tid == 0) record_status(p.status, RA_ERR_POSITION_RANGE);
    return;
  }
  const int64_t j0 = (int64_t)split * p.chunk;
  if (j0 >= L) return;
  const int64_t j1 = min(L, j0 + p.chunk);
  const int T = (int)((j1 - j0 + 127) / 128);  // <= C::TILES (plan)
  const int last_rows = (int)(j1 - j0 - 128 * (int64_t)(T - 1));  // valid rows of the last tile

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  auto bar = [&](int i) { return sbase + C::OFF_BAR + 8u * (uint32_t)i; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
  const Ctl ctl{abort_flag, p.status};

  if (tid == 0) {
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(bar(C::B_FULL + i), 1);
      mbar_init(bar(C::B_EMPTY + i), 1);
    }
    mbar_init(bar(C::B_QFULL), 128);
    mbar_init(bar(C::B_SFULL), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::B_PFULL + i), 128);
      mbar_init(bar(C::B_PEMPTY + i), 1);
    }
    mbar_init(bar(C::B_OFULL), 1);
    mbar_init(bar(C::B_DONE), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kWarpTma && lane == 0) {
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWarpTma) {
    // ================================================================ TMA
    if (lane == 0) {
      int issued = 0;
      for (int n = 0; n < 2 * T; ++n) {
        const int st = n % C::NS;
        if (n >= C::NS &&
            !wait_bar(bar(C::B_EMPTY + st), (uint32_t)((n / C::NS - 1) & 1), ctl))
          break;
        const bool isv = n >= T;
        const int row = (int)(row0 + j0 + 128 * (int64_t)(isv ? n - T : n));
        const CUtensorMap *map = isv ? &tmap_v : &tmap_k;
        const int *perm = isv ? p.vperm : p.kperm;
        const int c1 = perm[0] == 0 ? row : hk, c2 = perm[1] == 0 ? row : hk;
        const uint32_t dst = sbase + C::OFF_KV + (uint32_t)(st * kTileBytes);
        mbar_arrive_expect_tx(bar(C::B_FULL + st), (uint32_t)kTileBytes);
        tma_load_3d(dst, map, bar(C::B_FULL + st), 0, c1, c2);
        tma_load_3d(dst + kHalfBytes, map, bar(C::B_FULL + st), 64, c1, c2);
        issued = n + 1;
      }
      if (*abort_flag)  // copies in flight land before the block exits
        for (int n = max(0, issued - C::NS); n < issued; ++n)
          wait_bar_drain(bar(C::B_FULL + n % C::NS), (uint32_t)((n / C::NS) & 1));
    }
  } else if (warp == kWarpMma) {
    // ================================================================ MMA
    // whole warp; one elected lane issues
    constexpr uint32_t ab = std::is_same<TIn, __nv_bfloat16>::value ? 1u : 0u;
    constexpr uint32_t IDESC_S = idesc_f16_ab(ab, 0u, 0u, NPAD);  // K x Q^T
    constexpr uint32_t IDESC_O = idesc_f16_ab(ab, 1u, 0u, NPAD);  // V^T (MN-major) x P^T
    constexpr uint32_t HI = sdesc_hi_sw128(1024);
    const uint32_t k_lo0 = sdesc_lo(sbase + C::OFF_KV, 16);
    const uint32_t v_lo0 = sdesc_lo(sbase + C::OFF_KV, kHalfBytes);
    const uint32_t q_lo0 = sdesc_lo(sbase + C::OFF_Q, 16);
    const uint32_t p_lo0 = sdesc_lo(sbase + C::OFF_P, 16);
    bool ok = wait_all(bar(C::B_QFULL), 0u, ctl);
    for (int t = 0; ok && t < T; ++t) {
      const int st = t % C::NS;
      if (!wait_all(bar(C::B_FULL + st), (uint32_t)((t / C::NS) & 1), ctl)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t a_lo = k_lo0 + (uint32_t)(st * kTileBytes >> 4);
      const uint32_t dS = tmem + (uint32_t)(NPAD * (1 + t));
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t oa = (uint32_t)(((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4);
        const uint32_t ob = (uint32_t)(((kk >> 2) * (NPAD * 128) + (kk & 3) * 32) >> 4);
        mma_ss_w(dS, sdesc_join(a_lo + oa, HI), sdesc_join(q_lo0 + ob, HI), IDESC_S,
               kk > 0 ? 1u : 0u);
      }
      tc_commit_w(bar(C::B_EMPTY + st));
    }
    if (ok) tc_commit_w(bar(C::B_SFULL));
    for (int t = 0; ok && t < T; ++t) {
      const int n = T + t, st = n % C::NS;
      if (!wait_all(bar(C::B_FULL + st), (uint32_t)((n / C::NS) & 1), ctl) ||
          !wait_all(bar(C::B_PFULL + (t & 1)), (uint32_t)((t >> 1) & 1), ctl)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t a_lo = v_lo0 + (uint32_t)(st * kTileBytes >> 4);
      const uint32_t b_lo = p_lo0 + (uint32_t)((t & 1) * C::PB >> 4);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t oa = (uint32_t)((kk * 2048) >> 4);  // 16 keys x 128 bytes
        const uint32_t ob = (uint32_t)(((kk >> 2) * (NPAD * 128) + (kk & 3) * 32) >> 4);
        mma_ss_w(tmem, sdesc_join(a_lo + oa, HI), sdesc_join(b_lo + ob, HI), IDESC_O,
               (t > 0 || kk > 0) ? 1u : 0u);
      }
      tc_commit_w(bar(C::B_EMPTY + st));
      tc_commit_w(bar(C::B_PEMPTY + (t & 1)));
    }
    if (ok) tc_commit_w(bar(C::B_OFULL));
    // every issued MMA completes before tensor memory is released
    tc_commit_w(bar(C::B_DONE));
    wait_bar_drain(bar(C::B_DONE), 0u);

  } else {
    // ======================================================= softmax (0-3)
    // Q rows into the B-operand layout: row c = query column (group head
    // c / Sq, query c % Sq), 128-byte swizzle, two 64-dim atoms; padding zero.
    for (int e = tid; e < NPAD * 16; e += 128) {
      const int r = e >> 4, cc = e & 15;
      uint4 val = make_uint4(0u, 0u, 0u, 0u);
      if (r < p.n_cols) {
        const int hg = r / p.Sq, i = r - hg * p.Sq;
        const TIn *src = static_cast<const TIn *>(p.q) + b * p.sq0 +
                         (int64_t)(hk * p.G + hg) * p.sq1 + i * p.sq2 + cc * 8;
        val = *reinterpret_cast<const uint4 *>(src);
      }
      *reinterpret_cast<uint4 *>(smem + C::OFF_Q + (cc >> 3) * (NPAD * 128) + r * 128 +
                                 (((cc & 7) ^ (r & 7)) << 4)) = val;
    }
    fence_proxy_async_smem();
    mbar_arrive(bar(C::B_QFULL));

    float *red = reinterpret_cast<float *>(smem + C::OFF_RED);
    float *msl = reinterpret_cast<float *>(smem + C::OFF_M);
    float *lsum = reinterpret_cast<float *>(smem + C::OFF_L);
    const uint32_t lanes = tmem + ((uint32_t)(warp * 32) << 16);
    const int64_t over0 = j0 + tid - (L - p.Sq);  // key j of tile t: over = over0 + 128 t
    const float sl2 = p.scale_log2;

    // ---- pass 1: column maxima of the raw scores
    bool ok = __all_sync(0xffffffffu, wait_bar(bar(C::B_SFULL), 0u, ctl));
    tc_fence_after();
    {
      float mloc[NPAD];
#pragma unroll
      for (int c = 0; c < NPAD; ++c) mloc[c] = -INFINITY;
      for (int t = 0; ok && t < T; ++t) {
        const int64_t over = over0 + 128 * t;
#pragma unroll
        for (int ch = 0; ch < NPAD / 16; ++ch) {
          uint32_t r[16];
          tmem_ld16(lanes + (uint32_t)(NPAD * (1 + t) + 16 * ch), r);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int c = 16 * ch + k;
            if (visible(over, c, p.n_cols, p.Sq)) mloc[c] = fmaxf(mloc[c], __uint_as_float(r[k]));
          }
        }
      }
#pragma unroll
      for (int c = 0; c < NPAD; ++c) {
        const float v = warp_max(mloc[c]);
        if (lane == 0) red[warp * NPAD + c] = v;
      }
    }
    named_bar_sync(1, 128);
    if (tid < NPAD) {
      const float m = fmaxf(fmaxf(red[tid], red[NPAD + tid]),
                            fmaxf(red[2 * NPAD + tid], red[3 * NPAD + tid]));
      msl[tid] = m * sl2;  // -inf when no key of the chunk is visible to the column
    }
    named_bar_sync(1, 128);

    // ---- pass 2: P = 2^(s sl2 - m sl2) into P^T tiles, column sums
    float lloc[NPAD];
#pragma unroll
    for (int c = 0; c < NPAD; ++c) lloc[c] = 0.f;
    const int atom = tid >> 6, sw = (tid & 63) >> 3, sub = (tid & 7) * 2;
    for (int t = 0; t < T; ++t) {
      const int buf = t & 1;
      if (ok && t >= 2)
        ok = __all_sync(0xffffffffu,
                        wait_bar(bar(C::B_PEMPTY + buf), (uint32_t)(((t >> 1) - 1) & 1), ctl));
      if (!ok) break;
      const int64_t over = over0 + 128 * t;
      uint8_t *pb = smem + C::OFF_P + buf * C::PB + atom * (NPAD * 128) + sub;
#pragma unroll
      for (int ch = 0; ch < NPAD / 16; ++ch) {
        uint32_t r[16];
        tmem_ld16(lanes + (uint32_t)(NPAD * (1 + t) + 16 * ch), r);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int c = 16 * ch + k;
          const float pv = visible(over, c, p.n_cols, p.Sq)
                               ? ex2(fmaf(__uint_as_float(r[k]), sl2, -msl[c]))
                               : 0.f;
          lloc[c] += pv;
          *reinterpret_cast<TIn *>(pb + c * 128 + ((sw ^ (c & 7)) << 4)) = Elem<TIn>::store(pv);
        }
      }
      if (t == T - 1 && tid >= last_rows) {
        // rows past the sequence in the last V tile may hold anything (even
        // NaN, which a zero probability would not cancel): zero them
        const int n = T + t, st = n % C::NS;
        if (wait_bar(bar(C::B_FULL + st), (uint32_t)((n / C::NS) & 1), ctl)) {
          uint8_t *row = smem + C::OFF_KV + st * kTileBytes + tid * 128;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            *reinterpret_cast<uint4 *>(row + 16 * k) = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4 *>(row + kHalfBytes + 16 * k) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(C::B_PFULL + buf));
    }
    ok = __all_sync(0xffffffffu, ok && !*abort_flag);
#pragma unroll
    for (int c = 0; c < NPAD; ++c) {
      const float v = warp_sum(lloc[c]);
      if (lane == 0) red[warp * NPAD + c] = v;
    }
    named_bar_sync(1, 128);
    if (tid < NPAD) lsum[tid] = (red[tid] + red[NPAD + tid]) + (red[2 * NPAD + tid] + red[3 * NPAD + tid]);
    named_bar_sync(1, 128);

    // ---- epilogue: thread tid holds head dim tid of every column of O^T
    if (ok) ok = __all_sync(0xffffffffu, wait_bar(bar(C::B_OFULL), 0u, ctl));
    tc_fence_after();
    if (ok) {
#pragma unroll
      for (int ch = 0; ch < NPAD / 16; ++ch) {
        uint32_t r[16];
        tmem_ld16(lanes + (uint32_t)(16 * ch), r);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int c = 16 * ch + k;
          if (c >= p.n_cols) continue;
          const float l = lsum[c];
          const float val = l > 0.f ? __uint_as_float(r[k]) / l : 0.f;
          const int hg = c / p.Sq, i = c - hg * p.Sq, h = hk * p.G + hg;
          if (p.splits == 1) {
            static_cast<TIn *>(p.o)[b * p.so0 + (int64_t)h * p.so1 + i * p.so2 + tid] =
                Elem<TIn>::store(val);
          } else {
            const int64_t wrow = (((int64_t)b * p.Hq + h) * p.Sq + i) * p.splits + split;
            p.ws_o[wrow * 128 + tid] = val;
          }
        }
      }
      if (tid < p.n_cols) {
        const int c = tid, hg = c / p.Sq, i = c - hg * p.Sq, h = hk * p.G + hg;
        const float l = lsum[c];
        const float lse = l > 0.f ? msl[c] * 0.6931471805599453f + logf(l) : -INFINITY;
        if (p.splits == 1) {
          if (p.lse) p.lse[((int64_t)b * p.Hq + h) * p.Sq + i] = lse;
        } else {
          p.ws_lse[(((int64_t)b * p.Hq + h) * p.Sq + i) * p.splits + split] = lse;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------- host
// A cache buffer as a tensor map over (row, kv head): box 64 of the 128
// head dims x 128 rows, 128-byte swizzle; rows past the buffer read as zero.
cudaError_t make_cache_map(void *base, int64_t rows, int Hkv, const int64_t strides[2],
                           ra_dtype dt, CUtensorMap *map, int perm[2]) {
  const int64_t size[3] = {rows, Hkv, 1}, stride[3] = {strides[0], strides[1], 0};
  int p3[3];
  const cudaError_t e = make_row_tile_map(base, dt == RA_BF16, 128, 2, size, stride, map, p3);
  perm[0] = p3[0];
  perm[1] = p3[1];
  return e;
}

template <typename TIn, int NPAD>
cudaError_t launch_typed(const CUtensorMap &mk, const CUtensorMap &mv, const DTcParams &p,
                         const DecodeArgs &a, cudaStream_t s) {
  using C = DCfg<NPAD>;
  static PerDeviceOnce once;
  const cudaError_t attr_err = once.run([] {
    return cudaFuncSetAttribute(attn_decode_tc_kernel<TIn, NPAD>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;
  if (a.plan.chunk > (int64_t)C::TILES * 128) return cudaErrorInvalidValue;  // plan mismatch
  const dim3 grid((unsigned)a.plan.splits, (unsigned)a.Hkv, (unsigned)a.B);
  attn_decode_tc_kernel<TIn, NPAD><<<grid, kThreads, C::SMEM, s>>>(mk, mv, p);
  note_launch("attn_decode_tc_kernel");
  return cudaGetLastError();
}

template <typename TIn>
cudaError_t launch_npad(const CUtensorMap &mk, const CUtensorMap &mv, const DTcParams &p,
                        const DecodeArgs &a, cudaStream_t s) {
  if (p.n_cols <= 16) return launch_typed<TIn, 16>(mk, mv, p, a, s);
  if (p.n_cols <= 32) return launch_typed<TIn, 32>(mk, mv, p, a, s);
  return launch_typed<TIn, 64>(mk, mv, p, a, s);
}

}  // namespace

cudaError_t launch_attn_decode_tc(const DecodeArgs &a, cudaStream_t s) {
  const int G = a.Hq / a.Hkv;
  if (a.D != 128 || a.dt == RA_F32 || G * a.Sq > 64) return cudaErrorNotSupported;
  if (a.cache.rows > 0x7fffffff || a.Hkv > 65535 || a.B > 65535) return cudaErrorNotSupported;
  DTcParams p{};
  CUtensorMap mk, mv;
  cudaError_t e = make_cache_map(a.cache.k, a.cache.rows, a.Hkv, a.cache.k_strides, a.dt, &mk,
                                 p.kperm);
  if (e == cudaSuccess)
    e = make_cache_map(a.cache.v, a.cache.rows, a.Hkv, a.cache.v_strides, a.dt, &mv, p.vperm);
  if (e != cudaSuccess) return e;
  p.q = a.q; p.o = a.o; p.lse = a.lse;
  p.sq0 = a.sq[0]; p.sq1 = a.sq[1]; p.sq2 = a.sq[2];
  p.so0 = a.so[0]; p.so1 = a.so[1]; p.so2 = a.so[2];
  p.seq_start = a.cache.seq_start; p.n_seqs = a.cache.n_seqs; p.cache_rows = a.cache.rows;
  p.seq_ids = a.seq_ids; p.kv_len = a.kv_len; p.max_kv_len = a.max_kv_len;
  p.Hq = a.Hq; p.G = G; p.Sq = a.Sq; p.n_cols = G * a.Sq;
  p.scale_log2 = (float)((double)a.scale * 1.4426950408889634);
  p.splits = a.plan.splits; p.chunk = a.plan.chunk;
  if (a.plan.splits > 1) {
    p.ws_o = static_cast<float *>(a.workspace);
    p.ws_lse = reinterpret_cast<float *>(static_cast<char *>(a.workspace) + a.plan.ws_lse_offset);
  }
  p.status = a.status;
  return a.dt == RA_BF16 ? launch_npad<__nv_bfloat16>(mk, mv, p, a, s)
                         : launch_npad<__half>(mk, mv, p, a, s);
}

}  // namespace ra

// Rotation of 128-row tiles into tcgen05 operand layout (shared by the
// tensor-core kernels): rows are rotated in fp32 with the fp32 cos/sin table
// and written as fp16 into 128-byte-swizzled shared memory, 64 columns per
// 16 KB sub-tile ("RoPE and FlashAttention: relative positions and online
// softmax", section 1: NeoX pairs (i, i + r/2) or GPT-J pairs (2i, 2i+1)).
// The params type P provides apply_rope, rot_dim, layout, cos_t, sin_t and
// table_rows.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "common.cuh"

namespace ra {
namespace rot {

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
template <int D, typename TIn, typename P>
__device__ __forceinline__ void rotate_row(const TIn *src, bool valid, int64_t pos, uint8_t *tile,
                                           int row, const P &p) {
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

// ------------------------------------------------ full-rotation tile path
// Used when rot_dim == D.  Thread t of the rotation warpgroup owns NP pairs
// (chunk c = t % CH of a row) over RPG consecutive rows starting at row
// g * RPG (g = t / CH), so the CH lanes of a row read its 16-byte chunks
// contiguously.  cos/sin come from the table row of the group's first
// position; each following row advances them by one step of angle addition
// with (cos theta_i, sin theta_i) from table row 1, in fp32:
//   cos((p+1)theta) = cos(p theta) cos theta - sin(p theta) sin theta,
//   sin((p+1)theta) = sin(p theta) cos theta + cos(p theta) sin theta.
// Arithmetic runs on packed fp32 pairs (two pairs per instruction).  For
// GPT-J the even/odd members of the pairs in a 16-byte chunk play the roles
// of the NeoX low/high halves, so both layouts share one code path.
template <int D, int LAYOUT>
struct FullRot {
  static constexpr int NP = (LAYOUT == RA_NEOX) ? 8 : 4;          // pairs per thread per row
  static constexpr int CH = (LAYOUT == RA_NEOX) ? D / 16 : D / 8;  // threads per row
  static constexpr int RPG = CH;                                   // rows per thread
  static constexpr int LD = (LAYOUT == RA_NEOX) ? 2 : 1;           // 16-byte loads per row
  static constexpr int NG = NP / 2;                                // float2 groups per row
};

template <typename TIn> __device__ __forceinline__ float2 unpack2(uint32_t w);
template <> __device__ __forceinline__ float2 unpack2<__nv_bfloat16>(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
template <> __device__ __forceinline__ float2 unpack2<__half>(uint32_t w) {
  return __half22float2(*reinterpret_cast<const __half2 *>(&w));
}
__device__ __forceinline__ uint32_t w_of(const uint4 &u, int k) {
  return k == 0 ? u.x : (k == 1 ? u.y : (k == 2 ? u.z : u.w));
}

template <int D, typename TIn, int LAYOUT>
__device__ __forceinline__ void full_rot_load(
    const TIn *rows, int64_t row_stride, int64_t nvalid, int t,
    uint4 (&raw)[FullRot<D, LAYOUT>::RPG][FullRot<D, LAYOUT>::LD]) {
  using F = FullRot<D, LAYOUT>;
  const int c = t % F::CH, r0 = (t / F::CH) * F::RPG;
#pragma unroll
  for (int r = 0; r < F::RPG; ++r) {
    const bool ok = r0 + r < nvalid;
    const uint4 *src = reinterpret_cast<const uint4 *>(rows + (ok ? (r0 + r) : 0) * row_stride);
#pragma unroll
    for (int l = 0; l < F::LD; ++l)
      raw[r][l] = ok ? __ldg(src + ((LAYOUT == RA_NEOX) ? c + l * (D / 16) : c))
                     : make_uint4(0u, 0u, 0u, 0u);
  }
}

// cos/sin of this thread's pairs at `pos` (table row), as float2 groups.
template <int D, int LAYOUT, typename P>
__device__ __forceinline__ void full_rot_table(const P &p, int64_t pos, int t,
                                               float2 (&cv)[FullRot<D, LAYOUT>::NG],
                                               float2 (&sv)[FullRot<D, LAYOUT>::NG]) {
  using F = FullRot<D, LAYOUT>;
  const int pair0 = (t % F::CH) * F::NP;
  const float4 *c4 = reinterpret_cast<const float4 *>(p.cos_t + pos * (D / 2) + pair0);
  const float4 *s4 = reinterpret_cast<const float4 *>(p.sin_t + pos * (D / 2) + pair0);
#pragma unroll
  for (int q = 0; q < F::NP / 4; ++q) {
    const float4 a = __ldg(c4 + q), b = __ldg(s4 + q);
    cv[2 * q] = make_float2(a.x, a.y);
    cv[2 * q + 1] = make_float2(a.z, a.w);
    sv[2 * q] = make_float2(b.x, b.y);
    sv[2 * q + 1] = make_float2(b.z, b.w);
  }
}

template <int D, typename TIn, int LAYOUT>
__device__ __forceinline__ void full_rot_store(
    const uint4 (&raw)[FullRot<D, LAYOUT>::RPG][FullRot<D, LAYOUT>::LD],
    float2 (&cb)[FullRot<D, LAYOUT>::NG], float2 (&sb)[FullRot<D, LAYOUT>::NG],
    const float2 (&cst)[FullRot<D, LAYOUT>::NG], const float2 (&sst)[FullRot<D, LAYOUT>::NG],
    uint8_t *tile, int t) {
  using F = FullRot<D, LAYOUT>;
  const int c = t % F::CH, r0 = (t / F::CH) * F::RPG;
#pragma unroll
  for (int r = 0; r < F::RPG; ++r) {
    const int row = r0 + r;
    uint32_t olo[4], ohi[4];
#pragma unroll
    for (int j = 0; j < F::NG; ++j) {
      float2 L, H;
      if (LAYOUT == RA_NEOX) {
        L = unpack2<TIn>(w_of(raw[r][0], j));
        H = unpack2<TIn>(w_of(raw[r][1], j));
      } else {  // words 2j and 2j+1 hold pairs (a, b); evens -> L, odds -> H
        const float2 u = unpack2<TIn>(w_of(raw[r][0], 2 * j));
        const float2 v = unpack2<TIn>(w_of(raw[r][0], 2 * j + 1));
        L = make_float2(u.x, v.x);
        H = make_float2(u.y, v.y);
      }
      const float2 lc = __fmul2_rn(L, cb[j]);
      const float2 hc = __fmul2_rn(H, cb[j]);
      const float2 a = __ffma2_rn(make_float2(-H.x, -H.y), sb[j], lc);  // lo*c - hi*s
      const float2 b = __ffma2_rn(L, sb[j], hc);                         // hi*c + lo*s
      if (LAYOUT == RA_NEOX) {
        olo[j] = f16x2(a.x, a.y);
        ohi[j] = f16x2(b.x, b.y);
      } else {
        olo[2 * j] = f16x2(a.x, b.x);
        olo[2 * j + 1] = f16x2(a.y, b.y);
      }
    }
    const int sw = row & 7;
    if (LAYOUT == RA_NEOX) {
      *reinterpret_cast<uint4 *>(tile + (c >> 3) * 16384 + row * 128 + (((c & 7) ^ sw) << 4)) =
          make_uint4(olo[0], olo[1], olo[2], olo[3]);
      const int ch = c + D / 16;
      *reinterpret_cast<uint4 *>(tile + (ch >> 3) * 16384 + row * 128 + (((ch & 7) ^ sw) << 4)) =
          make_uint4(ohi[0], ohi[1], ohi[2], ohi[3]);
    } else {
      *reinterpret_cast<uint4 *>(tile + (c >> 3) * 16384 + row * 128 + (((c & 7) ^ sw) << 4)) =
          make_uint4(olo[0], olo[1], olo[2], olo[3]);
    }
    if (r + 1 < F::RPG) {
#pragma unroll
      for (int j = 0; j < F::NG; ++j) {
        const float2 cn = __ffma2_rn(cb[j], cst[j], __fmul2_rn(make_float2(-sb[j].x, -sb[j].y), sst[j]));
        sb[j] = __ffma2_rn(sb[j], cst[j], __fmul2_rn(cb[j], sst[j]));
        cb[j] = cn;
      }
    }
  }
}

// Whole-tile rotation without prefetch (Q tiles, once per CTA).
template <int D, typename TIn, int LAYOUT, typename P>
__device__ __forceinline__ void rotate_tile_full(const TIn *rows, int64_t row_stride,
                                                 int64_t nvalid, int64_t pos0, uint8_t *tile,
                                                 int t, const P &p) {
  using F = FullRot<D, LAYOUT>;
  uint4 raw[F::RPG][F::LD];
  float2 cb[F::NG], sb[F::NG], cst[F::NG], sst[F::NG];
  const int64_t r0 = (t / F::CH) * F::RPG;
  full_rot_load<D, TIn, LAYOUT>(rows, row_stride, nvalid, t, raw);
  full_rot_table<D, LAYOUT>(p, r0 < nvalid ? pos0 + r0 : 0, t, cb, sb);
  full_rot_table<D, LAYOUT>(p, p.table_rows > 1 ? 1 : 0, t, cst, sst);
  full_rot_store<D, TIn, LAYOUT>(raw, cb, sb, cst, sst, tile, t);
}

}  // namespace rot
}  // namespace ra

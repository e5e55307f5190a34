// extern "C" entry points of librope_attn.so (declared in include/rope_attn.h):
// host-side argument validation, the per-device status word and kernel
// dispatch.  Every check runs before the first CUDA call, so a rejected call
// touches no device state.
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "internal.h"

namespace {

// First error recorded by any kernel on this device since the last read.
__device__ int g_ra_status_word;

thread_local char g_last_error[512] = "no error";
thread_local char g_last_launch[256] = "";

constexpr int kMaxDevices = 64;

// Split-KV workspace of attn_decode_noalloc: one region per device, resolved
// once per device with cudaGetSymbolAddress (no allocation at call time).
static __device__ __align__(256) unsigned char g_decode_scratch[RA_DECODE_STATIC_SCRATCH_BYTES];
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices];

std::mutex g_status_mu;
int *g_status_ptr[kMaxDevices];

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t dtype_size(ra_dtype dt) { return dt == RA_F32 ? 4 : 2; }
bool dtype_ok(int dt) { return dt == RA_F32 || dt == RA_BF16 || dt == RA_F16; }
bool layout_ok(int l) { return l == RA_NEOX || l == RA_GPTJ; }

// Byte footprint of a [n0][n1][D] strided array (strides in elements, >= 0).
struct Region {
  const char *base;
  int64_t span;  // bytes from base to one past the last element
  int64_t ts;    // outer (token) stride in bytes
  int64_t foot;  // bytes covered by one outer index
};

Region region(const void *p, int64_t n0, int64_t s0, int64_t n1, int64_t s1, int64_t D, size_t es) {
  Region r;
  r.base = static_cast<const char *>(p);
  r.foot = ((n1 - 1) * s1 + D) * (int64_t)es;
  r.span = (n0 - 1) * s0 * (int64_t)es + r.foot;
  r.ts = s0 * (int64_t)es;
  return r;
}

// True when the two strided regions provably share no byte: disjoint spans,
// or equal outer strides with per-row windows that do not meet (e.g. the q
// and k slices of one packed qkv buffer).
bool disjoint(const Region &a, const Region &b) {
  if (a.base + a.span <= b.base || b.base + b.span <= a.base) return true;
  if (a.ts != b.ts || a.ts <= 0 || a.foot > a.ts || b.foot > b.ts) return false;
  const Region &x = a.base <= b.base ? a : b;
  const Region &y = a.base <= b.base ? b : a;
  const int64_t r = (int64_t)(y.base - x.base) % x.ts;
  return x.foot <= r && r + y.foot <= x.ts;
}

}  // namespace

namespace ra {

ra_status fail(ra_status st, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return st;
}

void clear_launches() { g_last_launch[0] = '\0'; }

void note_launch(const char *kernel) {
  const size_t n = strlen(g_last_launch);
  snprintf(g_last_launch + n, sizeof g_last_launch - n, "%s%s", n ? " " : "", kernel);
}

void *decode_scratch_ptr(cudaError_t *err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (*err != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

int *device_status_ptr(cudaError_t *err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_status_mu);
  if (!g_status_ptr[dev]) {
    void *p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_ra_status_word);
    if (*err != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<int *>(p);
  }
  return g_status_ptr[dev];
}

bool plan_bwd_workspace(ra_dtype dt, int B, int Hq, int Hkv, int64_t Sq, int64_t Sk, int D,
                        BwdWorkspace *w) {
  if (B < 0 || Hq < 0 || Hkv < 0 || Sq < 0 || Sk < 0 || D < 0) return false;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  size_t off = up((size_t)B * Hq * (size_t)Sq * sizeof(float));  // D_i row terms
  w->qrot_off = w->krot_off = 0;
  if (dt != RA_F32) {  // rotated fp16 operands of the tensor-core kernels
    w->qrot_off = off;
    off += up((size_t)B * Hq * (size_t)Sq * D * 2);
    w->krot_off = off;
    off += up((size_t)B * Hkv * (size_t)Sk * D * 2);
  }
  w->bytes = off;
  return true;
}

int sm_count_current() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    return 148;
  return n;
}

}  // namespace ra

using ra::fail;

namespace {

// True when the rows of a [n0][n1][D] strided array share no byte (strides
// in elements): taken in increasing stride order, each dimension of size > 1
// steps past everything the smaller ones cover.
bool rows_distinct(int64_t n0, int64_t s0, int64_t n1, int64_t s1, int64_t D) {
  int64_t n[2] = {n0, n1}, st[2] = {s0, s1};
  if (st[0] > st[1]) {
    std::swap(n[0], n[1]);
    std::swap(st[0], st[1]);
  }
  int64_t ext = D;
  for (int j = 0; j < 2; ++j) {
    if (n[j] <= 1) continue;
    if (st[j] < ext) return false;
    ext = (n[j] - 1) * st[j] + ext;
  }
  return true;
}

int64_t span4(int64_t n0, int64_t s0, int64_t n1, int64_t s1, int64_t n2, int64_t s2, int64_t D,
              size_t es) {
  return ((n0 - 1) * s0 + (n1 - 1) * s1 + (n2 - 1) * s2 + D) * (int64_t)es;
}

bool spans_apart(const void *a, int64_t na, const void *b, int64_t nb) {
  const char *x = static_cast<const char *>(a), *y = static_cast<const char *>(b);
  return x + na <= y || y + nb <= x;
}

// Host checks shared by the two cache calls; nullptr when the cache is valid.
const char *cache_problem(const ra_kv_cache *c, int Hkv, int D, size_t es) {
  if (!c) return "cache must be non-NULL";
  if (!c->k || !c->v || !c->seq_start) return "cache k, v and seq_start must be non-NULL";
  if (c->rows < 1 || c->n_seqs < 1) return "cache rows and n_seqs must be >= 1";
  for (int j = 0; j < 2; ++j)
    if (c->k_strides[j] < 0 || c->v_strides[j] < 0) return "cache strides must be >= 0";
  if (!rows_distinct(c->rows, c->k_strides[0], Hkv, c->k_strides[1], D) ||
      !rows_distinct(c->rows, c->v_strides[0], Hkv, c->v_strides[1], D))
    return "cache strides make two rows share memory";
  if (!aligned(c->k, es) || !aligned(c->v, es) || !aligned(c->seq_start, 8))
    return "cache buffers misaligned";
  return nullptr;
}

}  // namespace

static ra_status cuda_fail(cudaError_t e, const char *what) {
  return fail(RA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

extern "C" {

const char *ra_status_string(ra_status st) {
  switch (st) {
    case RA_OK: return "RA_OK";
    case RA_ERR_INVALID_ARG: return "RA_ERR_INVALID_ARG: invalid argument";
    case RA_ERR_UNSUPPORTED: return "RA_ERR_UNSUPPORTED: no kernel for this case";
    case RA_ERR_ALIGNMENT: return "RA_ERR_ALIGNMENT: misaligned pointer or stride";
    case RA_ERR_OVERLAP: return "RA_ERR_OVERLAP: output overlaps an input";
    case RA_ERR_CUDA: return "RA_ERR_CUDA: CUDA runtime error";
    case RA_ERR_DEVICE_TIMEOUT: return "RA_ERR_DEVICE_TIMEOUT: kernel barrier wait timed out";
    case RA_ERR_POSITION_RANGE: return "RA_ERR_POSITION_RANGE: position outside the cos/sin table";
    case RA_ERR_RANGE: return "RA_ERR_RANGE: a tensor-core operand is outside the fp16 range";
  }
  return "unknown ra_status";
}

const char *ra_last_error(void) { return g_last_error; }

const char *ra_last_launch(void) { return g_last_launch; }

ra_status rope_tables_build(float *cos_out, float *sin_out, int64_t rows, int rot_dim,
                            double base, int freq_dim, cudaStream_t s) {
  return rope_tables_build_scaled(cos_out, sin_out, rows, rot_dim, base, freq_dim, 1.0, s);
}

ra_status rope_tables_build_scaled(float *cos_out, float *sin_out, int64_t rows, int rot_dim,
                                   double base, int freq_dim, double pos_scale, cudaStream_t s) {
  if (!(pos_scale > 0.0) || !isfinite(pos_scale))
    return fail(RA_ERR_INVALID_ARG, "pos_scale must be finite and > 0");
  if (rows < 0) return fail(RA_ERR_INVALID_ARG, "rows must be >= 0 (got %lld)", (long long)rows);
  if (rot_dim < 2 || (rot_dim & 1))
    return fail(RA_ERR_INVALID_ARG, "rot_dim must be even and >= 2 (got %d)", rot_dim);
  if (!(base > 0.0) || !isfinite(base))
    return fail(RA_ERR_INVALID_ARG, "base must be finite and > 0");
  if (freq_dim < 0) return fail(RA_ERR_INVALID_ARG, "freq_dim must be >= 0");
  if (rows > 0 && (!cos_out || !sin_out)) return fail(RA_ERR_INVALID_ARG, "null table pointer");
  if (!aligned(cos_out, 4) || !aligned(sin_out, 4))
    return fail(RA_ERR_ALIGNMENT, "tables must be 4-byte aligned");
  if (rows == 0) return RA_OK;
  const ra::TableArgs a{cos_out, sin_out, rows, rot_dim, freq_dim, base, pos_scale};
  const cudaError_t e = ra::launch_table_build(a, s);
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "rope_tables_build launch");
}

ra_status rope_apply_qk(void *q, void *k, void *q_out, void *k_out, ra_dtype dt, int64_t T,
                        int Hq, int Hkv, int D, int rot_dim, ra_layout layout,
                        const int64_t strides_q[2], const int64_t strides_k[2],
                        const int64_t strides_qo[2], const int64_t strides_ko[2],
                        const void *positions, int pos_is_int64, const float *cos_t,
                        const float *sin_t, int64_t table_rows, cudaStream_t s) {
  if (!dtype_ok(dt)) return fail(RA_ERR_INVALID_ARG, "unknown dtype %d", (int)dt);
  if (!layout_ok(layout)) return fail(RA_ERR_INVALID_ARG, "unknown layout %d", (int)layout);
  if (T < 0 || Hq < 0 || Hkv < 0) return fail(RA_ERR_INVALID_ARG, "T, Hq, Hkv must be >= 0");
  if (D < 2 || (D & 1)) return fail(RA_ERR_INVALID_ARG, "D must be even and >= 2 (got %d)", D);
  if (rot_dim < 2 || (rot_dim & 1) || rot_dim > D)
    return fail(RA_ERR_INVALID_ARG, "rot_dim must be even with 2 <= rot_dim <= D (got %d)", rot_dim);
  if ((Hq > 0) != (q != nullptr) || (Hkv > 0) != (k != nullptr))
    return fail(RA_ERR_INVALID_ARG, "q (k) must be non-NULL exactly when Hq (Hkv) > 0");
  if (table_rows < 1) return fail(RA_ERR_INVALID_ARG, "table_rows must be >= 1");
  if (!positions || !cos_t || !sin_t)
    return fail(RA_ERR_INVALID_ARG, "positions and tables must be non-NULL");
  const bool qin = q_out == nullptr || q_out == q;
  const bool kin = k_out == nullptr || k_out == k;
  if ((Hq > 0 && !strides_q) || (Hkv > 0 && !strides_k) || (Hq > 0 && !qin && !strides_qo) ||
      (Hkv > 0 && !kin && !strides_ko))
    return fail(RA_ERR_INVALID_ARG, "stride arrays must be non-NULL for every tensor used");
  const int64_t zero2[2] = {0, 0};
  const int64_t *sq = Hq > 0 ? strides_q : zero2, *sk = Hkv > 0 ? strides_k : zero2;
  const int64_t *sqo = (Hq > 0 && !qin) ? strides_qo : sq;
  const int64_t *sko = (Hkv > 0 && !kin) ? strides_ko : sk;
  for (int j = 0; j < 2; ++j)
    if (sq[j] < 0 || sk[j] < 0 || sqo[j] < 0 || sko[j] < 0)
      return fail(RA_ERR_INVALID_ARG, "strides must be >= 0");
  if (T == 0 || Hq + Hkv == 0) return RA_OK;

  const size_t es = dtype_size(dt);
  // overlap rules: an output equals its input or shares no byte with any input/output
  if (Hq > 0 && Hkv > 0) {
    const Region rq = region(q, T, sq[0], Hq, sq[1], D, es);
    const Region rk = region(k, T, sk[0], Hkv, sk[1], D, es);
    const Region rqo = region(qin ? q : q_out, T, sqo[0], Hq, sqo[1], D, es);
    const Region rko = region(kin ? k : k_out, T, sko[0], Hkv, sko[1], D, es);
    if (!disjoint(rqo, rk) || !disjoint(rko, rq) || !disjoint(rqo, rko))
      return fail(RA_ERR_OVERLAP, "q/k outputs overlap the other tensor");
  }
  if (Hq > 0 && !qin &&
      !disjoint(region(q, T, sq[0], Hq, sq[1], D, es), region(q_out, T, sqo[0], Hq, sqo[1], D, es)))
    return fail(RA_ERR_OVERLAP, "q_out partially overlaps q");
  if (Hkv > 0 && !kin &&
      !disjoint(region(k, T, sk[0], Hkv, sk[1], D, es), region(k_out, T, sko[0], Hkv, sko[1], D, es)))
    return fail(RA_ERR_OVERLAP, "k_out partially overlaps k");

  if (!aligned(positions, pos_is_int64 ? 8 : 4) || !aligned(cos_t, 4) || !aligned(sin_t, 4))
    return fail(RA_ERR_ALIGNMENT, "positions/tables misaligned");
  const void *ptrs[4] = {q, k, qin ? q : q_out, kin ? k : k_out};
  for (const void *p : ptrs)
    if (p && !aligned(p, es)) return fail(RA_ERR_ALIGNMENT, "q/k buffers must be element-aligned");

  // vector path: 16-byte aligned pointers, strides, pair offsets and tail
  const int V = (int)(16 / es);
  const int half = rot_dim / 2;
  bool vec = aligned(cos_t, 16) && aligned(sin_t, 16);
  for (const void *p : ptrs) vec = vec && (!p || aligned(p, 16));
  for (int j = 0; j < 2; ++j)
    vec = vec && sq[j] % V == 0 && sk[j] % V == 0 && sqo[j] % V == 0 && sko[j] % V == 0;
  vec = vec && (layout == RA_NEOX ? half % V == 0 : rot_dim % V == 0);
  const bool copy_tail = !(qin && kin);
  if (copy_tail) vec = vec && (D - rot_dim) % V == 0;
  const int slices = (layout == RA_NEOX ? half / V : rot_dim / V) + (copy_tail ? (D - rot_dim) / V : 0);
  vec = vec && slices >= 1 && slices <= 1024;

  cudaError_t e;
  int *status = ra::device_status_ptr(&e);
  if (!status) return cuda_fail(e, "status word");
  ra::RopeArgs a{};
  a.q = q; a.k = k; a.q_out = q_out; a.k_out = k_out; a.dt = dt; a.T = T; a.Hq = Hq;
  a.Hkv = Hkv; a.D = D; a.rot_dim = rot_dim; a.layout = layout;
  for (int j = 0; j < 2; ++j) {
    a.sq[j] = sq[j]; a.sk[j] = sk[j]; a.sqo[j] = sqo[j]; a.sko[j] = sko[j];
  }
  a.positions = positions; a.pos_is_int64 = pos_is_int64 ? 1 : 0;
  a.cos_t = cos_t; a.sin_t = sin_t; a.table_rows = table_rows; a.status = status;
  e = ra::launch_rope_apply(a, vec, s);
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "rope_apply_qk launch");
}

ra_status attn_fwd_causal_rope(const void *q, const void *k, const void *v, void *o, float *lse,
                               ra_dtype dt, int B, int Hq, int Hkv, int64_t Sq, int64_t Sk,
                               int D, int64_t kv_offset, int apply_rope, int rot_dim,
                               ra_layout layout, const float *cos_t, const float *sin_t,
                               int64_t table_rows, float softmax_scale,
                               const int64_t strides_q[3], const int64_t strides_k[3],
                               const int64_t strides_v[3], const int64_t strides_o[3],
                               cudaStream_t s) {
  if (!dtype_ok(dt)) return fail(RA_ERR_INVALID_ARG, "unknown dtype %d", (int)dt);
  if (B < 1 || Hq < 1 || Hkv < 1) return fail(RA_ERR_INVALID_ARG, "B, Hq, Hkv must be >= 1");
  if (Hq % Hkv) return fail(RA_ERR_INVALID_ARG, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
  if (Sq < 0 || Sk < 1) return fail(RA_ERR_INVALID_ARG, "need Sq >= 0 and Sk >= 1");
  if (kv_offset < 0)
    return fail(RA_ERR_INVALID_ARG, "kv_offset must be >= 0: a negative offset leaves query rows "
                                    "with no admissible key");
  if (D < 2 || (D & 1)) return fail(RA_ERR_INVALID_ARG, "D must be even and >= 2");
  if (!q || !k || !v || !o) return fail(RA_ERR_INVALID_ARG, "q, k, v, o must be non-NULL");
  if (!strides_q || !strides_k || !strides_v || !strides_o)
    return fail(RA_ERR_INVALID_ARG, "stride arrays must be non-NULL");
  for (int j = 0; j < 3; ++j)
    if (strides_q[j] < 0 || strides_k[j] < 0 || strides_v[j] < 0 || strides_o[j] < 0)
      return fail(RA_ERR_INVALID_ARG, "strides must be >= 0");
  if (apply_rope) {
    if (!layout_ok(layout)) return fail(RA_ERR_INVALID_ARG, "unknown layout %d", (int)layout);
    if (rot_dim < 2 || (rot_dim & 1) || rot_dim > D)
      return fail(RA_ERR_INVALID_ARG, "rot_dim must be even with 2 <= rot_dim <= D");
    if (!cos_t || !sin_t) return fail(RA_ERR_INVALID_ARG, "tables must be non-NULL");
    const int64_t need = Sk > kv_offset + Sq ? Sk : kv_offset + Sq;
    if (table_rows < need)
      return fail(RA_ERR_INVALID_ARG, "table_rows %lld < needed %lld", (long long)table_rows,
                  (long long)need);
    if (!aligned(cos_t, 16) || !aligned(sin_t, 16))
      return fail(RA_ERR_ALIGNMENT, "tables must be 16-byte aligned");
  }
  if (!(softmax_scale <= 0.f) && !isfinite(softmax_scale))
    return fail(RA_ERR_INVALID_ARG, "softmax_scale must be finite");
  if (Sq == 0) return RA_OK;
  const size_t es = dtype_size(dt);
  if (!aligned(q, es) || !aligned(k, es) || !aligned(v, es) || !aligned(o, es) ||
      (lse && !aligned(lse, 4)))
    return fail(RA_ERR_ALIGNMENT, "buffers must be element-aligned");
  // the output must not overlap any input
  {
    const char *ob = static_cast<const char *>(o);
    const int64_t ospan = (((int64_t)B - 1) * strides_o[0] + ((int64_t)Hq - 1) * strides_o[1] +
                           (Sq - 1) * strides_o[2] + D) * (int64_t)es;
    const void *ins[3] = {q, k, v};
    const int64_t *sts[3] = {strides_q, strides_k, strides_v};
    const int64_t heads[3] = {Hq, Hkv, Hkv};
    const int64_t lens[3] = {Sq, Sk, Sk};
    for (int t = 0; t < 3; ++t) {
      const char *ib = static_cast<const char *>(ins[t]);
      const int64_t ispan = (((int64_t)B - 1) * sts[t][0] + (heads[t] - 1) * sts[t][1] +
                             (lens[t] - 1) * sts[t][2] + D) * (int64_t)es;
      if (!(ob + ospan <= ib || ib + ispan <= ob))
        return fail(RA_ERR_OVERLAP, "o overlaps an input");
    }
    if (lse) {
      const char *lb = reinterpret_cast<const char *>(lse);
      const int64_t lspan = (int64_t)B * Hq * Sq * 4;
      if (!(lb + lspan <= ob || ob + ospan <= lb)) return fail(RA_ERR_OVERLAP, "lse overlaps o");
    }
  }

  ra::AttnArgs a{};
  a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse; a.dt = dt;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.Sq = Sq; a.Sk = Sk; a.D = D; a.kv_offset = kv_offset;
  a.apply_rope = apply_rope ? 1 : 0;
  a.rot_dim = apply_rope ? rot_dim : D;
  a.layout = layout_ok(layout) ? layout : RA_NEOX;
  a.cos_t = cos_t; a.sin_t = sin_t; a.table_rows = table_rows;
  a.scale = softmax_scale > 0.f ? softmax_scale : (float)(1.0 / sqrt((double)D));
  for (int j = 0; j < 3; ++j) {
    a.sq[j] = strides_q[j]; a.sk[j] = strides_k[j]; a.sv[j] = strides_v[j]; a.so[j] = strides_o[j];
  }

  if (dt == RA_F32) {
    if (D > 256) return fail(RA_ERR_UNSUPPORTED, "fp32 attention supports D <= 256 (got %d)", D);
    cudaError_t e;
    a.status = ra::device_status_ptr(&e);
    if (!a.status) return cuda_fail(e, "status word");
    ra::clear_launches();
    e = ra::launch_attn_simt(a, s);
    if (e == cudaSuccess) ra::note_launch("attn_simt_kernel");
    return e == cudaSuccess ? RA_OK : cuda_fail(e, "attention (fp32) launch");
  }
  if (D != 64 && D != 128)
    return fail(RA_ERR_UNSUPPORTED, "tensor-core attention supports D in {64, 128} (got %d)", D);
  if (apply_rope && (layout == RA_NEOX ? (rot_dim / 2) % 8 : rot_dim % 8))
    return fail(RA_ERR_UNSUPPORTED, "tensor-core attention needs rot_dim/2 %% 8 == 0 (NeoX) or "
                                    "rot_dim %% 8 == 0 (GPT-J)");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
    return fail(RA_ERR_ALIGNMENT, "tensor-core attention needs 16-byte aligned q, k, v, o");
  for (int j = 0; j < 3; ++j)
    if (strides_q[j] % 8 || strides_k[j] % 8 || strides_v[j] % 8 || strides_o[j] % 8)
      return fail(RA_ERR_ALIGNMENT, "tensor-core attention needs strides that are multiples of 8");
  cudaError_t e;
  a.status = ra::device_status_ptr(&e);
  if (!a.status) return cuda_fail(e, "status word");
  ra::clear_launches();
  e = ra::launch_attn_tc(a, s);
  if (e == cudaSuccess) ra::note_launch("attn_tc_kernel");
  if (e == cudaErrorNotSupported) return fail(RA_ERR_UNSUPPORTED, "no tensor-core variant");
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "attention (tensor core) launch");
}

size_t attn_bwd_workspace_size(ra_dtype dt, int B, int Hq, int Hkv, int64_t Sq, int64_t Sk,
                               int D) {
  ra::BwdWorkspace w;
  if (!dtype_ok(dt) || !ra::plan_bwd_workspace(dt, B, Hq, Hkv, Sq, Sk, D, &w)) return (size_t)-1;
  return w.bytes;
}

ra_status attn_bwd_causal_rope(const void *q, const void *k, const void *v, const void *o,
                               const float *lse, const void *dout, void *dq, void *dk, void *dv,
                               ra_dtype dt, int B, int Hq, int Hkv, int64_t Sq, int64_t Sk, int D,
                               int64_t kv_offset, int apply_rope, int rot_dim, ra_layout layout,
                               const float *cos_t, const float *sin_t, int64_t table_rows,
                               float softmax_scale, const int64_t strides_q[3],
                               const int64_t strides_k[3], const int64_t strides_v[3],
                               const int64_t strides_o[3], const int64_t strides_do[3],
                               const int64_t strides_dq[3], const int64_t strides_dk[3],
                               const int64_t strides_dv[3], void *workspace,
                               size_t workspace_bytes, cudaStream_t s) {
  if (!dtype_ok(dt)) return fail(RA_ERR_INVALID_ARG, "unknown dtype %d", (int)dt);
  if (B < 1 || Hq < 1 || Hkv < 1) return fail(RA_ERR_INVALID_ARG, "B, Hq, Hkv must be >= 1");
  if (Hq % Hkv) return fail(RA_ERR_INVALID_ARG, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
  if (Sq < 0 || Sk < 1) return fail(RA_ERR_INVALID_ARG, "need Sq >= 0 and Sk >= 1");
  if (kv_offset < 0) return fail(RA_ERR_INVALID_ARG, "kv_offset must be >= 0");
  if (D < 2 || (D & 1)) return fail(RA_ERR_INVALID_ARG, "D must be even and >= 2");
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv)
    return fail(RA_ERR_INVALID_ARG, "tensors must be non-NULL");
  const int64_t *st[8] = {strides_q, strides_k, strides_v, strides_o,
                          strides_do, strides_dq, strides_dk, strides_dv};
  for (const int64_t *x : st) {
    if (!x) return fail(RA_ERR_INVALID_ARG, "stride arrays must be non-NULL");
    for (int j = 0; j < 3; ++j)
      if (x[j] < 0) return fail(RA_ERR_INVALID_ARG, "strides must be >= 0");
  }
  if (apply_rope) {
    if (!layout_ok(layout)) return fail(RA_ERR_INVALID_ARG, "unknown layout %d", (int)layout);
    if (rot_dim < 2 || (rot_dim & 1) || rot_dim > D)
      return fail(RA_ERR_INVALID_ARG, "rot_dim must be even with 2 <= rot_dim <= D");
    if (!cos_t || !sin_t) return fail(RA_ERR_INVALID_ARG, "tables must be non-NULL");
    const int64_t need = Sk > kv_offset + Sq ? Sk : kv_offset + Sq;
    if (table_rows < need)
      return fail(RA_ERR_INVALID_ARG, "table_rows %lld < needed %lld", (long long)table_rows,
                  (long long)need);
    if (!aligned(cos_t, 16) || !aligned(sin_t, 16))
      return fail(RA_ERR_ALIGNMENT, "tables must be 16-byte aligned");
  }
  if (!(softmax_scale <= 0.f) && !isfinite(softmax_scale))
    return fail(RA_ERR_INVALID_ARG, "softmax_scale must be finite");
  ra::BwdWorkspace wsp;
  ra::plan_bwd_workspace(dt, B, Hq, Hkv, Sq, Sk, D, &wsp);
  const size_t need_ws = wsp.bytes;
  if (need_ws > 0 && (!workspace || workspace_bytes < need_ws))
    return fail(RA_ERR_INVALID_ARG, "workspace of %zu bytes required", need_ws);
  if (workspace && !aligned(workspace, 256))
    return fail(RA_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  const size_t es = dtype_size(dt);
  const void *ptrs[8] = {q, k, v, o, dout, dq, dk, dv};
  for (const void *x : ptrs)
    if (!aligned(x, es)) return fail(RA_ERR_ALIGNMENT, "buffers must be element-aligned");
  if (!aligned(lse, 4)) return fail(RA_ERR_ALIGNMENT, "lse must be 4-byte aligned");
  // outputs dq, dk, dv and the workspace must not overlap any input or each other
  {
    const int64_t lens[8] = {Sq, Sk, Sk, Sq, Sq, Sq, Sk, Sk};
    const int64_t heads[8] = {Hq, Hkv, Hkv, Hq, Hq, Hq, Hkv, Hkv};
    int64_t span[8];
    for (int t = 0; t < 8; ++t)
      span[t] = lens[t] > 0 ? span4(B, st[t][0], heads[t], st[t][1], lens[t], st[t][2], D, es) : 0;
    const void *all[10] = {q, k, v, o, dout, lse, dq, dk, dv, workspace};
    const int64_t n[10] = {span[0], span[1], span[2], span[3], span[4], (int64_t)B * Hq * Sq * 4,
                           span[5], span[6], span[7], workspace ? (int64_t)need_ws : 0};
    for (int w = 6; w < 10; ++w) {
      if (!all[w] || n[w] == 0) continue;
      for (int r = 0; r < 10; ++r)
        if (r != w && all[r] && n[r] > 0 && !spans_apart(all[w], n[w], all[r], n[r]))
          return fail(RA_ERR_OVERLAP, "gradient outputs and workspace must not overlap "
                                      "anything else");
    }
  }
  if (dt != RA_F32) {
    if (D != 64 && D != 128)
      return fail(RA_ERR_UNSUPPORTED, "tensor-core backward supports D in {64, 128} (got %d)", D);
    if (apply_rope && (layout == RA_NEOX ? (rot_dim / 2) % 8 : rot_dim % 8))
      return fail(RA_ERR_UNSUPPORTED, "tensor-core backward needs rot_dim/2 %% 8 == 0 (NeoX) "
                                      "or rot_dim %% 8 == 0 (GPT-J)");
    for (const void *x : ptrs)
      if (!aligned(x, 16)) return fail(RA_ERR_ALIGNMENT, "tensor-core backward needs 16-byte "
                                                         "aligned tensors");
    for (const int64_t *x : st)
      for (int j = 0; j < 3; ++j)
        if (x[j] % 8) return fail(RA_ERR_ALIGNMENT, "tensor-core backward needs strides that "
                                                    "are multiples of 8");
  } else if (D > 256) {
    return fail(RA_ERR_UNSUPPORTED, "fp32 backward supports D <= 256 (got %d)", D);
  }
  // keys no query can see still get (zero) gradients, so even Sq == 0 launches
  ra::BwdArgs a{};
  ra::AttnArgs &f = a.f;
  f.q = q; f.k = k; f.v = v; f.dt = dt;
  f.B = B; f.Hq = Hq; f.Hkv = Hkv; f.Sq = Sq; f.Sk = Sk; f.D = D; f.kv_offset = kv_offset;
  f.apply_rope = apply_rope ? 1 : 0;
  f.rot_dim = apply_rope ? rot_dim : D;
  f.layout = layout_ok(layout) ? layout : RA_NEOX;
  f.cos_t = cos_t; f.sin_t = sin_t; f.table_rows = table_rows;
  f.scale = softmax_scale > 0.f ? softmax_scale : (float)(1.0 / sqrt((double)D));
  for (int j = 0; j < 3; ++j) {
    f.sq[j] = strides_q[j]; f.sk[j] = strides_k[j]; f.sv[j] = strides_v[j];
    a.sod[j] = strides_o[j]; a.sdo[j] = strides_do[j]; a.sdq[j] = strides_dq[j];
    a.sdk[j] = strides_dk[j]; a.sdv[j] = strides_dv[j];
  }
  a.o = o; a.dout = dout; a.lse = lse; a.dq = dq; a.dk = dk; a.dv = dv;
  a.dsum = static_cast<float *>(workspace);
  a.qrot = wsp.qrot_off ? static_cast<char *>(workspace) + wsp.qrot_off : nullptr;
  a.krot = wsp.krot_off ? static_cast<char *>(workspace) + wsp.krot_off : nullptr;
  cudaError_t e;
  f.status = ra::device_status_ptr(&e);
  if (!f.status) return cuda_fail(e, "status word");
  ra::clear_launches();
  if (Sq > 0) {
    e = ra::launch_bwd_rowterm(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "backward row-term launch");
  }
  e = dt == RA_F32 ? ra::launch_attn_bwd_simt(a, s) : ra::launch_attn_bwd_tc(a, s);
  if (e == cudaErrorNotSupported) return fail(RA_ERR_UNSUPPORTED, "no backward kernel for the case");
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "backward launch");
}

ra_status rope_append_kv(void *q, void *q_out, const void *k_new, const void *v_new,
                         const ra_kv_cache *cache, ra_dtype dt, int64_t T, int Hq, int Hkv, int D,
                         int rot_dim, ra_layout layout, const int64_t strides_q[2],
                         const int64_t strides_qo[2], const int64_t strides_kn[2],
                         const int64_t strides_vn[2], const int32_t *seq_ids,
                         const void *positions, int pos_is_int64, const float *cos_t,
                         const float *sin_t, int64_t table_rows, cudaStream_t s) {
  if (!dtype_ok(dt)) return fail(RA_ERR_INVALID_ARG, "unknown dtype %d", (int)dt);
  if (!layout_ok(layout)) return fail(RA_ERR_INVALID_ARG, "unknown layout %d", (int)layout);
  if (T < 0 || Hq < 0 || Hkv < 1) return fail(RA_ERR_INVALID_ARG, "need T >= 0, Hq >= 0, Hkv >= 1");
  if (D < 2 || (D & 1)) return fail(RA_ERR_INVALID_ARG, "D must be even and >= 2 (got %d)", D);
  if (rot_dim < 2 || (rot_dim & 1) || rot_dim > D)
    return fail(RA_ERR_INVALID_ARG, "rot_dim must be even with 2 <= rot_dim <= D (got %d)", rot_dim);
  if ((Hq > 0) != (q != nullptr)) return fail(RA_ERR_INVALID_ARG, "q must be non-NULL exactly when Hq > 0");
  if (!k_new || !v_new) return fail(RA_ERR_INVALID_ARG, "k_new and v_new must be non-NULL");
  const size_t es = dtype_size(dt);
  if (const char *why = cache_problem(cache, Hkv, D, es)) return fail(RA_ERR_INVALID_ARG, "%s", why);
  if (table_rows < 1) return fail(RA_ERR_INVALID_ARG, "table_rows must be >= 1");
  if (!positions || !cos_t || !sin_t)
    return fail(RA_ERR_INVALID_ARG, "positions and tables must be non-NULL");
  const bool qin = q_out == nullptr || q_out == q;
  if (!strides_kn || !strides_vn || (Hq > 0 && !strides_q) || (Hq > 0 && !qin && !strides_qo))
    return fail(RA_ERR_INVALID_ARG, "stride arrays must be non-NULL for every tensor used");
  const int64_t zero2[2] = {0, 0};
  const int64_t *sq = Hq > 0 ? strides_q : zero2;
  const int64_t *sqo = (Hq > 0 && !qin) ? strides_qo : sq;
  for (int j = 0; j < 2; ++j)
    if (sq[j] < 0 || sqo[j] < 0 || strides_kn[j] < 0 || strides_vn[j] < 0)
      return fail(RA_ERR_INVALID_ARG, "strides must be >= 0");
  if (T == 0) return RA_OK;

  // overlap: the written regions (q_out or q, cache K, cache V) share no byte
  // with each other or with the inputs; q_out may equal q
  const Region rkn = region(k_new, T, strides_kn[0], Hkv, strides_kn[1], D, es);
  const Region rvn = region(v_new, T, strides_vn[0], Hkv, strides_vn[1], D, es);
  const Region rkc = region(cache->k, cache->rows, cache->k_strides[0], Hkv, cache->k_strides[1], D, es);
  const Region rvc = region(cache->v, cache->rows, cache->v_strides[0], Hkv, cache->v_strides[1], D, es);
  if (!disjoint(rkc, rvc)) return fail(RA_ERR_OVERLAP, "cache K and V rows overlap");
  for (const Region *r : {&rkn, &rvn})
    if (!disjoint(rkc, *r) || !disjoint(rvc, *r))
      return fail(RA_ERR_OVERLAP, "the cache overlaps k_new or v_new");
  if (Hq > 0) {
    const Region rq = region(q, T, sq[0], Hq, sq[1], D, es);
    const Region rqo = region(qin ? q : q_out, T, sqo[0], Hq, sqo[1], D, es);
    for (const Region *w : {&rq, &rqo})
      for (const Region *r : {&rkn, &rvn, &rkc, &rvc})
        if (!disjoint(*w, *r)) return fail(RA_ERR_OVERLAP, "q or q_out overlaps k, v or the cache");
    if (!qin && !disjoint(rq, rqo)) return fail(RA_ERR_OVERLAP, "q_out partially overlaps q");
  }

  if (!aligned(positions, pos_is_int64 ? 8 : 4) || !aligned(cos_t, 4) || !aligned(sin_t, 4) ||
      (seq_ids && !aligned(seq_ids, 4)))
    return fail(RA_ERR_ALIGNMENT, "positions, seq_ids or tables misaligned");
  const void *ptrs[6] = {q, qin ? q : q_out, k_new, v_new, cache->k, cache->v};
  for (const void *p : ptrs)
    if (p && !aligned(p, es)) return fail(RA_ERR_ALIGNMENT, "buffers must be element-aligned");

  // vector path: 16-byte aligned pointers and strides, whole 16-byte slices
  const int V = (int)(16 / es);
  const int half = rot_dim / 2;
  bool vec = aligned(cos_t, 16) && aligned(sin_t, 16);
  for (const void *p : ptrs) vec = vec && (!p || aligned(p, 16));
  for (int j = 0; j < 2; ++j)
    vec = vec && sq[j] % V == 0 && sqo[j] % V == 0 && strides_kn[j] % V == 0 &&
          strides_vn[j] % V == 0 && cache->k_strides[j] % V == 0 && cache->v_strides[j] % V == 0;
  vec = vec && (layout == RA_NEOX ? half % V == 0 : rot_dim % V == 0) && (D - rot_dim) % V == 0;

  cudaError_t e;
  int *status = ra::device_status_ptr(&e);
  if (!status) return cuda_fail(e, "status word");
  ra::AppendArgs a{};
  a.q = q; a.q_out = q_out; a.k_new = k_new; a.v_new = v_new; a.cache = *cache; a.dt = dt;
  a.T = T; a.Hq = Hq; a.Hkv = Hkv; a.D = D; a.rot_dim = rot_dim; a.layout = layout;
  for (int j = 0; j < 2; ++j) {
    a.sq[j] = sq[j]; a.sqo[j] = sqo[j]; a.skn[j] = strides_kn[j]; a.svn[j] = strides_vn[j];
  }
  a.seq_ids = seq_ids; a.positions = positions; a.pos_is_int64 = pos_is_int64 ? 1 : 0;
  a.cos_t = cos_t; a.sin_t = sin_t; a.table_rows = table_rows; a.status = status;
  ra::clear_launches();
  e = ra::launch_rope_append(a, vec, s);
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "rope_append_kv launch");
}

size_t attn_decode_workspace_size(ra_dtype dt, int B, int Hq, int Hkv, int Sq, int D,
                                  int64_t max_kv_len) {
  ra::DecodePlan plan;
  if (!dtype_ok(dt) || !ra::plan_decode(dt, B, Hq, Hkv, Sq, D, max_kv_len, &plan))
    return (size_t)-1;
  return plan.ws_bytes;
}

ra_status attn_decode(const void *q, void *o, float *lse, const ra_kv_cache *cache, ra_dtype dt,
                      int B, int Hq, int Hkv, int Sq, int D, const int32_t *seq_ids,
                      const int32_t *kv_len, int64_t max_kv_len, float softmax_scale,
                      const int64_t strides_q[3], const int64_t strides_o[3], void *workspace,
                      size_t workspace_bytes, cudaStream_t s) {
  if (!dtype_ok(dt)) return fail(RA_ERR_INVALID_ARG, "unknown dtype %d", (int)dt);
  if (B < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv)
    return fail(RA_ERR_INVALID_ARG, "need B >= 0, Hq and Hkv >= 1, Hq a multiple of Hkv");
  if (Sq < 1) return fail(RA_ERR_INVALID_ARG, "Sq must be >= 1");
  if (D < 2 || (D & 1) || D > 256)
    return fail(RA_ERR_INVALID_ARG, "D must be even with 2 <= D <= 256 (got %d)", D);
  if (max_kv_len < Sq) return fail(RA_ERR_INVALID_ARG, "max_kv_len must be >= Sq");
  if (!(softmax_scale <= 0.f) && !isfinite(softmax_scale))
    return fail(RA_ERR_INVALID_ARG, "softmax_scale must be finite");
  if (!q || !o || !kv_len) return fail(RA_ERR_INVALID_ARG, "q, o and kv_len must be non-NULL");
  if (!strides_q || !strides_o) return fail(RA_ERR_INVALID_ARG, "stride arrays must be non-NULL");
  for (int j = 0; j < 3; ++j)
    if (strides_q[j] < 0 || strides_o[j] < 0) return fail(RA_ERR_INVALID_ARG, "strides must be >= 0");
  const size_t es = dtype_size(dt);
  if (const char *why = cache_problem(cache, Hkv, D, es)) return fail(RA_ERR_INVALID_ARG, "%s", why);
  ra::DecodePlan plan;
  if (!ra::plan_decode(dt, B, Hq, Hkv, Sq, D, max_kv_len, &plan))
    return fail(RA_ERR_INVALID_ARG, "sizes out of range for the split plan");
  if (plan.ws_bytes > 0) {
    if (!workspace) return fail(RA_ERR_INVALID_ARG, "workspace required (%zu bytes)", plan.ws_bytes);
    if (workspace_bytes < plan.ws_bytes)
      return fail(RA_ERR_INVALID_ARG, "workspace of %zu bytes < %zu required", workspace_bytes,
                  plan.ws_bytes);
    if (!aligned(workspace, 256)) return fail(RA_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  }
  if (B == 0) return RA_OK;
  if (!aligned(q, es) || !aligned(o, es) || (lse && !aligned(lse, 4)) || !aligned(kv_len, 4) ||
      (seq_ids && !aligned(seq_ids, 4)))
    return fail(RA_ERR_ALIGNMENT, "buffers must be element-aligned");
  // written: o, lse, workspace; read: q, cache K and V
  {
    const int64_t qspan = span4(B, strides_q[0], Hq, strides_q[1], Sq, strides_q[2], D, es);
    const int64_t ospan = span4(B, strides_o[0], Hq, strides_o[1], Sq, strides_o[2], D, es);
    const int64_t kspan = span4(cache->rows, cache->k_strides[0], Hkv, cache->k_strides[1], 1, 0, D, es);
    const int64_t vspan = span4(cache->rows, cache->v_strides[0], Hkv, cache->v_strides[1], 1, 0, D, es);
    const int64_t lspan = (int64_t)B * Hq * Sq * 4;
    const int64_t wspan = (int64_t)plan.ws_bytes;
    struct { const void *p; int64_t n; } rd[3] = {{q, qspan}, {cache->k, kspan}, {cache->v, vspan}};
    struct { const void *p; int64_t n; } wr[3] = {{o, ospan}, {lse, lse ? lspan : 0},
                                                  {workspace, workspace ? wspan : 0}};
    for (int w = 0; w < 3; ++w) {
      if (!wr[w].p || wr[w].n == 0) continue;
      for (int r = 0; r < 3; ++r)
        if (!spans_apart(wr[w].p, wr[w].n, rd[r].p, rd[r].n))
          return fail(RA_ERR_OVERLAP, "an output or the workspace overlaps q or the cache");
      for (int w2 = w + 1; w2 < 3; ++w2)
        if (wr[w2].p && wr[w2].n && !spans_apart(wr[w].p, wr[w].n, wr[w2].p, wr[w2].n))
          return fail(RA_ERR_OVERLAP, "o, lse and the workspace must not overlap");
    }
  }
  // the tensor-core kernel loads K and V with TMA and Q / stores O in 16-byte pieces
  if (plan.tc) {
    bool ok = aligned(cache->k, 16) && aligned(cache->v, 16) && aligned(q, 16) && aligned(o, 16);
    for (int j = 0; j < 2; ++j) ok = ok && cache->k_strides[j] % 8 == 0 && cache->v_strides[j] % 8 == 0;
    for (int j = 0; j < 3; ++j) ok = ok && strides_q[j] % 8 == 0 && strides_o[j] % 8 == 0;
    plan.tc = ok;  // same split plan on the CUDA-core kernel otherwise
  }

  cudaError_t e;
  ra::DecodeArgs a{};
  a.status = ra::device_status_ptr(&e);
  if (!a.status) return cuda_fail(e, "status word");
  a.q = q; a.o = o; a.lse = lse; a.cache = *cache; a.dt = dt;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.Sq = Sq; a.D = D;
  a.seq_ids = seq_ids; a.kv_len = kv_len; a.max_kv_len = max_kv_len;
  a.scale = softmax_scale > 0.f ? softmax_scale : (float)(1.0 / sqrt((double)D));
  for (int j = 0; j < 3; ++j) {
    a.sq[j] = strides_q[j]; a.so[j] = strides_o[j];
  }
  a.workspace = workspace; a.plan = plan;
  ra::clear_launches();
  e = ra::launch_attn_decode(a, s);
  if (e == cudaErrorNotSupported) return fail(RA_ERR_UNSUPPORTED, "no decode kernel for the case");
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "attn_decode launch");
}

ra_status attn_decode_noalloc(const void *q, void *o, float *lse, const ra_kv_cache *cache,
                              ra_dtype dt, int B, int Hq, int Hkv, int Sq, int D,
                              const int32_t *seq_ids, const int32_t *kv_len, int64_t max_kv_len,
                              float softmax_scale, const int64_t strides_q[3],
                              const int64_t strides_o[3], cudaStream_t s) {
  if (!dtype_ok(dt)) return fail(RA_ERR_INVALID_ARG, "unknown dtype %d", (int)dt);
  ra::DecodePlan plan;
  if (!ra::plan_decode(dt, B, Hq, Hkv, Sq, D, max_kv_len, &plan))
    return fail(RA_ERR_INVALID_ARG, "sizes out of range for the split plan");
  if (plan.ws_bytes > (size_t)RA_DECODE_STATIC_SCRATCH_BYTES)
    return fail(RA_ERR_UNSUPPORTED, "needs %zu bytes of split workspace, more than the %u-byte "
                "static region", plan.ws_bytes, (unsigned)RA_DECODE_STATIC_SCRATCH_BYTES);
  void *ws = nullptr;
  if (plan.ws_bytes > 0) {
    cudaError_t e;
    ws = ra::decode_scratch_ptr(&e);
    if (!ws) return cuda_fail(e, "static decode workspace");
  }
  return attn_decode(q, o, lse, cache, dt, B, Hq, Hkv, Sq, D, seq_ids, kv_len, max_kv_len,
                     softmax_scale, strides_q, strides_o, ws, plan.ws_bytes, s);
}

ra_status ra_get_device_status(cudaStream_t s) {
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_ra_status_word, sizeof v);
  if (e != cudaSuccess) return cuda_fail(e, "read status word");
  const int zero = 0;
  e = cudaMemcpyToSymbol(g_ra_status_word, &zero, sizeof zero);
  if (e != cudaSuccess) return cuda_fail(e, "clear status word");
  if (v == 0) return RA_OK;
  return fail((ra_status)v, "device reported %s", ra_status_string((ra_status)v));
}

}  // extern "C"

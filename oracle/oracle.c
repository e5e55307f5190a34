/*
 * oracle.c -- plain fp64 CPU reference for rotary position embedding (RoPE)
 * and causal softmax attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path loads this file or
 * the library built from it: only the test-suite, the package smoke check and
 * the benchmark's CPU-baseline leg do.  It shares no code, header, table or
 * constant with the CUDA library; the two meet only through seeded inputs.
 *
 * Every routine is the plain definition written out, in double precision,
 * with libm's cos/sin/exp/log/pow.  There is no tiling, fusion or reordering
 * beyond what the definitions state.  Inputs given as float are exact upcasts
 * of the bf16/fp16/fp32 tensors under test.
 *
 * Sources (page title, section):
 *  [RF]  "RoPE and FlashAttention: relative positions and online softmax",
 *        section 1 (rotation of each 2-D pair by position * theta_i,
 *        theta_i = base^(-2i/d)), section 2 (the interleaved rope() routine
 *        and its absolute-position angles), section 4 (S = QK^T/sqrt(d),
 *        P = softmax(S), O = PV), section 5 (max m, denominator l, weighted
 *        numerator u; output u/l), and the offset-causal mask j <= off + i
 *        used by its tiled-attention test.
 *  [TR]  "Write Triton Rope Kernel", Required reasoning process steps 1 and 6
 *        (NeoX halves: lo*c - hi*s, hi*c + lo*s; GPT-J pairs (2i, 2i+1)),
 *        Kernel design rules (partial RoPE rotates the first rot_dim dims,
 *        the tail is untouched), Correctness requirements (table built with
 *        theta_i = base^(-2i/D), angle = position * theta_i).
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared oracle.c -lm -lpthread
 * (-ffp-contract=off keeps x86 and aarch64 results bit-identical).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_NEOX = 0, ORACLE_GPTJ = 1 };

/* ---------------------------------------------------------------- threads */

typedef void (*item_fn)(void *ctx, int64_t item, double *scratch);

typedef struct {
  item_fn fn;
  void *ctx;
  int64_t n_items;
  int64_t next; /* shared work counter */
  size_t scratch_doubles;
} pool_t;

static void *pool_worker(void *arg) {
  pool_t *p = (pool_t *)arg;
  double *scratch = NULL;
  if (p->scratch_doubles) scratch = (double *)malloc(p->scratch_doubles * sizeof(double));
  for (;;) {
    int64_t it = __atomic_fetch_add(&p->next, 1, __ATOMIC_RELAXED);
    if (it >= p->n_items) break;
    p->fn(p->ctx, it, scratch);
  }
  free(scratch);
  return NULL;
}

/* Runs fn(ctx, i, scratch) for every i in [0, n_items) on nthreads threads. */
static void run_items(item_fn fn, void *ctx, int64_t n_items, int nthreads,
                      size_t scratch_doubles) {
  pool_t p = {fn, ctx, n_items, 0, scratch_doubles};
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 512) nthreads = 512;
  if ((int64_t)nthreads > n_items) nthreads = (int)(n_items > 0 ? n_items : 1);
  pthread_t tid[512];
  int started = 0;
  for (int t = 1; t < nthreads; ++t)
    if (pthread_create(&tid[started], NULL, pool_worker, &p) == 0) ++started;
  pool_worker(&p);
  for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
}

/* ------------------------------------------------------------------- RoPE */

/* theta_i = base^(-2i/F) for i in [0, rot_dim/2); F = freq_dim, or rot_dim
 * when freq_dim <= 0.  [RF] section 1; [TR] Correctness requirements. */
void oracle_rope_freqs(int rot_dim, int freq_dim, double base, double *theta) {
  const int F = freq_dim > 0 ? freq_dim : rot_dim;
  for (int i = 0; i < rot_dim / 2; ++i) theta[i] = pow(base, -(2.0 * i) / (double)F);
}

/* cos/sin of p * theta_i for p in [0, rows): two [rows, rot_dim/2] arrays.
 * [TR] Inputs to gather (table shape [max_seq_len, D/2]) and Correctness
 * requirements (angle = position * theta_i). */
void oracle_rope_tables(int64_t rows, int rot_dim, int freq_dim, double base,
                        double *cos_out, double *sin_out) {
  const int half = rot_dim / 2;
  double *theta = (double *)malloc((size_t)(half > 0 ? half : 1) * sizeof(double));
  oracle_rope_freqs(rot_dim, freq_dim, base, theta);
  for (int64_t p = 0; p < rows; ++p)
    for (int i = 0; i < half; ++i) {
      const double a = (double)p * theta[i];
      cos_out[p * half + i] = cos(a);
      sin_out[p * half + i] = sin(a);
    }
  free(theta);
}

/* Position-interpolated tables: cos/sin of (p / pos_scale) * theta_i, i.e.
 * positions divided by an extension factor before the angle is formed
 * ("RoPE and FlashAttention ...", section 3, Position Interpolation).  With
 * pos_scale = 1 this is oracle_rope_tables. */
void oracle_rope_tables_scaled(int64_t rows, int rot_dim, int freq_dim, double base,
                               double pos_scale, double *cos_out, double *sin_out) {
  const int half = rot_dim / 2;
  double *theta = (double *)malloc((size_t)(half > 0 ? half : 1) * sizeof(double));
  oracle_rope_freqs(rot_dim, freq_dim, base, theta);
  for (int64_t p = 0; p < rows; ++p)
    for (int i = 0; i < half; ++i) {
      const double a = ((double)p / pos_scale) * theta[i];
      cos_out[p * half + i] = cos(a);
      sin_out[p * half + i] = sin(a);
    }
  free(theta);
}

/* Rotates one row x[0..D) at integer position p into y (y may equal x).
 * NeoX pairs (i, i + rot_dim/2), GPT-J pairs (2i, 2i+1), i < rot_dim/2;
 * dims [rot_dim, D) are copied unchanged.  [TR] steps 1, 5, 6, 8. */
static void rope_row(const double *x, double *y, int D, int rot_dim, int layout,
                     const double *theta, int64_t p) {
  const int half = rot_dim / 2;
  for (int d = rot_dim; d < D; ++d) y[d] = x[d];
  for (int i = 0; i < half; ++i) {
    const double a = (double)p * theta[i];
    const double c = cos(a), s = sin(a);
    const int lo = layout == ORACLE_NEOX ? i : 2 * i;
    const int hi = layout == ORACLE_NEOX ? i + half : 2 * i + 1;
    const double xl = x[lo], xh = x[hi];
    y[lo] = xl * c - xh * s;
    y[hi] = xh * c + xl * s;
  }
}

/* Rotates n_rows rows of length D (row r at x + r*D) at positions[r]. */
int oracle_rope_rows(const double *x, int64_t n_rows, int D, const int64_t *positions,
                     int rot_dim, int freq_dim, double base, int layout, double *y) {
  if (D <= 0 || rot_dim < 2 || rot_dim > D || (rot_dim & 1) || (D & 1) || !(base > 0.0))
    return -1;
  if (layout != ORACLE_NEOX && layout != ORACLE_GPTJ) return -1;
  double *theta = (double *)malloc((size_t)(rot_dim / 2) * sizeof(double));
  oracle_rope_freqs(rot_dim, freq_dim, base, theta);
  for (int64_t r = 0; r < n_rows; ++r)
    rope_row(x + r * D, y + r * D, D, rot_dim, layout, theta, positions[r]);
  free(theta);
  return 0;
}

/* -------------------------------------------------------------- attention */

typedef struct {
  const float *q, *v;
  const double *kr; /* rotated (or plain) K, fp64, [B, Hkv, Sk, D] */
  int B, Hq, Hkv, D, apply_rope, rot_dim, layout;
  int64_t Sq, Sk, kv_offset;
  double scale;
  const double *theta;
  const int64_t *rows;
  double *o_out, *lse_out;
} attn_ctx;

typedef struct {
  const float *k;
  double *kr;
  int D, apply_rope, rot_dim, layout;
  int64_t Sk;
  const double *theta;
} krot_ctx;

/* K row j of every (b, kv-head) is rotated at absolute position j.  [RF] 2. */
static void krot_item(void *vctx, int64_t item, double *scratch) {
  (void)scratch;
  krot_ctx *c = (krot_ctx *)vctx;
  const int64_t j = item % c->Sk;
  const float *src = c->k + item * c->D;
  double *dst = c->kr + item * c->D;
  for (int d = 0; d < c->D; ++d) dst[d] = (double)src[d];
  if (c->apply_rope) rope_row(dst, dst, c->D, c->rot_dim, c->layout, c->theta, j);
}

/* One output row (b, h, i): query at absolute position kv_offset + i attends
 * to keys j with j <= kv_offset + i and j < Sk ([RF] section 5's offset-causal
 * mask); two-pass softmax: m = max_j s_ij, l = sum_j exp(s_ij - m),
 * O = sum_j exp(s_ij - m) V_j / l, LSE = m + ln l.  q-head h reads kv-head
 * h / (Hq / Hkv). */
static void attn_item(void *vctx, int64_t item, double *s) {
  attn_ctx *c = (attn_ctx *)vctx;
  const int D = c->D;
  const int64_t r = c->rows[item];
  const int64_t i = r % c->Sq;
  const int64_t bh = r / c->Sq;
  const int h = (int)(bh % c->Hq), b = (int)(bh / c->Hq);
  const int hk = h / (c->Hq / c->Hkv);
  double *qr = s + c->Sk; /* scratch: Sk scores, then D query values */
  const float *qsrc = c->q + r * D;
  for (int d = 0; d < D; ++d) qr[d] = (double)qsrc[d];
  if (c->apply_rope) rope_row(qr, qr, D, c->rot_dim, c->layout, c->theta, c->kv_offset + i);
  int64_t jend = c->kv_offset + i + 1;
  if (jend > c->Sk) jend = c->Sk;
  const double *kb = c->kr + ((int64_t)b * c->Hkv + hk) * c->Sk * D;
  const float *vb = c->v + ((int64_t)b * c->Hkv + hk) * c->Sk * D;
  double m = -INFINITY;
  for (int64_t j = 0; j < jend; ++j) {
    const double *kj = kb + j * D;
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += qr[d] * kj[d];
    s[j] = c->scale * acc;
    if (s[j] > m) m = s[j];
  }
  double *o = c->o_out + item * D;
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  double l = 0.0;
  for (int64_t j = 0; j < jend; ++j) {
    const double p = exp(s[j] - m);
    l += p;
    const float *vj = vb + j * D;
    for (int d = 0; d < D; ++d) o[d] += p * (double)vj[d];
  }
  for (int d = 0; d < D; ++d) o[d] /= l;
  c->lse_out[item] = m + log(l);
}

/* Causal attention with optional RoPE on Q and K, for the selected flat rows
 * r = (b*Hq + h)*Sq + i.  q: [B,Hq,Sq,D], k and v: [B,Hkv,Sk,D], contiguous
 * float.  Outputs o_out [n_rows, D] and lse_out [n_rows] in fp64.
 * Returns 0, or -1 on invalid arguments (including any query row that would
 * have no admissible key, which the method leaves undefined). */
int oracle_attention(const float *q, const float *k, const float *v, int B, int Hq, int Hkv,
                     int64_t Sq, int64_t Sk, int D, int64_t kv_offset, int apply_rope,
                     int rot_dim, int freq_dim, double base, int layout, double scale,
                     const int64_t *rows, int64_t n_rows, double *o_out, double *lse_out,
                     int nthreads) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || Sq < 0 || Sk < 1 || D < 1) return -1;
  if (kv_offset < 0) return -1; /* row 0 would see no key */
  if (apply_rope) {
    if ((D & 1) || rot_dim < 2 || rot_dim > D || (rot_dim & 1) || !(base > 0.0)) return -1;
    if (layout != ORACLE_NEOX && layout != ORACLE_GPTJ) return -1;
  }
  for (int64_t t = 0; t < n_rows; ++t)
    if (rows[t] < 0 || rows[t] >= (int64_t)B * Hq * Sq) return -1;
  double *theta = NULL;
  if (apply_rope) {
    theta = (double *)malloc((size_t)(rot_dim / 2) * sizeof(double));
    oracle_rope_freqs(rot_dim, freq_dim, base, theta);
  }
  const int64_t nk = (int64_t)B * Hkv * Sk;
  double *kr = (double *)malloc((size_t)nk * D * sizeof(double));
  if (!kr) {
    free(theta);
    return -2;
  }
  krot_ctx kc = {k, kr, D, apply_rope, rot_dim, layout, Sk, theta};
  run_items(krot_item, &kc, nk, nthreads, 0);
  attn_ctx ac = {q, v, kr, B, Hq, Hkv, D, apply_rope, rot_dim, layout, Sq, Sk, kv_offset,
                 scale, theta, rows, o_out, lse_out};
  run_items(attn_item, &ac, n_rows, nthreads, (size_t)Sk + (size_t)D);
  free(kr);
  free(theta);
  return 0;
}

/*
 * rope_attn.h -- C ABI of librope_attn.so: rotary position embedding (RoPE)
 * and causal attention with RoPE fused in, for NVIDIA GB300 (sm_103a).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers named *device* must point to memory the current CUDA device can
 *   read/write (cudaMalloc, PyTorch CUDA tensors).  Pointers named *host*
 *   are ordinary host memory.  The caller owns every buffer; no entry point
 *   allocates or frees memory.
 * - Work is enqueued on the stream `s` (0 = legacy default stream) of the
 *   current device and runs asynchronously; entry points return as soon as
 *   the kernels are launched.
 * - Errors are returned as ra_status codes, never thrown.  Every argument
 *   check happens on the host before any launch or device memory access, so
 *   a rejected call has no side effect.  ra_last_error() gives a readable
 *   reason.
 * - Errors found by a kernel while it runs (a position outside the table, a
 *   value outside the fp16 range of the tensor-core operands) are recorded
 *   in a per-device status word that ra_get_device_status() reads and
 *   clears.
 * - Element strides are counted in elements, not bytes; the innermost
 *   (head-dimension) stride is always 1.
 *
 * Sources (page title, section) for what each call computes:
 *  [RF] "RoPE and FlashAttention: relative positions and online softmax":
 *       1 (pair rotation, theta_i = base^(-2i/d)), 2 (absolute positions,
 *       decoder cache convention), 3 (context extension: position
 *       interpolation, larger base), 4 (S = QK^T/sqrt(d), P = softmax(S),
 *       O = PV), 5 (online softmax with running max / denominator /
 *       numerator; offset-causal mask j <= off + i).
 *  [TR] "Write Triton Rope Kernel": layouts (NeoX halves vs GPT-J pairs),
 *       fp32 cos/sin tables [max_seq_len, D/2], per-token positions[],
 *       partial rot_dim, H_q != H_kv, in-place vs out-of-place, one launch
 *       for Q and K.
 *  [PM] "RoPE + PoPE Attention Kernels" (pope-memory-optimal README): rotate
 *       inside the attention kernel instead of materialising rotated Q/K.
 */
#ifndef ROPE_ATTN_H
#define ROPE_ATTN_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RA_OK = 0,
  RA_ERR_INVALID_ARG = -1,     /* a size, pointer or parameter is out of range        */
  RA_ERR_UNSUPPORTED = -2,     /* valid, but this build has no kernel for the case   */
  RA_ERR_ALIGNMENT = -3,       /* pointer or stride misaligned for the requested path */
  RA_ERR_OVERLAP = -4,         /* an output partially overlaps an input               */
  RA_ERR_CUDA = -5,            /* a CUDA runtime call failed (see ra_last_error)      */
  RA_ERR_DEVICE_TIMEOUT = -6,  /* a kernel gave up waiting on an internal barrier     */
  RA_ERR_POSITION_RANGE = -7,  /* a kernel met a position outside [0, table_rows)     */
  RA_ERR_RANGE = -8            /* a tensor-core operand left the fp16 range (results
                                  of that call are not valid)                          */
} ra_status;

typedef enum { RA_NEOX = 0, RA_GPTJ = 1 } ra_layout;
typedef enum { RA_F32 = 0, RA_BF16 = 1, RA_F16 = 2 } ra_dtype;

/*
 * rope_tables_build -- fill the fp32 cos/sin tables.
 *   Defines: theta_i = base^(-2i/F), i in [0, rot_dim/2), F = freq_dim, or
 *   rot_dim when freq_dim <= 0 ([RF] 1; [TR] Correctness requirements);
 *   cos_out[p][i] = cos(p * theta_i), sin_out[p][i] = sin(p * theta_i) for
 *   p in [0, rows).  The angle and both functions are evaluated in fp64 and
 *   rounded once to fp32 ([TR]: tables built in fp32 or better; [RF] 2:
 *   keep the angle policy explicit at long positions).
 *   cos_out, sin_out: device, each [rows][rot_dim/2] fp32, row stride
 *     rot_dim/2 elements, written entirely.
 *   rows >= 0, rot_dim even and >= 2, base > 0.
 */
ra_status rope_tables_build(float *cos_out, float *sin_out, int64_t rows, int rot_dim,
                            double base, int freq_dim, cudaStream_t s);

/*
 * rope_tables_build_scaled -- tables for position interpolation: like
 *   rope_tables_build with angle (p / pos_scale) * theta_i, i.e. positions
 *   divided by an extension factor before the angle is formed ([RF] 3,
 *   Position Interpolation).  pos_scale = 1 gives rope_tables_build's tables
 *   bit for bit; NTK-style scaling needs no new call (it is a larger `base`,
 *   whose value belongs to the checkpoint).  pos_scale must be finite and > 0.
 */
ra_status rope_tables_build_scaled(float *cos_out, float *sin_out, int64_t rows, int rot_dim,
                                   double base, int freq_dim, double pos_scale, cudaStream_t s);

/*
 * rope_apply_qk -- rotate Q and K of a packed token batch in one launch
 * ([TR] Required reasoning process, Kernel design rules; [RF] 2).
 *   Token t of every head is rotated at position positions[t] (never the
 *   token index).  Only the first rot_dim dims of each head are rotated:
 *     layout RA_NEOX: pairs (i, i + rot_dim/2);  RA_GPTJ: pairs (2i, 2i+1);
 *     lo' = lo*cos - hi*sin,  hi' = hi*cos + lo*sin,  i < rot_dim/2,
 *   with cos/sin read from table row positions[t] (row stride rot_dim/2).
 *   Arithmetic is fp32; results are rounded to dt (round to nearest even).
 *   Dims [rot_dim, D) are left untouched in place and copied out of place.
 *   V is never passed here.
 *   q: device [T][Hq][D] of dt, element strides strides_q = {token, head}.
 *   k: device [T][Hkv][D] of dt, strides strides_k.  q may be NULL iff
 *     Hq == 0, k may be NULL iff Hkv == 0.
 *   q_out, k_out: NULL or equal to q / k for in place (strides ignored);
 *     otherwise distinct device buffers with strides strides_qo / strides_ko
 *     that must not overlap any input or the other output (RA_ERR_OVERLAP).
 *   positions: device [T], int32 (pos_is_int64 = 0) or int64.
 *   cos_t, sin_t: device tables from rope_tables_build with the same
 *     rot_dim and table_rows rows.  A position outside [0, table_rows)
 *     leaves that token's outputs unwritten and records
 *     RA_ERR_POSITION_RANGE in the device status word.
 *   T >= 0 (T == 0: nothing launched), D even, 2 <= rot_dim <= D, rot_dim
 *   even.  Aligned vector access is used when every pointer is 16-byte
 *   aligned and every stride and offset is a multiple of 16 bytes; other
 *   cases take a scalar kernel.
 */
ra_status rope_apply_qk(void *q, void *k, void *q_out, void *k_out, ra_dtype dt, int64_t T,
                        int Hq, int Hkv, int D, int rot_dim, ra_layout layout,
                        const int64_t strides_q[2], const int64_t strides_k[2],
                        const int64_t strides_qo[2], const int64_t strides_ko[2],
                        const void *positions, int pos_is_int64, const float *cos_t,
                        const float *sin_t, int64_t table_rows, cudaStream_t s);

/*
 * attn_fwd_causal_rope -- causal softmax attention forward with RoPE applied
 * to Q and K inside the kernel ([PM]; [RF] 1, 4, 5).
 *   Query row i of (b, h) sits at absolute position kv_offset + i; key row j
 *   sits at position j.  With apply_rope != 0 both are rotated as in
 *   rope_apply_qk (same layout, rot_dim, tables) before the product; no
 *   rotated tensor is written to memory.  V is never rotated.
 *     s_ij = softmax_scale * <q~_i, k~_j>  for j <= kv_offset + i and j < Sk,
 *     O_i  = sum_j exp(s_ij - m_i) V_j / l_i,  l_i = sum_j exp(s_ij - m_i),
 *     LSE_i = m_i + ln(l_i)  (natural log, scale included).
 *   q-head h reads kv-head h / (Hq / Hkv) (grouped-query attention).
 *   q: device [B][Hq][Sq][D], strides strides_q = {b, h, s};
 *   k, v: device [B][Hkv][Sk][D], strides strides_k / strides_v;
 *   o: device [B][Hq][Sq][D] of dt, strides strides_o;
 *   lse: device fp32 [B][Hq][Sq] contiguous, or NULL (not written).
 *   dt RA_F32 runs an fp32 CUDA-core kernel (D <= 256).  RA_BF16 / RA_F16 run
 *   the tensor-core kernel (tcgen05): D in {64, 128}; every pointer 16-byte
 *   aligned and every stride a multiple of 8 elements; rotated Q/K enter the
 *   product as fp16, P and V as dt, accumulation fp32.
 *   fp16 range ([TR] Correctness requirements: precision of the rotated
 *   values): every rotated Q/K element must round to a finite fp16 value,
 *   |x| < 65520 (|x| <= 65504 after rounding).  A rotation |x~| <= |lo| + |hi|
 *   of its pair, so inputs with |x| <= 32752 always fit.  Otherwise the
 *   kernel records RA_ERR_RANGE in the device status word and O / LSE are
 *   not valid.  Every query row is checked; a key row is checked in the key
 *   tiles some query visits (rows that no query can see never enter a
 *   product).  Scores are exponentiated in fp32, each as one fused
 *   multiply-add of the score and the running row maximum in log2 units,
 *   so the exponent carries a rounding of about |m| 2^-24: scores up to
 *   ~1e4 in magnitude (after softmax_scale) keep the stated accuracy, and
 *   at ~1e9 and beyond the exponent can overflow and O / LSE become NaN.
 *   kv_offset >= 0 (so every row sees key 0; a negative offset would leave
 *   rows without keys and is rejected), Sk >= 1, Sq >= 0 (0: no launch).
 *   With apply_rope: 2 <= rot_dim <= D, even, and table_rows >=
 *   max(Sk, kv_offset + Sq).  softmax_scale <= 0 selects 1/sqrt(D).
 */
ra_status attn_fwd_causal_rope(const void *q, const void *k, const void *v, void *o, float *lse,
                               ra_dtype dt, int B, int Hq, int Hkv, int64_t Sq, int64_t Sk,
                               int D, int64_t kv_offset, int apply_rope, int rot_dim,
                               ra_layout layout, const float *cos_t, const float *sin_t,
                               int64_t table_rows, float softmax_scale,
                               const int64_t strides_q[3], const int64_t strides_k[3],
                               const int64_t strides_v[3], const int64_t strides_o[3],
                               cudaStream_t s);

/*
 * attn_bwd_workspace_size -- bytes of device workspace attn_bwd_causal_rope
 * needs: the fp32 row terms D_i = <dO_i, O_i> ([B][Hq][Sq]) and, for
 * bf16/fp16, fp16 copies of the rotated Q ([B][Hq][Sq][D]) and K
 * ([B][Hkv][Sk][D]) that the tensor-core kernels load tile by tile; -1 cast
 * to size_t for invalid sizes.
 */
size_t attn_bwd_workspace_size(ra_dtype dt, int B, int Hq, int Hkv, int64_t Sq, int64_t Sk,
                               int D);

/*
 * attn_bwd_causal_rope -- gradients of attn_fwd_causal_rope with respect to
 * the raw (unrotated) q, k and v ([RF] 5: the probabilities are rebuilt from
 * Q, K and the forward's LSE instead of being stored; [RF] 1-2 for the
 * rotation).  With q~, k~, s, P, O as in attn_fwd_causal_rope and dO the
 * gradient of the loss with respect to O:
 *     dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),  D_i = <dO_i, O_i>,
 *     dq~ = scale dS k~,  dk~ = scale dS^T q~,
 *     dq_i = R(kv_offset + i)^T dq~_i,  dk_j = R(j)^T dk~_j
 * (R^T: the rotation by the negated angle; dims past rot_dim unrotated); a
 * kv head's dk, dv sum over the q-heads of its group.  Keys no query sees
 * get zero gradients.
 *   q, k, v, layout, rot_dim, tables, kv_offset, softmax_scale: exactly as
 *   given to the forward call; o: its output; lse: its fp32 LSE [B][Hq][Sq]
 *   (contiguous); dout: like o.  dq like q, dk like k, dv like v, each with
 *   its own strides {b, h, s}; written entirely (not accumulated), dtype dt.
 *   workspace: device, 256-byte aligned, >= attn_bwd_workspace_size bytes,
 *   contents ignored and clobbered.
 *   dt RA_F32 runs CUDA-core kernels (D <= 256); RA_BF16 / RA_F16 run the
 *   tensor-core kernels (D in {64, 128}; 16-byte aligned tensors, strides
 *   multiples of 8 elements): rotated Q/K and dS enter the products as fp16,
 *   P, V and dO as dt, accumulation fp32.  Outputs may not overlap any input
 *   or each other (RA_ERR_OVERLAP).
 *   fp16 range: a rotated Q/K element that does not round to a finite fp16
 *   value, or a dS = P o (dP - D) term beyond it (|dP - D| grows with
 *   |dO| |V|), makes the call record RA_ERR_RANGE in the device status word
 *   (checked on the rotated copies and on the dQ~ / dK~ / dV accumulators,
 *   which a non-finite dS term always reaches); dq, dk, dv are then not
 *   valid.
 */
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
                               size_t workspace_bytes, cudaStream_t s);

/*
 * Decoder KV cache ([RF] 2: new K is appended rotated, V unrotated, and cached
 * K is never rotated again).  Row r of head h of the K cache starts at element
 * k[r * k_strides[0] + h * k_strides[1]] (D contiguous elements; likewise V),
 * r in [0, rows).  Cache sequence s owns the rows from seq_start[s] on: the
 * key at position j of sequence s lives in row seq_start[s] + j.  Token-major
 * ([rows][Hkv][D]), head-major ([Hkv][rows][D]) and interleaved K/V layouts
 * are all expressible.  The caller owns every buffer and keeps each
 * sequence's rows inside its own region.
 *   k, v: device, dt.  seq_start: device int64 [n_seqs].
 */
typedef struct {
  void *k;
  void *v;
  int64_t k_strides[2]; /* {row, head}, elements */
  int64_t v_strides[2];
  int64_t rows;
  const int64_t *seq_start;
  int64_t n_seqs;
} ra_kv_cache;

/*
 * rope_append_kv -- the decoder step of [RF] 2 in one launch: rotate the new
 * tokens' Q, rotate their K into the cache, copy their V into the cache.
 *   Token t belongs to cache sequence s = seq_ids[t] (seq_ids NULL: s = t)
 *   and sits at absolute position p = positions[t] (int32 or int64), its
 *   cache row being seq_start[s] + p.  With Q, K rotated as in rope_apply_qk
 *   (layout, rot_dim, tables):
 *     q_out[t][h]                = rot(q[t][h], p)    h < Hq (in place if q_out is NULL or q)
 *     cache.k[seq_start[s] + p][h] = rot(k_new[t][h], p)  all D dims (tail copied)
 *     cache.v[seq_start[s] + p][h] = v_new[t][h]          h < Hkv
 *   q [T][Hq][D], k_new / v_new [T][Hkv][D]: device, dt, strides {token,
 *   head} in strides_q / strides_kn / strides_vn (q_out: strides_qo).  Hq may
 *   be 0 (q NULL: cache append only).
 *   A token whose s is outside [0, n_seqs), whose p is outside [0, table_rows)
 *   or whose row is outside [0, cache.rows) is skipped (nothing of it is
 *   written) and RA_ERR_POSITION_RANGE is recorded in the status word.
 *   Rejected on the host: cache rows overlapping each other or an input
 *   (RA_ERR_OVERLAP), q_out partly overlapping q.  Two tokens writing one
 *   cache row is the caller's error (the result is one of them).
 */
ra_status rope_append_kv(void *q, void *q_out, const void *k_new, const void *v_new,
                         const ra_kv_cache *cache, ra_dtype dt, int64_t T, int Hq, int Hkv, int D,
                         int rot_dim, ra_layout layout, const int64_t strides_q[2],
                         const int64_t strides_qo[2], const int64_t strides_kn[2],
                         const int64_t strides_vn[2], const int32_t *seq_ids,
                         const void *positions, int pos_is_int64, const float *cos_t,
                         const float *sin_t, int64_t table_rows, cudaStream_t s);

/*
 * attn_decode_workspace_size -- bytes of device workspace attn_decode needs
 * for these sizes on the current device (0: none).  Deterministic for fixed
 * arguments and device; -1 cast to size_t for invalid sizes.
 */
size_t attn_decode_workspace_size(ra_dtype dt, int B, int Hq, int Hkv, int Sq, int D,
                                  int64_t max_kv_len);

/*
 * attn_decode -- causal attention of Sq new queries per sequence over a KV
 * cache that already holds rotated K ([RF] 2, 4, 5; the offset mask of [RF]
 * 5).  Q must already be rotated (rope_append_kv); nothing is rotated here.
 *   Batch entry b reads cache sequence s = seq_ids[b] (NULL: s = b) with
 *   L = kv_len[b] keys at positions 0..L-1 (device int32 [B]); its query i
 *   sits at position L - Sq + i and sees keys j <= L - Sq + i:
 *     s_ij = softmax_scale * <q_i, k_j>, O_i = sum_j softmax(s_i)_j v_j,
 *     LSE_i = m_i + ln(l_i) (natural log, scale included).
 *   q-head h reads kv-head h / (Hq / Hkv).
 *   q, o: device [B][Hq][Sq][D] of dt, strides {b, h, s} (token-major decode
 *   batches are {Sq*Hq*D, D, Hq*D}); lse: device fp32 [B][Hq][Sq] or NULL.
 *   The keys are split into chunks processed in parallel and merged by their
 *   log-sum-exp (split-KV); the partial results live in `workspace` (device,
 *   256-byte aligned, >= attn_decode_workspace_size bytes, contents ignored
 *   on entry and clobbered).  Calls sharing a workspace must be ordered on
 *   one stream.
 *   max_kv_len >= max_b kv_len[b] (host value; it sizes the split).  An entry
 *   with L < Sq, L > max_kv_len, s outside [0, n_seqs) or rows outside the
 *   cache leaves its outputs unwritten and records RA_ERR_POSITION_RANGE.
 *   bf16/fp16 with D = 128 and (Hq/Hkv)*Sq <= 64 run on the tensor cores
 *   (tcgen05; K, V loaded by TMA: cache pointers 16-byte aligned, strides
 *   multiples of 8 elements); every other case (fp32, D <= 256 even) runs a
 *   CUDA-core kernel.  softmax_scale <= 0 selects 1/sqrt(D).
 */
ra_status attn_decode(const void *q, void *o, float *lse, const ra_kv_cache *cache, ra_dtype dt,
                      int B, int Hq, int Hkv, int Sq, int D, const int32_t *seq_ids,
                      const int32_t *kv_len, int64_t max_kv_len, float softmax_scale,
                      const int64_t strides_q[3], const int64_t strides_o[3], void *workspace,
                      size_t workspace_bytes, cudaStream_t s);

/*
 * attn_decode_noalloc -- attn_decode with its split workspace in a fixed
 * region of device memory inside the library instead of a caller buffer;
 * the call itself allocates nothing (no cudaMalloc, no library allocator).
 * The pages have no counterpart.  It serves callers that cannot hand out
 * scratch memory: a serving loop whose device memory budget is fixed when
 * it starts, a host framework that owns every device allocation, or a path
 * where a cudaMalloc (which may synchronise the device) is not acceptable.
 *   Same arguments, results and errors as attn_decode without the workspace
 *   pair.  The region holds RA_DECODE_STATIC_SCRATCH_BYTES on every device
 *   that loads the library, for the life of the process.  Sizes whose
 *   attn_decode_workspace_size exceeds it return RA_ERR_UNSUPPORTED before
 *   any launch or device memory access; the split plan, and so whether a
 *   shape fits, depends on the device's SM count as well as on the sizes.
 *   Nothing in the region has to start at zero: each call writes every
 *   partial result it reads, so what an earlier call left there is never
 *   used.
 *   The region's device address is looked up (cudaGetSymbolAddress) by the
 *   first call on each device, with that device current.  One region per
 *   device: calls that may overlap in time on the GPU (different streams,
 *   or work queued concurrently) race on it and give wrong results; order
 *   them on one stream.
 */
#define RA_DECODE_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)
ra_status attn_decode_noalloc(const void *q, void *o, float *lse, const ra_kv_cache *cache,
                              ra_dtype dt, int B, int Hq, int Hkv, int Sq, int D,
                              const int32_t *seq_ids, const int32_t *kv_len, int64_t max_kv_len,
                              float softmax_scale, const int64_t strides_q[3],
                              const int64_t strides_o[3], cudaStream_t s);

/*
 * ra_get_device_status -- synchronise stream s, then read and clear the
 * current device's status word.  Returns RA_OK, the first error a kernel
 * recorded since the last call, or RA_ERR_CUDA if the stream reported an
 * asynchronous CUDA error.
 */
ra_status ra_get_device_status(cudaStream_t s);

/* Static English name of a status code (never NULL). */
const char *ra_status_string(ra_status st);

/* Reason for the last non-OK status returned on this host thread (never NULL). */
const char *ra_last_error(void);

/*
 * Kernels launched by the last successful call of attn_fwd_causal_rope,
 * attn_bwd_causal_rope, rope_append_kv or attn_decode on this host thread, space-separated (e.g.
 * "attn_decode_tc_kernel attn_decode_merge_kernel"); "" before any.  A
 * dispatch aid (which variant ran); never NULL.  No counterpart on the pages.
 */
const char *ra_last_launch(void);

#ifdef __cplusplus
}
#endif
#endif /* ROPE_ATTN_H */

// Internal declarations shared by the translation units of librope_attn.so.
// Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/rope_attn.h"

namespace ra {

// Status word of the current device (a __device__ int in api.cu).  Kernels
// record the first error with atomicCAS(status, 0, code).
int *device_status_ptr(cudaError_t *err);

// Records a readable reason for the current host thread and returns st.
ra_status fail(ra_status st, const char *fmt, ...);

// Launch record read by ra_last_launch(): cleared at the start of a call,
// one kernel name appended per launch.
void clear_launches();
void note_launch(const char *kernel);

struct TableArgs {
  float *cos_out, *sin_out;
  int64_t rows;
  int rot_dim, freq_dim;
  double base;
  double pos_scale;  // angle = (p / pos_scale) * theta_i
};

struct RopeArgs {
  void *q, *k, *q_out, *k_out;
  ra_dtype dt;
  int64_t T;
  int Hq, Hkv, D, rot_dim;
  ra_layout layout;
  int64_t sq[2], sk[2], sqo[2], sko[2];
  const void *positions;
  int pos_is_int64;
  const float *cos_t, *sin_t;
  int64_t table_rows;
  int *status;
};

struct AttnArgs {
  const void *q, *k, *v;
  void *o;
  float *lse;
  ra_dtype dt;
  int B, Hq, Hkv;
  int64_t Sq, Sk;
  int D;
  int64_t kv_offset;
  int apply_rope, rot_dim;
  ra_layout layout;
  const float *cos_t, *sin_t;
  int64_t table_rows;
  float scale;
  int64_t sq[3], sk[3], sv[3], so[3];
  int *status;
};

struct AppendArgs {
  void *q, *q_out;
  const void *k_new, *v_new;
  ra_kv_cache cache;
  ra_dtype dt;
  int64_t T;
  int Hq, Hkv, D, rot_dim;
  ra_layout layout;
  int64_t sq[2], sqo[2], skn[2], svn[2];
  const int32_t *seq_ids;
  const void *positions;
  int pos_is_int64;
  const float *cos_t, *sin_t;
  int64_t table_rows;
  int *status;
};

// Split-KV plan of one decode call: keys of a sequence are cut into `splits`
// chunks of `chunk` keys (a multiple of 128); splits == 1 writes O directly.
struct DecodePlan {
  bool tc;          // tensor-core kernel (else CUDA cores)
  int splits;
  int64_t chunk;
  size_t ws_bytes;  // 0 when splits == 1
  size_t ws_lse_offset;
};
// Returns false for invalid sizes.
bool plan_decode(ra_dtype dt, int B, int Hq, int Hkv, int Sq, int D, int64_t max_kv_len,
                 DecodePlan *plan);

struct DecodeArgs {
  const void *q;
  void *o;
  float *lse;
  ra_kv_cache cache;
  ra_dtype dt;
  int B, Hq, Hkv, Sq, D;
  const int32_t *seq_ids, *kv_len;
  int64_t max_kv_len;
  float scale;
  int64_t sq[3], so[3];
  void *workspace;
  DecodePlan plan;
  int *status;
};

struct BwdArgs {
  AttnArgs f;  // q, k, v, sizes, rope, scale, strides of the forward call
  const void *o, *dout;
  const float *lse;
  void *dq, *dk, *dv;
  int64_t sod[3], sdo[3], sdq[3], sdk[3], sdv[3];
  float *dsum;  // workspace: fp32 [B][Hq][Sq]
  void *qrot, *krot;  // workspace (16-bit inputs): rotated fp16 Q [B][Hq][Sq][D], K [B][Hkv][Sk][D]
};
// Workspace layout of attn_bwd_causal_rope: byte offsets of the rotated Q
// and K copies (0 when unused) and the total size.
struct BwdWorkspace {
  size_t qrot_off, krot_off, bytes;
};
bool plan_bwd_workspace(ra_dtype dt, int B, int Hq, int Hkv, int64_t Sq, int64_t Sk, int D,
                        BwdWorkspace *w);

cudaError_t launch_table_build(const TableArgs &a, cudaStream_t s);
// D_i = <dO_i, O_i> into a.dsum (any dtype).
cudaError_t launch_bwd_rowterm(const BwdArgs &a, cudaStream_t s);
cudaError_t launch_attn_bwd_simt(const BwdArgs &a, cudaStream_t s);
cudaError_t launch_attn_bwd_tc(const BwdArgs &a, cudaStream_t s);
cudaError_t launch_rope_append(const AppendArgs &a, bool vectorized, cudaStream_t s);
// Runs the split kernel (tensor-core or CUDA-core, as planned) and the merge.
cudaError_t launch_attn_decode(const DecodeArgs &a, cudaStream_t s);
// Tensor-core split kernel only (decode_tc.cu); cudaErrorNotSupported when it
// has no variant for the case.
cudaError_t launch_attn_decode_tc(const DecodeArgs &a, cudaStream_t s);
int sm_count_current();

// One-time set-up (kernel attributes) per device: a function attribute
// belongs to the device that was current when it was set, so a process that
// drives several GPUs sets it on each.  run() returns the set-up's result.
class PerDeviceOnce {
 public:
  template <typename F>
  cudaError_t run(F &&f) {
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return f();
    std::lock_guard<std::mutex> lock(mutex_);
    if (!done_[dev]) {
      result_[dev] = f();
      done_[dev] = true;
    }
    return result_[dev];
  }

 private:
  static constexpr int kMaxDevices = 64;
  std::mutex mutex_;
  bool done_[kMaxDevices] = {};
  cudaError_t result_[kMaxDevices] = {};
};

// A 16-bit tensor (bf16 or fp16) whose rows of D elements are contiguous,
// addressed by n_outer (1..3) further coordinates with the given sizes and
// element strides; coordinate 0 is the row.  The tiled tensor map sorts them
// by increasing stride (size-1 dims last) into map dims 1..n_outer, writes
// perm[map dim - 1] = coordinate, and uses a box of 64 elements x 128 rows
// (1 along the other dims) with the 128-byte swizzle; rows past the end read
// as zero.  cudaErrorNotSupported without the driver's encoder.
cudaError_t make_row_tile_map(const void *base, bool bf16, int D, int n_outer,
                              const int64_t size[3], const int64_t stride[3], CUtensorMap *map,
                              int perm[3]);
cudaError_t launch_rope_apply(const RopeArgs &a, bool vectorized, cudaStream_t s);
cudaError_t launch_attn_simt(const AttnArgs &a, cudaStream_t s);
// Returns cudaErrorNotSupported when the tensor-core kernel has no variant
// for the case (the caller maps it to RA_ERR_UNSUPPORTED).
cudaError_t launch_attn_tc(const AttnArgs &a, cudaStream_t s);

}  // namespace ra

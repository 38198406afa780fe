// Internal launch interfaces between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "topt.h"

namespace topt {

// ------------------------------------------------------------------ decode
size_t decode_workspace_bytes(const topt_decode_args& a);
long decode_max_pairs();
int decode_max_cache();
cudaError_t decode_launch(const topt_decode_args& a, cudaStream_t s);
size_t decode_noalloc_capacity();
cudaError_t decode_noalloc_launch(const topt_decode_args& a, cudaStream_t s);

// ----------------------------------------------------------------- prefill
size_t prefill_workspace_bytes(const topt_prefill_args& a);
void prefill_tile_shape(const topt_prefill_args& a, int32_t* rows, int32_t* keys);
// withhold_k: test hook of topt_prefill_test_timeout (tensor-core path only)
cudaError_t prefill_launch(const topt_prefill_args& a, cudaStream_t s, int withhold_k = 0);
// tensor-core path (bf16): 128-row blocks; v16 is the fp16 copy of V
// (prefill_tc_v16_bytes), vmax/vexp one word per (batch, kv head), bsum the
// column sums of 128-row blocks of V (prefill_tc_bsum_bytes; VMC only).
// prefill_tc.cu runs the preparation and the pre-softmax kernel (64-key
// tiles); post-softmax thresholds launch the kernel of prefill_tc_post.cu
// (128-key tiles) on the prepared buffers.
size_t prefill_tc_v16_bytes(const topt_prefill_args& a);
size_t prefill_tc_bsum_bytes(const topt_prefill_args& a);
int prefill_tc_rows();
int prefill_tc_keys(int mode);
cudaError_t prefill_tc_run(const topt_prefill_args& a, void* v16, uint32_t* vmax, int32_t* vexp,
                           float* bsum, cudaStream_t s, int withhold_k);
int prefill_tc_post_keys();
cudaError_t prefill_tc_post_launch(const topt_prefill_args& a, void* v16, const int32_t* vexp,
                                   const float* bsum, cudaStream_t s, int withhold_k);

// --------------------------------------------------------------- calibrate
size_t calibrate_workspace_bytes(const topt_calib_args& a, size_t rows_per_pass);
size_t calibrate_min_rows_per_pass();
cudaError_t calibrate_launch(const topt_calib_args& a, cudaStream_t s);
// offline-calibrated SDC estimate E~, calibrated beside a pre-softmax theta
size_t calibrate_sdc_workspace_bytes(const topt_sdc_calib_args& a, size_t rows_per_pass);
cudaError_t calibrate_sdc_launch(const topt_sdc_calib_args& a, cudaStream_t s);
// multi-k cumulative calibration: fixed workspace + one head's scores per head
size_t calibrate_multik_fixed_bytes(const topt_mkc_args& a);
size_t calibrate_multik_head_bytes(const topt_mkc_args& a);
int calibrate_multik_max_samples();
cudaError_t calibrate_multik_launch(const topt_mkc_args& a, cudaStream_t s);
// Calibration scores of bf16 rows on the tensor cores (calib_tc.cu): rows
// [it0, it0 + nrows) of the flattened (seq, head h0 .. h0+Hp-1, row) index of
// q [N][Hq][R][D] against keys [N][Hkv][Nk][D]; row it, key j < row_len[i]
// goes to ws[(it - it0) * Nk + j] (times `scale`).  _ok: the shape and
// pointers suit the kernel (16-byte aligned q and keys, d = 64 or 128).
struct CalibScoreArgs {
  const void* q;
  const void* keys;
  const int32_t* row_len;
  int N, Hq, Hkv, R, Nk, D, h0, Hp;
  float scale;
  long it0;
  int nrows;
  float* ws;
  int32_t* status;
};
bool calib_scores_tc_ok(const CalibScoreArgs& a);
cudaError_t calib_scores_tc(const CalibScoreArgs& a, cudaStream_t s);
cudaError_t select_kth_launch(const float* x, int32_t rows, int32_t stride,
                              const int32_t* row_len, int32_t k, float* out,
                              int32_t* status, cudaStream_t s);

// ------------------------------------------------------------------- vmean
cudaError_t vmean_launch(const topt_vmean_args& a, cudaStream_t s);

}  // namespace topt

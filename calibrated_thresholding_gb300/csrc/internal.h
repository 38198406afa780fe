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
// tensor-core path (bf16): 128-row x 128-key tiles; v16 is the fp16 copy of V
// (prefill_tc_v16_bytes), vmax/vexp one word per (batch, kv head), bsum the
// column sums of 128-row blocks of V (prefill_tc_bsum_bytes; VMC only).
size_t prefill_tc_v16_bytes(const topt_prefill_args& a);
size_t prefill_tc_bsum_bytes(const topt_prefill_args& a);
int prefill_tc_rows();
int prefill_tc_keys();
cudaError_t prefill_tc_run(const topt_prefill_args& a, void* v16, uint32_t* vmax, int32_t* vexp,
                           float* bsum, cudaStream_t s, int withhold_k);

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
cudaError_t select_kth_launch(const float* x, int32_t rows, int32_t stride,
                              const int32_t* row_len, int32_t k, float* out,
                              int32_t* status, cudaStream_t s);

// ------------------------------------------------------------------- vmean
cudaError_t vmean_launch(const topt_vmean_args& a, cudaStream_t s);

}  // namespace topt

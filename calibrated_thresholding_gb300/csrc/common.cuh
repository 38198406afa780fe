// Shared device helpers of libtopt (CUDA, sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "topt.h"

namespace topt {

constexpr int kWarp = 32;

// Round a byte count up to 256 so every workspace sub-buffer stays aligned.
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Records the caller's profiling event `ev` (a cudaEvent_t, or NULL) on s;
// under stream capture as an external event node.
inline cudaError_t record_event(void* ev, cudaStream_t s) {
  if (!ev) return cudaSuccess;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cs);
  if (e != cudaSuccess) return e;
  return cs == cudaStreamCaptureStatusActive
             ? cudaEventRecordWithFlags(static_cast<cudaEvent_t>(ev), s, cudaEventRecordExternal)
             : cudaEventRecord(static_cast<cudaEvent_t>(ev), s);
}

__device__ __forceinline__ void set_status(int32_t* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------- loads --
// 16-byte streaming load: not kept in L1, evicted first from L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint4 ld_stream16(const void* p, uint64_t pol) {
  uint4 r;
  asm volatile(
      "ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p), "l"(pol));
  return r;
}

__device__ __forceinline__ uint4 ld_nc16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void st_hint_f32(float* p, float v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(pol) : "memory");
}

__device__ __forceinline__ float ld_hint_f32(const float* p, uint64_t pol) {
  float v;
  asm volatile("ld.global.L2::cache_hint.f32 %0, [%1], %2;" : "=f"(v) : "l"(p), "l"(pol));
  return v;
}

// ------------------------------------------------------------- bf16 math --
// A 32-bit word holds two bf16: element 2i in the low half, 2i+1 in the high.
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

// D = A(16x16, row) * B(16x8, col) + D with bf16 inputs and fp32 accumulation.
__device__ __forceinline__ void mma_16816_bf16(float c[4], const uint32_t a[4], const uint32_t b[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// ------------------------------------------------------ softmax partials --
// (m, z) represents sum_j exp(a_j - m) = z.  m = -inf means "empty".
struct MaxSum {
  float m, z;
};

__device__ __forceinline__ void ms_merge(float& m, float& z, float m2, float z2) {
  if (m2 == -CUDART_INF_F) return;
  if (m == -CUDART_INF_F) {
    m = m2;
    z = z2;
    return;
  }
  float mn = fmaxf(m, m2);
  z = z * __expf(m - mn) + z2 * __expf(m2 - mn);
  m = mn;
}

__device__ __forceinline__ void ms_warp_merge(float& m, float& z, int lane_mask_start = 1) {
#pragma unroll
  for (int off = lane_mask_start; off < kWarp; off <<= 1) {
    float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    float z2 = __shfl_xor_sync(0xffffffffu, z, off);
    ms_merge(m, z, m2, z2);
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}
__device__ __forceinline__ int warp_sum_int(int v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// --------------------------------------------------- threshold on scores --
// Keep iff x >= theta.  Pre-softmax x = a.  Post-softmax x = exp(a - m) / Z,
// and s >= theta  <=>  a >= m + ln(theta) + ln(Z)  for theta > 0; theta <= 0
// keeps every valid key.  Returns the bound on a.
__device__ __forceinline__ float score_bound(int mode, float theta, float m, float z) {
  if (mode == TOPT_PRE) return theta;
  if (!(theta > 0.f)) return -CUDART_INF_F;
  return m + logf(theta) + logf(z);
}

// Normalisation of one output row [TopTheta §3.2.1 Eq. 4, §3.2.2 Eq. 6-7].
// num = sum_{kept} exp(a_j - m) v_j, R = sum_{kept} exp(a_j - m), Z = all;
// e_off is the row's offline-calibrated E~ (TOPT_SDC_OFFLINE).
// Writes scale (multiplies num) and beta (multiplies mu when VMC is on).
__device__ __forceinline__ void out_scale_beta(int mode, int sdc, float gamma, float theta,
                                               float m, float Z, float R, int L, int kept,
                                               float e_off, float& scale, float& beta) {
  if (mode == TOPT_POST) {
    scale = 1.f / Z;
    beta = 1.f - R / Z;
    return;
  }
  if (sdc == TOPT_SDC_NONE) {
    scale = R > 0.f ? 1.f / R : 0.f;
    beta = 0.f;
    return;
  }
  float E;
  if (sdc == TOPT_SDC_EXACT) {
    E = fmaxf(Z - R, 0.f);
  } else if (sdc == TOPT_SDC_OFFLINE) {
    E = e_off;
  } else {
    E = (L > kept) ? gamma * (float)(L - kept) * __expf(theta - m) : 0.f;
  }
  float denom = R + E;
  scale = denom > 0.f ? 1.f / denom : 0.f;
  beta = denom > 0.f ? E / denom : 1.f;
}

}  // namespace topt

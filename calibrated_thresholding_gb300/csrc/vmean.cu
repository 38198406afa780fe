// Running mean of V rows for V-mean compensation.
//
// [TopTheta] = "Top-Theta Attention: Sparsifying Transformers by Compensated
// Thresholding" (arXiv 2502.08363v2), §3.2.2: mu is the mean V row (Eq. 5)
// and is kept as a running mean during generative decoding.
//
// mu <- mu + (sum of the t new rows - t * mu) / (n_old + t), which equals
// (n_old * mu + sum) / (n_old + t).  One CTA per (batch, KV head); 16-byte
// loads, LPR lanes per row, rows strided over the CTA, then a shared-memory
// reduction over the row lanes.  Given the step's new rows, the same threads
// first append them to the caches (rows n_old..) and average the values they
// loaded.
#include "common.cuh"
#include "internal.h"

namespace topt {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void load8f(const __nv_bfloat16* src, float f[8]) {
  const uint4 w = *reinterpret_cast<const uint4*>(src);
  f[0] = bf16lo(w.x); f[1] = bf16hi(w.x); f[2] = bf16lo(w.y); f[3] = bf16hi(w.y);
  f[4] = bf16lo(w.z); f[5] = bf16hi(w.z); f[6] = bf16lo(w.w); f[7] = bf16hi(w.w);
}
__device__ __forceinline__ void load8f(const float* src, float f[8]) {
  const float4 a = *reinterpret_cast<const float4*>(src);
  const float4 b = *reinterpret_cast<const float4*>(src + 4);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// Eight consecutive elements, copied as raw bytes.
__device__ __forceinline__ void copy8(__nv_bfloat16* dst, const __nv_bfloat16* src) {
  *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
}
__device__ __forceinline__ void copy8(float* dst, const float* src) {
  reinterpret_cast<float4*>(dst)[0] = reinterpret_cast<const float4*>(src)[0];
  reinterpret_cast<float4*>(dst)[1] = reinterpret_cast<const float4*>(src)[1];
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) vmean_kernel(int Hkv, int Nmax, int t, T* __restrict__ v,
                                                         const T* __restrict__ v_new, T* __restrict__ k,
                                                         const T* __restrict__ k_new,
                                                         const int32_t* __restrict__ n_old,
                                                         float* __restrict__ mu, int32_t* status) {
  constexpr int LPR = D / 8;
  constexpr int RL = kThreads / LPR;  // row lanes
  __shared__ float red[RL][D];
  // Launched so that it may start while the previous kernel of the stream
  // drains: wait for that kernel's writes, then let the next kernel be
  // scheduled (it waits for this one in turn).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int pair = blockIdx.x;
  const int b = pair / Hkv;
  const int n0 = n_old[b];
  if (n0 < 0 || n0 + t > Nmax) {
    if (threadIdx.x == 0) set_status(status, TOPT_EINVAL);
    return;
  }
  const int dl = threadIdx.x % LPR;
  const int rl = threadIdx.x / LPR;
  T* base = v + ((size_t)pair * Nmax + n0) * D + dl * 8;
  const T* src = v_new ? v_new + (size_t)pair * t * D + dl * 8 : base;
  float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int i = rl; i < t; i += RL) {
    float f[8];
    load8f(src + (size_t)i * D, f);
    if (v_new) copy8(base + (size_t)i * D, src + (size_t)i * D);
#pragma unroll
    for (int e = 0; e < 8; ++e) s[e] += f[e];
  }
  if (k_new) {
    T* kb = k + ((size_t)pair * Nmax + n0) * D + dl * 8;
    const T* ks = k_new + (size_t)pair * t * D + dl * 8;
    for (int i = rl; i < t; i += RL) copy8(kb + (size_t)i * D, ks + (size_t)i * D);
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) red[rl][dl * 8 + e] = s[e];
  __syncthreads();
  for (int dd = threadIdx.x; dd < D; dd += kThreads) {
    float tot = 0.f;
    for (int u = 0; u < RL; ++u) tot += red[u][dd];
    float* m = mu + (size_t)pair * D + dd;
    const float old = *m;
    *m = old + (tot - (float)t * old) / (float)(n0 + t);
  }
}

template <typename T>
cudaError_t launch_t(const topt_vmean_args& a, cudaStream_t s) {
  T* v = static_cast<T*>(a.v_cache);
  const T* v_new = static_cast<const T*>(a.v_new);
  T* k = static_cast<T*>(a.k_cache);
  const T* k_new = static_cast<const T*>(a.k_new);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.batch * a.n_kv_heads));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.head_dim == 128)
    return cudaLaunchKernelEx(&cfg, vmean_kernel<T, 128>, a.n_kv_heads, a.cache_len, a.n_new, v, v_new, k, k_new,
                              a.n_old, a.mu, a.status);
  return cudaLaunchKernelEx(&cfg, vmean_kernel<T, 64>, a.n_kv_heads, a.cache_len, a.n_new, v, v_new, k, k_new,
                            a.n_old, a.mu, a.status);
}

}  // namespace

cudaError_t vmean_launch(const topt_vmean_args& a, cudaStream_t s) {
  return a.dtype == TOPT_BF16 ? launch_t<__nv_bfloat16>(a, s) : launch_t<float>(a, s);
}

}  // namespace topt

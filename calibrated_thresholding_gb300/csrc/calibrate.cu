// Threshold calibration, [TopTheta §3.1, Algorithm 1], one layer per call.
//
// [TopTheta] = "Top-Theta Attention: Sparsifying Transformers by Compensated
// Thresholding" (arXiv 2502.08363v2).
//
// For every calibration row the observed threshold is the k-th largest score
// of the row (the (n-k)/n quantile read as an order statistic) or, for
// post-softmax thresholds, the softmax value of that score [TopTheta §3.1,
// the remark after Figure 2].  theta_r is the mean of the observations of row
// id r plus alpha standard deviations.  Rows are processed in passes that
// fit the caller's workspace:
//   calib_scores_kernel   scores of up to `rows_per_pass` rows -> workspace
//   calib_select_kernel   one CTA per row: 4 x 8-bit radix select of the
//                         k-th largest on order-preserving uint32 keys, then
//                         fp64 atomic accumulation of sum, sum of squares and
//                         count at [head][L-1]
//   calib_finalize_kernel one CTA per head: mean + alpha*std, dense rows,
//                         nearest calibrated row id for the rest.
#include "common.cuh"
#include "internal.h"

namespace topt {
namespace {

constexpr int kScoreKeys = 128;  // keys per score CTA (one per thread)
constexpr int kScoreRows = 8;    // query rows per score CTA
constexpr int kSelThreads = 256;
constexpr int kFinThreads = 1024;

// Order-preserving map float -> uint32 (-0.0 is folded onto +0.0).
__device__ __forceinline__ uint32_t f2key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key2f(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

struct SelectSmem {
  unsigned hist[256];
  unsigned sel[2];
  float red[kSelThreads / kWarp];
};

// Exact k-th largest (1-based, 1 <= k <= L) of row[0..L-1], computed by the
// whole CTA with four 8-bit digit passes from the most significant digit.
__device__ float cta_select_kth(const float* __restrict__ row, int L, int k, SelectSmem& sm) {
  uint32_t prefix = 0u, pmask = 0u;
  unsigned kk = (unsigned)k;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kSelThreads) sm.hist[i] = 0u;
    __syncthreads();
    for (int j = tid; j < L; j += kSelThreads) {
      const uint32_t key = f2key(row[j]);
      if ((key & pmask) == prefix) atomicAdd(&sm.hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid < kWarp) {
      // Lane l owns bins 255-8l down to 248-8l (descending order of value).
      unsigned cnt[8];
      unsigned tot = 0u;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        cnt[e] = sm.hist[255 - 8 * lane - e];
        tot += cnt[e];
      }
      unsigned incl = tot;
#pragma unroll
      for (int off = 1; off < kWarp; off <<= 1) {
        const unsigned v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      const unsigned excl = incl - tot;
      if (excl < kk && kk <= incl) {
        unsigned c = excl;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (c + cnt[e] >= kk) {
            sm.sel[0] = 255u - 8u * lane - e;
            sm.sel[1] = kk - c;
            break;
          }
          c += cnt[e];
        }
      }
    }
    __syncthreads();
    prefix |= sm.sel[0] << shift;
    pmask |= 0xffu << shift;
    kk = sm.sel[1];
  }
  return key2f(prefix);
}

__device__ float cta_reduce_max(float v, SelectSmem& sm) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sm.red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = sm.red[0];
  for (int w = 1; w < kSelThreads / kWarp; ++w) r = fmaxf(r, sm.red[w]);
  return r;
}

__device__ float cta_reduce_sum(float v, SelectSmem& sm) {
  v = warp_sum(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sm.red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = 0.f;
  for (int w = 0; w < kSelThreads / kWarp; ++w) r += sm.red[w];
  return r;
}

// Eight consecutive elements as fp32 (16-byte aligned source).
__device__ __forceinline__ void load8(const __nv_bfloat16* src, float f[8]) {
  const uint4 w = *reinterpret_cast<const uint4*>(src);
  f[0] = bf16lo(w.x); f[1] = bf16hi(w.x); f[2] = bf16lo(w.y); f[3] = bf16hi(w.y);
  f[4] = bf16lo(w.z); f[5] = bf16hi(w.z); f[6] = bf16lo(w.w); f[7] = bf16hi(w.w);
}
__device__ __forceinline__ void load8(const float* src, float f[8]) {
  const float4 a = *reinterpret_cast<const float4*>(src);
  const float4 b = *reinterpret_cast<const float4*>(src + 4);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

struct CalibParams {
  int N, Hq, Hkv, R, Nk, Lmax, mode, k;
  float alpha, sm_scale;
  const void* q;
  const void* keys;
  const int32_t* row_len;
  double* acc;
  int32_t* count;
  float* theta;
  int32_t* status;
};

// Scores of rows [it0, it0 + nrows) of the flattened (seq, head, row) index.
template <typename T, int D>
__global__ void __launch_bounds__(kScoreKeys) calib_scores_kernel(const CalibParams p, long it0,
                                                                  int nrows, float* __restrict__ ws) {
  __shared__ float qs[kScoreRows][D];
  __shared__ int s_L[kScoreRows];
  __shared__ long s_kofs[kScoreRows];
  const int r0 = blockIdx.y * kScoreRows;
  const T* Q = static_cast<const T*>(p.q);
  const T* K = static_cast<const T*>(p.keys);
  for (int idx = threadIdx.x; idx < kScoreRows * D; idx += kScoreKeys) {
    const int r = idx / D, dd = idx - r * D;
    const long it = it0 + r0 + r;
    qs[r][dd] = (r0 + r < nrows) ? to_f32<T>(Q[it * D + dd]) : 0.f;
  }
  if (threadIdx.x < kScoreRows) {
    const int r = threadIdx.x;
    const long it = it0 + r0 + r;
    int L = 0;
    long kofs = 0;
    if (r0 + r < nrows) {
      const long i = it % p.R;
      const long nh = it / p.R;
      const long h = nh % p.Hq;
      const long n = nh / p.Hq;
      L = p.row_len[i];
      if (L < 1 || L > p.Nk) L = 0;
      kofs = ((n * p.Hkv) + h / (p.Hq / p.Hkv)) * (long)p.Nk * D;
    }
    s_L[r] = L;
    s_kofs[r] = kofs;
  }
  __syncthreads();
  const int j = blockIdx.x * kScoreKeys + threadIdx.x;
  for (int r = 0; r < kScoreRows; ++r) {
    if (j >= s_L[r]) continue;
    const T* krow = K + s_kofs[r] + (long)j * D;
    float acc = 0.f;
#pragma unroll 4
    for (int dd = 0; dd < D; dd += 8) {
      float kf[8];
      load8(krow + dd, kf);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc = fmaf(kf[e], qs[r][dd + e], acc);
    }
    ws[(long)(r0 + r) * p.Nk + j] = acc * p.sm_scale;
  }
}

// One CTA per row of the pass: select, transform, accumulate.
__global__ void __launch_bounds__(kSelThreads) calib_select_kernel(const CalibParams p, long it0,
                                                                   const float* __restrict__ ws) {
  __shared__ SelectSmem sm;
  const long it = it0 + blockIdx.x;
  const long i = it % p.R;
  const long h = (it / p.R) % p.Hq;
  const int L = p.row_len[i];
  if (L < 1 || L > p.Nk || L > p.Lmax) {
    if (threadIdx.x == 0) set_status(p.status, TOPT_EINVAL);
    return;
  }
  if (L <= p.k) return;  // dense row, not calibrated [Algorithm 1 starts at row k]
  const float* row = ws + (long)blockIdx.x * p.Nk;
  const float kth = cta_select_kth(row, L, p.k, sm);
  float sample = kth;
  if (p.mode == TOPT_POST) {
    float m = -CUDART_INF_F;
    for (int j = threadIdx.x; j < L; j += kSelThreads) m = fmaxf(m, row[j]);
    m = cta_reduce_max(m, sm);
    float z = 0.f;
    for (int j = threadIdx.x; j < L; j += kSelThreads) z += expf(row[j] - m);
    z = cta_reduce_sum(z, sm);
    sample = expf(kth - m) / z;
  }
  if (threadIdx.x == 0) {
    const size_t cell = (size_t)h * p.Lmax + (L - 1);
    atomicAdd(p.acc + cell, (double)sample);
    atomicAdd(p.acc + (size_t)p.Hq * p.Lmax + cell, (double)sample * (double)sample);
    atomicAdd(p.count + cell, 1);
  }
}

__global__ void __launch_bounds__(kSelThreads) select_kth_kernel(const float* __restrict__ x, int stride,
                                                                 const int32_t* row_len, int k,
                                                                 float* out, int32_t* status) {
  __shared__ SelectSmem sm;
  const int r = blockIdx.x;
  const int L = row_len[r];
  if (L < 0 || L > stride) {
    if (threadIdx.x == 0) {
      set_status(status, TOPT_EINVAL);
      out[r] = CUDART_NAN_F;
    }
    return;
  }
  if (L < k) {
    if (threadIdx.x == 0) out[r] = -CUDART_INF_F;
    return;
  }
  const float v = cta_select_kth(x + (size_t)r * stride, L, k, sm);
  if (threadIdx.x == 0) out[r] = v;
}

__global__ void calib_zero_kernel(double* acc, int32_t* count, size_t cells) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < cells; i += (size_t)gridDim.x * blockDim.x) {
    acc[i] = 0.0;
    acc[cells + i] = 0.0;
    count[i] = 0;
  }
}

__device__ __forceinline__ float calib_value(const CalibParams& p, size_t cell) {
  const int n = p.count[cell];
  const double s1 = p.acc[cell];
  const double s2 = p.acc[(size_t)p.Hq * p.Lmax + cell];
  const double mean = s1 / n;
  double sd = 0.0;
  if (n > 1) {
    const double var = (s2 - (double)n * mean * mean) / (double)(n - 1);
    sd = var > 0.0 ? sqrt(var) : 0.0;
  }
  return (float)(mean + (double)p.alpha * sd);
}

// One CTA per head.  Segment-wise forward/backward sweeps find, for every row
// id, the nearest calibrated row below and above.
__global__ void __launch_bounds__(kFinThreads) calib_finalize_kernel(const CalibParams p) {
  __shared__ int s_last[kFinThreads], s_first[kFinThreads];
  const int h = blockIdx.x;
  const int Lmax = p.Lmax;
  const int seg = (Lmax + kFinThreads - 1) / kFinThreads;
  const int lo = min(threadIdx.x * seg, Lmax);
  const int hi = min(lo + seg, Lmax);
  const int32_t* cnt = p.count + (size_t)h * Lmax;
  float* th = p.theta + (size_t)h * Lmax;
  int last = -1, first = -1;
  for (int i = lo; i < hi; ++i)
    if (cnt[i] > 0) {
      last = i;
      if (first < 0) first = i;
    }
  s_last[threadIdx.x] = last;
  s_first[threadIdx.x] = first;
  __syncthreads();
  int prev = -1, next = -1;
  for (int u = 0; u < (int)threadIdx.x; ++u) prev = max(prev, s_last[u]);
  for (int u = kFinThreads - 1; u > (int)threadIdx.x; --u)
    if (s_first[u] >= 0) next = s_first[u];
  // forward: nearest calibrated index at or below i, stored as int bits
  for (int i = lo; i < hi; ++i) {
    if (cnt[i] > 0) prev = i;
    th[i] = __int_as_float(prev);
  }
  // backward: nearest at or above, then decide
  for (int i = hi - 1; i >= lo; --i) {
    if (cnt[i] > 0) next = i;
    const int below = __float_as_int(th[i]);
    const int L = i + 1;
    float v;
    if (cnt[i] > 0) {
      v = calib_value(p, (size_t)h * Lmax + i);
    } else if (L <= p.k || (below < 0 && next < 0)) {
      v = -CUDART_INF_F;
    } else {
      int pick;
      if (below < 0) pick = next;
      else if (next < 0) pick = below;
      else pick = (i - below <= next - i) ? below : next;
      v = calib_value(p, (size_t)h * Lmax + pick);
    }
    th[i] = v;
  }
}

template <typename T, int D>
cudaError_t calib_pass(const CalibParams& p, long it0, int nrows, float* ws, cudaStream_t s) {
  dim3 g1((p.Nk + kScoreKeys - 1) / kScoreKeys, (nrows + kScoreRows - 1) / kScoreRows);
  calib_scores_kernel<T, D><<<g1, kScoreKeys, 0, s>>>(p, it0, nrows, ws);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  calib_select_kernel<<<nrows, kSelThreads, 0, s>>>(p, it0, ws);
  return cudaGetLastError();
}

}  // namespace

size_t calibrate_min_rows_per_pass() { return kScoreRows; }

size_t calibrate_workspace_bytes(const topt_calib_args& a, size_t rows_per_pass) {
  return align256(rows_per_pass * (size_t)a.n_keys * sizeof(float));
}

cudaError_t calibrate_launch(const topt_calib_args& a, cudaStream_t s) {
  CalibParams p;
  p.N = a.n_seqs;
  p.Hq = a.n_q_heads;
  p.Hkv = a.n_kv_heads;
  p.R = a.n_rows;
  p.Nk = a.n_keys;
  p.Lmax = a.theta_len;
  p.mode = a.mode;
  p.k = a.k;
  p.alpha = a.alpha;
  p.sm_scale = 1.0f / sqrtf((float)a.head_dim);
  p.q = a.q;
  p.keys = a.keys;
  p.row_len = a.row_len;
  p.acc = a.acc;
  p.count = a.count;
  p.theta = a.theta;
  p.status = a.status;
  const size_t cells = (size_t)a.n_q_heads * a.theta_len;
  cudaError_t e;
  if (a.flags & TOPT_CALIB_RESET) {
    calib_zero_kernel<<<(unsigned)((cells + 255) / 256 < 4096 ? (cells + 255) / 256 : 4096), 256, 0, s>>>(
        a.acc, a.count, cells);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const long total = (long)a.n_seqs * a.n_q_heads * a.n_rows;
  if (total > 0) {
    size_t per_row = (size_t)a.n_keys * sizeof(float);
    long rows_per_pass = (long)(a.workspace_bytes / per_row);
    rows_per_pass = rows_per_pass / kScoreRows * kScoreRows;
    if (rows_per_pass > (1L << 20)) rows_per_pass = 1L << 20;
    if (rows_per_pass < kScoreRows) return cudaErrorInvalidValue;
    float* ws = static_cast<float*>(a.workspace);
    for (long it0 = 0; it0 < total; it0 += rows_per_pass) {
      const int nrows = (int)((total - it0) < rows_per_pass ? (total - it0) : rows_per_pass);
      if (a.dtype == TOPT_BF16) {
        e = a.head_dim == 128 ? calib_pass<__nv_bfloat16, 128>(p, it0, nrows, ws, s)
                              : calib_pass<__nv_bfloat16, 64>(p, it0, nrows, ws, s);
      } else {
        e = a.head_dim == 128 ? calib_pass<float, 128>(p, it0, nrows, ws, s)
                              : calib_pass<float, 64>(p, it0, nrows, ws, s);
      }
      if (e != cudaSuccess) return e;
    }
  }
  if (a.flags & TOPT_CALIB_FINALIZE) {
    calib_finalize_kernel<<<a.n_q_heads, kFinThreads, 0, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t select_kth_launch(const float* x, int32_t rows, int32_t stride, const int32_t* row_len,
                              int32_t k, float* out, int32_t* status, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  select_kth_kernel<<<rows, kSelThreads, 0, s>>>(x, stride, row_len, k, out, status);
  return cudaGetLastError();
}

}  // namespace topt

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
// The second half of the file is multi-k cumulative calibration
// [TopTheta App. D, Algorithm 2]: every threshold table theta(k) of a list of
// targets k from one pass over the calibration rows.
#include <atomic>

#include <cfloat>

#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace topt {
namespace {

constexpr int kScoreKeys = 128;  // keys per score CTA (one per thread)
constexpr int kScoreRows = 8;    // query rows per score CTA
constexpr int kSelThreads = 256;
constexpr int kFinThreads = 1024;
constexpr long kMaxPassRows = 65535L * kScoreRows;  // grid.y limit of the score kernel

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

// Key of the k-th largest (1-based, 1 <= k <= count) of the elements that
// `visit` hands out, computed by the whole CTA with four 8-bit digit passes
// from the most significant digit.  visit(f) calls f(key) once for every
// element of this thread's share; it runs once per pass.
template <class Visit>
__device__ uint32_t cta_select_key(const Visit& visit, unsigned kk, SelectSmem& sm) {
  uint32_t prefix = 0u, pmask = 0u;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += blockDim.x) sm.hist[i] = 0u;
    __syncthreads();
    visit([&](uint32_t key) {
      if ((key & pmask) == prefix) atomicAdd(&sm.hist[(key >> shift) & 255u], 1u);
    });
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
  return prefix;
}

// Exact k-th largest (1-based, 1 <= k <= L) of row[0..L-1].
__device__ float cta_select_kth(const float* __restrict__ row, int L, int k, SelectSmem& sm) {
  // four independent loads in flight per thread before any is used
  const auto visit = [&](auto&& f) {
    const int nt = blockDim.x;
    int j = threadIdx.x;
    for (; j + 3 * nt < L; j += 4 * nt) {
      const float x0 = row[j], x1 = row[j + nt], x2 = row[j + 2 * nt], x3 = row[j + 3 * nt];
      f(f2key(x0));
      f(f2key(x1));
      f(f2key(x2));
      f(f2key(x3));
    }
    for (; j < L; j += nt) f(f2key(row[j]));
  };
  return key2f(cta_select_key(visit, (unsigned)k, sm));
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
  int h0, Hp;  // the score kernel covers query heads h0 .. h0+Hp-1
  int fit;     // FINALIZE writes the fitted function of ln L (TOPT_CALIB_FIT)
  float alpha, sm_scale;
  const void* q;
  const void* keys;
  const int32_t* row_len;
  double* acc;
  int32_t* count;
  float* theta;
  int32_t* status;
};

// Scores of rows [it0, it0 + nrows) of the flattened (seq, head, row) index
// over the heads h0 .. h0+Hp-1; row it0 + r goes to ws row r.
template <typename T, int D>
__global__ void __launch_bounds__(kScoreKeys) calib_scores_kernel(const CalibParams p, long it0,
                                                                  int nrows, float* __restrict__ ws) {
  __shared__ float qs[kScoreRows][D];
  __shared__ int s_L[kScoreRows];
  __shared__ long s_kofs[kScoreRows];
  __shared__ long s_qofs[kScoreRows];
  const int r0 = blockIdx.y * kScoreRows;
  const T* Q = static_cast<const T*>(p.q);
  const T* K = static_cast<const T*>(p.keys);
  if (threadIdx.x < kScoreRows) {
    const int r = threadIdx.x;
    const long it = it0 + r0 + r;
    int L = 0;
    long kofs = 0, qofs = -1;
    if (r0 + r < nrows) {
      const long i = it % p.R;
      const long nh = it / p.R;
      const long h = p.h0 + nh % p.Hp;
      const long n = nh / p.Hp;
      L = p.row_len[i];
      if (L < 1 || L > p.Nk) L = 0;
      kofs = ((n * p.Hkv) + h / (p.Hq / p.Hkv)) * (long)p.Nk * D;
      qofs = ((n * p.Hq + h) * p.R + i) * D;
    }
    s_L[r] = L;
    s_kofs[r] = kofs;
    s_qofs[r] = qofs;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < kScoreRows * D; idx += kScoreKeys) {
    const int r = idx / D, dd = idx - r * D;
    qs[r][dd] = s_qofs[r] >= 0 ? to_f32<T>(Q[s_qofs[r] + dd]) : 0.f;
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

// One head's row of a threshold table, written by one CTA of kFinThreads:
// has(i) says whether row id L = i+1 was calibrated, val(i) its value.
// Rows with L <= k are dense (-inf); any other row takes the nearest
// calibrated row id (ties: the shorter row); no calibrated row: dense.
// Segment-wise forward/backward sweeps find, for every row id, the nearest
// calibrated row below and above; out[] holds the forward result as int bits
// in between.
template <class Has, class Val>
__device__ void fill_nearest_rows(int Lmax, int k, const Has& has, const Val& val, float* out) {
  __shared__ int s_last[kFinThreads], s_first[kFinThreads];
  const int seg = (Lmax + kFinThreads - 1) / kFinThreads;
  const int lo = min((int)threadIdx.x * seg, Lmax);
  const int hi = min(lo + seg, Lmax);
  int last = -1, first = -1;
  for (int i = lo; i < hi; ++i)
    if (has(i)) {
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
    if (has(i)) prev = i;
    out[i] = __int_as_float(prev);
  }
  // backward: nearest at or above, then decide
  for (int i = hi - 1; i >= lo; --i) {
    const bool hit = has(i);
    if (hit) next = i;
    const int below = __float_as_int(out[i]);
    const int L = i + 1;
    float v;
    if (hit) {
      v = val(i);
    } else if (L <= k || (below < 0 && next < 0)) {
      v = -CUDART_INF_F;
    } else {
      int pick;
      if (below < 0) pick = next;
      else if (next < 0) pick = below;
      else pick = (i - below <= next - i) ? below : next;
      v = val(pick);
    }
    out[i] = v;
  }
}

// One head's row of a threshold table from a least-squares line (degree
// min(1, n - 1)) in x = ln L through the n usable calibrated row ids L > k:
// y = theta (PRE) or ln theta (POST, theta > 0 only).  Every L > k takes the
// fitted value (exp of it for POST, kept between the smallest normal float and
// the head's largest calibrated value, so that an extrapolated row neither
// drops every key nor reads as "keep all"); L <= k and a head without usable
// row ids are dense.  The pages mention a fitted function of the sequence length
// without its form; a line in ln L extrapolates past the calibrated lengths
// far better than a quadratic.  fp64 normal equations (the sums cover a
// quadratic), solved by one thread.
constexpr int kFitDegree = 1;  // degree of the fitted polynomial in ln L (at most 2)

template <class Has, class Val>
__device__ void fit_rows(int Lmax, int k, int mode, const Has& has, const Val& val, float* out) {
  constexpr int kW = kFinThreads / kWarp;
  __shared__ double red[8][kW];
  __shared__ double S[8];      // the reduced sums
  __shared__ double A[3][4];   // normal equations | right-hand side
  __shared__ double coef[3];
  __shared__ int s_deg;
  __shared__ float s_cap;
  __shared__ float red_cap[kW];
  double m[8];  // sums of x^0..x^4, then of y x^0..y x^2
  float cap = 0.f;  // largest usable calibrated value (POST)
#pragma unroll
  for (int q = 0; q < 8; ++q) m[q] = 0.0;
  for (int i = threadIdx.x; i < Lmax; i += kFinThreads) {
    const int L = i + 1;
    if (L <= k || !has(i)) continue;
    double y = (double)val(i);
    if (mode == TOPT_POST) {
      if (!(y > 0.0)) continue;
      cap = fmaxf(cap, val(i));
      y = log(y);
    }
    const double x = log((double)L);
    double xp = 1.0;
#pragma unroll
    for (int q = 0; q < 5; ++q) {
      m[q] += xp;
      if (q < 3) m[5 + q] += xp * y;
      xp *= x;
    }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    double v = m[q];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0) red[q][warp] = v;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) cap = fmaxf(cap, __shfl_xor_sync(0xffffffffu, cap, off));
  if (lane == 0) red_cap[warp] = cap;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int q = 0; q < 8; ++q) {
      S[q] = 0.0;
      for (int w = 0; w < kW; ++w) S[q] += red[q][w];
    }
    float c = 0.f;
    for (int w = 0; w < kW; ++w) c = fmaxf(c, red_cap[w]);
    s_cap = c;
    const int n = (int)(S[0] + 0.5);
    const int deg = n < 2 ? n - 1 : kFitDegree;
    if (deg >= 0) {
      // A c = t with A[r][c] = sum x^(r+c), t[r] = sum y x^r; partial pivoting
      const int sz = deg + 1;
      for (int r = 0; r < sz; ++r) {
        for (int c = 0; c < sz; ++c) A[r][c] = S[r + c];
        A[r][3] = S[5 + r];
      }
      for (int c = 0; c < sz; ++c) {
        int piv = c;
        for (int r = c + 1; r < sz; ++r)
          if (fabs(A[r][c]) > fabs(A[piv][c])) piv = r;
        if (piv != c)
          for (int e = 0; e < 4; ++e) {
            const double t = A[c][e];
            A[c][e] = A[piv][e];
            A[piv][e] = t;
          }
        for (int r = c + 1; r < sz; ++r) {
          const double f = A[r][c] / A[c][c];
          for (int e = c; e < 4; ++e) A[r][e] -= f * A[c][e];
        }
      }
      coef[0] = coef[1] = coef[2] = 0.0;
      for (int r = sz - 1; r >= 0; --r) {
        double v = A[r][3];
        for (int e = r + 1; e < sz; ++e) v -= A[r][e] * coef[e];
        coef[r] = v / A[r][r];
      }
    }
    s_deg = deg;
  }
  __syncthreads();
  const int deg = s_deg;
  for (int i = threadIdx.x; i < Lmax; i += kFinThreads) {
    const int L = i + 1;
    if (L <= k || deg < 0) {
      out[i] = -CUDART_INF_F;
      continue;
    }
    const double x = log((double)L);
    const double y = coef[0] + x * (coef[1] + x * coef[2]);
    out[i] = mode == TOPT_POST ? fmaxf(fminf((float)exp(y), s_cap), FLT_MIN) : (float)y;
  }
}

// One CTA per head.
__global__ void __launch_bounds__(kFinThreads) calib_finalize_kernel(const CalibParams p) {
  const int h = blockIdx.x;
  const int32_t* cnt = p.count + (size_t)h * p.Lmax;
  const auto has = [&](int i) { return cnt[i] > 0; };
  const auto val = [&](int i) { return calib_value(p, (size_t)h * p.Lmax + i); };
  if (p.fit) fit_rows(p.Lmax, p.k, p.mode, has, val, p.theta + (size_t)h * p.Lmax);
  else fill_nearest_rows(p.Lmax, p.k, has, val, p.theta + (size_t)h * p.Lmax);
}

// ---------------------------------------------------------------------------
// Offline-calibrated SDC estimate [TopTheta §3.2.1, estimator 1]: the mean,
// per (head, row id), of each calibration row's discarded exponent sum
// E = sum_{a_j < theta} exp(a_j - m) under a pre-softmax threshold table.
// The same score passes as Algorithm 1; acc holds one sum per cell.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kSelThreads) calib_e_kernel(const CalibParams p, long it0,
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
  const float th = p.theta[(size_t)h * p.Lmax + (L - 1)];
  if (!(th > -CUDART_INF_F)) return;  // the row is kept whole: no sample
  const float* row = ws + (long)blockIdx.x * p.Nk;
  float m = -CUDART_INF_F;
  for (int j = threadIdx.x; j < L; j += kSelThreads) m = fmaxf(m, row[j]);
  m = cta_reduce_max(m, sm);
  float e = 0.f;
  for (int j = threadIdx.x; j < L; j += kSelThreads) {
    const float x = row[j];
    if (x < th) e += expf(x - m);
  }
  e = cta_reduce_sum(e, sm);
  if (threadIdx.x == 0) {
    const size_t cell = (size_t)h * p.Lmax + (L - 1);
    atomicAdd(p.acc + cell, (double)e);
    atomicAdd(p.count + cell, 1);
  }
}

__global__ void calib_e_zero_kernel(double* acc, int32_t* count, size_t cells) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < cells; i += (size_t)gridDim.x * blockDim.x) {
    acc[i] = 0.0;
    count[i] = 0;
  }
}

// One CTA per head: sample means, nearest sampled row id elsewhere, 0 where
// theta is -inf or the head has no sample.
__global__ void __launch_bounds__(kFinThreads) calib_e_finalize_kernel(const CalibParams p, float* e_tilde) {
  const int h = blockIdx.x;
  const size_t off = (size_t)h * p.Lmax;
  const float* th = p.theta + off;
  const auto has = [&](int i) { return p.count[off + i] > 0 && th[i] > -CUDART_INF_F; };
  const auto val = [&](int i) { return (float)(p.acc[off + i] / (double)p.count[off + i]); };
  fill_nearest_rows(p.Lmax, 0, has, val, e_tilde + off);
  __syncthreads();
  for (int i = threadIdx.x; i < p.Lmax; i += kFinThreads) {
    const float v = e_tilde[off + i];
    e_tilde[off + i] = (th[i] > -CUDART_INF_F && v > -CUDART_INF_F) ? v : 0.f;
  }
}

// Scores of rows [it0, it0 + nrows) into ws: the tensor-core kernel for bf16
// rows it suits (calib_tc.cu), the CUDA-core kernel above otherwise.
template <typename T, int D>
cudaError_t calib_scores(const CalibParams& p, long it0, int nrows, float* ws, cudaStream_t s) {
  if constexpr (std::is_same<T, __nv_bfloat16>::value) {
    CalibScoreArgs a;
    a.q = p.q;
    a.keys = p.keys;
    a.row_len = p.row_len;
    a.N = p.N;
    a.Hq = p.Hq;
    a.Hkv = p.Hkv;
    a.R = p.R;
    a.Nk = p.Nk;
    a.D = D;
    a.h0 = p.h0;
    a.Hp = p.Hp;
    a.scale = p.sm_scale;
    a.it0 = it0;
    a.nrows = nrows;
    a.ws = ws;
    a.status = p.status;
    if (calib_scores_tc_ok(a)) return calib_scores_tc(a, s);
  }
  dim3 g((p.Nk + kScoreKeys - 1) / kScoreKeys, (nrows + kScoreRows - 1) / kScoreRows);
  calib_scores_kernel<T, D><<<g, kScoreKeys, 0, s>>>(p, it0, nrows, ws);
  return cudaGetLastError();
}

template <typename T, int D, bool kSdc = false>
cudaError_t calib_pass(const CalibParams& p, long it0, int nrows, float* ws, cudaStream_t s) {
  cudaError_t e = calib_scores<T, D>(p, it0, nrows, ws, s);
  if (e != cudaSuccess) return e;
  if (kSdc) calib_e_kernel<<<nrows, kSelThreads, 0, s>>>(p, it0, ws);
  else calib_select_kernel<<<nrows, kSelThreads, 0, s>>>(p, it0, ws);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Multi-k cumulative calibration [TopTheta App. D, Algorithm 2, Eq. 8].
//
// For the calibration rows of one head and one length r (N_r rows, pooled
// values x), Eq. 8 averages the effective k of the rows whose [min, max)
// holds theta.  With B(theta) = #{rows whose maximum is > theta},
// A(theta) = #{rows whose minimum is > theta} and P(theta) = #{x > theta}:
//   k_bar(theta) >= k  <=>  B - A > 0  and  P >= k B + (r - k) A,
// because every row with min <= theta < max has #{its x > theta} elements
// above theta, a row with min > theta has all r and a row with max <= theta
// none.  B and A change only at row maxima and minima ("events"); between
// two consecutive events the condition is monotone in theta.  So
// theta(k) = sup{theta : k_bar(theta) >= k} is found from the highest event
// e that starts a valid stretch [e, u) (u the next event above e):
//   theta(k) = min(u, the T-th largest x),  T = k B(e) + (r - k) A(e).
// The kernel sorts the events in shared memory, counts P at every event
// with two histograms of the pooled values, and makes one radix select per
// target k.
// ---------------------------------------------------------------------------
constexpr int kMkcMaxSamples = 4096;  // calibration rows of one head and length per call
constexpr int kMkcThreads = kSelThreads;
constexpr int kMkcMaxK = 8;            // targets selected together (one warp each)
constexpr int kMkcSmall = 8;           // rows of a group up to which events are counted in registers
static_assert(kMkcThreads / kWarp >= kMkcMaxK, "a warp per target");
constexpr int kIdxThreads = 1024;

struct MkcSmem {
  uint32_t mx[kMkcMaxSamples];      // row maxima (keys), sorted descending
  uint32_t mn[kMkcMaxSamples];      // row minima (keys), sorted descending
  uint32_t px[kMkcMaxSamples + 1];  // px[c] = #{x : #{mx >= x} <= c} after the scan
  uint32_t pn[kMkcMaxSamples + 1];  // same against the minima
};

struct MkcParams {
  int N, Hq, R, Nk, Lmax, n_k, h0, Hp, mode;
  const int32_t* ks;         // [n_k] target k values
  const int32_t* row_len;    // [R]
  int32_t* len_cnt;          // [Lmax + 1] rows of a sequence with L keys
  int32_t* len_start;        // [Lmax + 1] first slot of length L in `order`
  int32_t* order;            // [R] row ids grouped by length
  float* ws;                 // scores (log-softmax for POST) [N][Hp][R][Nk] of the pass
  float* gval;               // [n_k][Hq][Lmax] theta_L(k) of the calibrated lengths
  int32_t* status;
};

// Rows grouped by length: counting sort of row_len (one CTA).
__global__ void __launch_bounds__(kIdxThreads) mkc_index_kernel(const MkcParams p, int32_t* cur) {
  __shared__ int tot[kIdxThreads];
  int32_t* cnt = p.len_cnt;
  int32_t* start = p.len_start;
  int32_t* order = p.order;
  const int n = p.Lmax + 1;
  for (int i = threadIdx.x; i < n; i += kIdxThreads) cnt[i] = 0;
  for (int i = threadIdx.x; i < p.n_k; i += kIdxThreads)
    if (p.ks[i] < 1) set_status(p.status, TOPT_EINVAL);
  __syncthreads();
  for (int i = threadIdx.x; i < p.R; i += kIdxThreads) {
    const int L = p.row_len[i];
    if (L < 1 || L > p.Nk || L > p.Lmax) set_status(p.status, TOPT_EINVAL);
    else atomicAdd(&cnt[L], 1);
  }
  __syncthreads();
  const int seg = (n + kIdxThreads - 1) / kIdxThreads;
  const int lo = min((int)threadIdx.x * seg, n), hi = min(lo + seg, n);
  int t = 0;
  for (int i = lo; i < hi; ++i) t += cnt[i];
  tot[threadIdx.x] = t;
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int u = 0; u < kIdxThreads; ++u) {
      const int v = tot[u];
      tot[u] = run;
      run += v;
    }
  }
  __syncthreads();
  int run = tot[threadIdx.x];
  for (int i = lo; i < hi; ++i) {
    start[i] = run;
    cur[i] = run;
    run += cnt[i];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < p.R; i += kIdxThreads) {
    const int L = p.row_len[i];
    if (L >= 1 && L <= p.Nk && L <= p.Lmax) order[atomicAdd(&cur[L], 1)] = i;
  }
}

// POST: every score row of the pass becomes its log-softmax a - m - ln Z, in
// place.  It orders the pooled values as the softmax values do (exp is
// increasing) without the fp32 underflow of small probabilities to one tied
// zero; the selected threshold is exponentiated at the end.
__global__ void __launch_bounds__(kSelThreads) mkc_softmax_kernel(const MkcParams p) {
  __shared__ SelectSmem sm;
  const long lr = blockIdx.x;
  const int L = p.row_len[lr % p.R];
  if (L < 1 || L > p.Nk || L > p.Lmax) return;
  float* row = p.ws + lr * p.Nk;
  float m = -CUDART_INF_F;
  for (int j = threadIdx.x; j < L; j += kSelThreads) m = fmaxf(m, row[j]);
  m = cta_reduce_max(m, sm);
  float z = 0.f;
  for (int j = threadIdx.x; j < L; j += kSelThreads) z += expf(row[j] - m);
  z = cta_reduce_sum(z, sm);
  const float lz = logf(z);
  for (int j = threadIdx.x; j < L; j += kSelThreads) row[j] = (row[j] - m) - lz;
}

// Entries of a[0..n) (sorted descending) that are > key, or >= key.
__device__ __forceinline__ int count_gt(const uint32_t* a, int n, uint32_t key) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] > key) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}
__device__ __forceinline__ int count_ge(const uint32_t* a, int n, uint32_t key) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] >= key) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// Inclusive prefix sums of a[0..n) and b[0..n) by the whole CTA.
__device__ void cta_scan2(uint32_t* a, uint32_t* b, int n) {
  __shared__ uint32_t ta[kMkcThreads], tb[kMkcThreads];
  const int seg = (n + kMkcThreads - 1) / kMkcThreads;
  const int lo = min((int)threadIdx.x * seg, n), hi = min(lo + seg, n);
  uint32_t sa = 0u, sb = 0u;
  for (int i = lo; i < hi; ++i) {
    sa += a[i];
    sb += b[i];
  }
  ta[threadIdx.x] = sa;
  tb[threadIdx.x] = sb;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t ra = 0u, rb = 0u;
    for (int u = 0; u < kMkcThreads; ++u) {
      const uint32_t va = ta[u], vb = tb[u];
      ta[u] = ra;
      tb[u] = rb;
      ra += va;
      rb += vb;
    }
  }
  __syncthreads();
  uint32_t ra = ta[threadIdx.x], rb = tb[threadIdx.x];
  for (int i = lo; i < hi; ++i) {
    ra += a[i];
    rb += b[i];
    a[i] = ra;
    b[i] = rb;
  }
  __syncthreads();
}

// One CTA per (row length L, head of the pass).
__global__ void __launch_bounds__(kMkcThreads) mkc_group_kernel(const MkcParams p) {
  extern __shared__ __align__(16) unsigned char mkc_raw[];
  MkcSmem& sh = *reinterpret_cast<MkcSmem*>(mkc_raw);
  __shared__ SelectSmem sm;
  __shared__ uint32_t s_best[kMkcThreads / kWarp];
  __shared__ unsigned s_hist[kMkcMaxK][256];  // per target: histogram of the current digit
  __shared__ uint32_t s_act[kMkcMaxK], s_kk[kMkcMaxK], s_pre[kMkcMaxK], s_u[kMkcMaxK];
  const int L = blockIdx.x + 1;
  const int hl = blockIdx.y;
  const int c = p.len_cnt[L];
  if (c == 0 || L < 2) return;  // a row of one key has no interval
  bool wanted = false;
  for (int ki = 0; ki < p.n_k; ++ki) wanted |= (p.ks[ki] >= 1 && p.ks[ki] < L);
  if (!wanted) return;  // row id L <= k is dense for every target
  const long nr_l = (long)p.N * c;
  if (nr_l > kMkcMaxSamples) {
    if (threadIdx.x == 0) set_status(p.status, TOPT_EINVAL);
    return;
  }
  const int Nr = (int)nr_l;
  int cap = 1;
  while (cap < Nr) cap <<= 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int nw = kMkcThreads / kWarp;
  const int base = p.len_start[L];
  const auto rowp = [&](int s) -> const float* {
    const int n = s / c, idx = s - n * c;
    const int i = p.order[base + idx];
    return p.ws + (((long)n * p.Hp + hl) * p.R + i) * p.Nk;
  };
  // f(key) for the keys of row s that this lane owns (j = lane mod 32): eight
  // independent loads in flight before any of them is used (the workspace is
  // read from L2 again and again; one load at a time left the warps waiting)
  const auto row_keys = [&](int s, auto&& f) {
    const float* row = rowp(s);
    int j = lane;
    for (; j + 7 * kWarp < L; j += 8 * kWarp) {
      float x[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) x[u] = row[j + u * kWarp];
#pragma unroll
      for (int u = 0; u < 8; ++u) f(f2key(x[u]));
    }
    for (; j < L; j += kWarp) f(f2key(row[j]));
  };
  // 1. maximum and minimum of every row; padding (key 0) sorts last
  for (int s = warp; s < cap; s += nw) {
    uint32_t hi_k = 0u, lo_k = 0u;
    if (s < Nr) {
      lo_k = 0xffffffffu;
      row_keys(s, [&](uint32_t key) {
        hi_k = max(hi_k, key);
        lo_k = min(lo_k, key);
      });
      hi_k = __reduce_max_sync(0xffffffffu, hi_k);
      lo_k = __reduce_min_sync(0xffffffffu, lo_k);
    }
    if (lane == 0) {
      sh.mx[s] = hi_k;
      sh.mn[s] = lo_k;
    }
  }
  __syncthreads();
  // 2. bitonic sort of both event arrays, descending
  for (int size = 2; size <= cap; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = tid; t < cap / 2; t += kMkcThreads) {
        const int lo = 2 * t - (t & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        uint32_t a = sh.mx[lo], b = sh.mx[hi];
        if ((a < b) == desc) {
          sh.mx[lo] = b;
          sh.mx[hi] = a;
        }
        a = sh.mn[lo];
        b = sh.mn[hi];
        if ((a < b) == desc) {
          sh.mn[lo] = b;
          sh.mn[hi] = a;
        }
      }
      __syncthreads();
    }
  }
  // 3. P at every event.  Up to kMkcSmall rows: every thread counts
  // #{x > e} for each event e in registers, summed over the CTA into
  // px[t] (t-th maximum) and pn[t] (t-th minimum).  More rows: histograms of
  // #{events >= x} (x > e <=> #{events >= x} <= #{events > e}), scanned, read
  // at px[#{maxima > e}] and pn[#{minima > e}].
  const bool small = Nr <= kMkcSmall;
  for (int i = tid; i <= Nr; i += kMkcThreads) {
    sh.px[i] = 0u;
    sh.pn[i] = 0u;
  }
  __syncthreads();
  if (small) {
    uint32_t ex[kMkcSmall], en[kMkcSmall], cx[kMkcSmall], cn[kMkcSmall];
#pragma unroll
    for (int t = 0; t < kMkcSmall; ++t) {
      ex[t] = t < Nr ? sh.mx[t] : 0xffffffffu;  // padding: no key is above it
      en[t] = t < Nr ? sh.mn[t] : 0xffffffffu;
      cx[t] = cn[t] = 0u;
    }
    for (int s = warp; s < Nr; s += nw) {
      row_keys(s, [&](uint32_t key) {
#pragma unroll
        for (int t = 0; t < kMkcSmall; ++t) {
          cx[t] += key > ex[t];
          cn[t] += key > en[t];
        }
      });
    }
#pragma unroll
    for (int t = 0; t < kMkcSmall; ++t) {
      const uint32_t a = __reduce_add_sync(0xffffffffu, cx[t]);
      const uint32_t b2 = __reduce_add_sync(0xffffffffu, cn[t]);
      if (lane == 0 && t < Nr) {
        atomicAdd(&sh.px[t], a);
        atomicAdd(&sh.pn[t], b2);
      }
    }
    __syncthreads();
  } else {
    for (int s = warp; s < Nr; s += nw) {
      row_keys(s, [&](uint32_t key) {
        atomicAdd(&sh.px[count_ge(sh.mx, Nr, key)], 1u);
        atomicAdd(&sh.pn[count_ge(sh.mn, Nr, key)], 1u);
      });
    }
    __syncthreads();
    cta_scan2(sh.px, sh.pn, Nr + 1);
  }
  // 4. every target k: the highest valid event e (its stretch [e, u)) gives
  // T; theta(k) = min(u, the T-th largest pooled value).  The selections of
  // up to kMkcMaxK targets run together: four digit sweeps over the pooled
  // values, each filling one 256-bin histogram per target.
  const auto visit = [&](auto&& f) {
    for (int s = warp; s < Nr; s += nw) row_keys(s, f);
  };
  for (int k0 = 0; k0 < p.n_k; k0 += kMkcMaxK) {
    const int nk = min(kMkcMaxK, p.n_k - k0);
    for (int jj = 0; jj < nk; ++jj) {
      const int ki = k0 + jj;
      const int k = p.ks[ki];
      if (tid == 0) s_act[jj] = 0u;
      if (k < 1 || k >= L) continue;  // uniform over the CTA
      uint32_t best = 0u;
      for (int t = tid; t < 2 * Nr; t += kMkcThreads) {
        const bool from_max = t < Nr;
        const uint32_t e = from_max ? sh.mx[t] : sh.mn[t - Nr];
        const int bx = count_gt(sh.mx, Nr, e);
        const int a = count_gt(sh.mn, Nr, e);
        if (bx - a <= 0) continue;
        const uint32_t P = small ? (from_max ? sh.px[t] : sh.pn[t - Nr]) : (from_max ? sh.px[bx] : sh.pn[a]);
        const long T = (long)k * bx + (long)(L - k) * a;
        if ((long)P >= T) best = max(best, e);
      }
      best = __reduce_max_sync(0xffffffffu, best);
      __syncthreads();
      if (lane == 0) s_best[warp] = best;
      __syncthreads();
      best = 0u;
#pragma unroll
      for (int w = 0; w < nw; ++w) best = max(best, s_best[w]);
      if (tid == 0) {
        if (best == 0u) {  // no stretch reaches k
          p.gval[((size_t)ki * p.Hq + p.h0 + hl) * p.Lmax + (L - 1)] = -CUDART_INF_F;
        } else {
          const int bx = count_gt(sh.mx, Nr, best);
          const int a = count_gt(sh.mn, Nr, best);
          uint32_t u = sh.mx[bx - 1];  // bx >= 1: a valid stretch has a maximum above it
          if (a > 0) u = min(u, sh.mn[a - 1]);
          s_act[jj] = 1u;
          s_kk[jj] = (unsigned)((long)k * bx + (long)(L - k) * a);
          s_u[jj] = u;
          s_pre[jj] = 0u;
        }
      }
    }
    __syncthreads();
    uint32_t pmask = 0u;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < nk * 256; i += kMkcThreads) s_hist[i >> 8][i & 255] = 0u;
      __syncthreads();
      uint32_t pre[kMkcMaxK];
      bool act[kMkcMaxK];
#pragma unroll
      for (int jj = 0; jj < kMkcMaxK; ++jj) {
        act[jj] = jj < nk && s_act[jj] != 0u;
        pre[jj] = act[jj] ? s_pre[jj] : 0u;
      }
      visit([&](uint32_t key) {
#pragma unroll
        for (int jj = 0; jj < kMkcMaxK; ++jj)
          if (act[jj] && (key & pmask) == pre[jj]) atomicAdd(&s_hist[jj][(key >> shift) & 255u], 1u);
      });
      __syncthreads();
      if (warp < nk && s_act[warp] != 0u) {
        // warp jj: the digit of the kk-th largest; lane l owns bins
        // 255-8l down to 248-8l (descending order of value)
        const unsigned kk = s_kk[warp];
        unsigned cnt[8];
        unsigned tot = 0u;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          cnt[e] = s_hist[warp][255 - 8 * lane - e];
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
              s_pre[warp] |= (255u - 8u * lane - e) << shift;
              s_kk[warp] = kk - c;
              break;
            }
            c += cnt[e];
          }
        }
      }
      __syncthreads();
      pmask |= 0xffu << shift;
    }
    if (tid < nk && s_act[tid] != 0u) {
      const float v = key2f(min(s_pre[tid], s_u[tid]));
      p.gval[((size_t)(k0 + tid) * p.Hq + p.h0 + hl) * p.Lmax + (L - 1)] = p.mode == TOPT_POST ? expf(v) : v;
    }
    __syncthreads();
  }
}

// One CTA per (head, target k): the table of that k.
__global__ void __launch_bounds__(kFinThreads) mkc_finalize_kernel(const MkcParams p, float* theta) {
  const int h = blockIdx.x, ki = blockIdx.y;
  const int k = p.ks[ki];
  const size_t off = ((size_t)ki * p.Hq + h) * p.Lmax;
  const auto has = [&](int i) { return i + 1 > k && p.len_cnt[i + 1] > 0; };
  const auto val = [&](int i) { return p.gval[off + i]; };
  fill_nearest_rows(p.Lmax, k, has, val, theta + off);
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
  p.h0 = 0;
  p.Hp = a.n_q_heads;
  p.fit = (a.flags & TOPT_CALIB_FIT) != 0;
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
    if (rows_per_pass > kMaxPassRows) rows_per_pass = kMaxPassRows;
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

size_t calibrate_sdc_workspace_bytes(const topt_sdc_calib_args& a, size_t rows_per_pass) {
  return align256(rows_per_pass * (size_t)a.n_keys * sizeof(float));
}

cudaError_t calibrate_sdc_launch(const topt_sdc_calib_args& a, cudaStream_t s) {
  CalibParams p;
  p.N = a.n_seqs;
  p.Hq = a.n_q_heads;
  p.Hkv = a.n_kv_heads;
  p.R = a.n_rows;
  p.Nk = a.n_keys;
  p.Lmax = a.theta_len;
  p.mode = TOPT_PRE;
  p.k = 1;
  p.h0 = 0;
  p.Hp = a.n_q_heads;
  p.fit = 0;
  p.alpha = 0.f;
  p.sm_scale = 1.0f / sqrtf((float)a.head_dim);
  p.q = a.q;
  p.keys = a.keys;
  p.row_len = a.row_len;
  p.acc = a.acc;
  p.count = a.count;
  p.theta = const_cast<float*>(a.theta);  // read only here
  p.status = a.status;
  const size_t cells = (size_t)a.n_q_heads * a.theta_len;
  cudaError_t e;
  if (a.flags & TOPT_CALIB_RESET) {
    calib_e_zero_kernel<<<(unsigned)((cells + 255) / 256 < 4096 ? (cells + 255) / 256 : 4096), 256, 0, s>>>(
        a.acc, a.count, cells);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const long total = (long)a.n_seqs * a.n_q_heads * a.n_rows;
  if (total > 0) {
    long rows_per_pass = (long)(a.workspace_bytes / ((size_t)a.n_keys * sizeof(float)));
    rows_per_pass = rows_per_pass / kScoreRows * kScoreRows;
    if (rows_per_pass > kMaxPassRows) rows_per_pass = kMaxPassRows;
    if (rows_per_pass < kScoreRows) return cudaErrorInvalidValue;
    float* ws = static_cast<float*>(a.workspace);
    for (long it0 = 0; it0 < total; it0 += rows_per_pass) {
      const int nrows = (int)((total - it0) < rows_per_pass ? (total - it0) : rows_per_pass);
      if (a.dtype == TOPT_BF16) {
        e = a.head_dim == 128 ? calib_pass<__nv_bfloat16, 128, true>(p, it0, nrows, ws, s)
                              : calib_pass<__nv_bfloat16, 64, true>(p, it0, nrows, ws, s);
      } else {
        e = a.head_dim == 128 ? calib_pass<float, 128, true>(p, it0, nrows, ws, s)
                              : calib_pass<float, 64, true>(p, it0, nrows, ws, s);
      }
      if (e != cudaSuccess) return e;
    }
  }
  if (a.flags & TOPT_CALIB_FINALIZE) {
    calib_e_finalize_kernel<<<a.n_q_heads, kFinThreads, 0, s>>>(p, a.e_tilde);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Workspace of multi-k calibration: row index, per-k values, then the scores
// of as many heads as fit.
size_t calibrate_multik_fixed_bytes(const topt_mkc_args& a) {
  return 3 * align256((size_t)(a.theta_len + 1) * sizeof(int32_t)) +
         align256((size_t)a.n_rows * sizeof(int32_t)) +
         align256((size_t)a.n_k * a.n_q_heads * a.theta_len * sizeof(float));
}
size_t calibrate_multik_head_bytes(const topt_mkc_args& a) {
  return align256((size_t)a.n_seqs * a.n_rows * a.n_keys * sizeof(float));
}
int calibrate_multik_max_samples() { return kMkcMaxSamples; }

template <typename T, int D>
cudaError_t mkc_scores(const CalibParams& cp, long total, float* ws, cudaStream_t s) {
  for (long it0 = 0; it0 < total; it0 += kMaxPassRows) {
    const int nrows = (int)((total - it0) < kMaxPassRows ? (total - it0) : kMaxPassRows);
    cudaError_t e = calib_scores<T, D>(cp, it0, nrows, ws + it0 * (long)cp.Nk, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t calibrate_multik_launch(const topt_mkc_args& a, cudaStream_t s) {
  // the group kernel's shared-memory limit, raised once per device
  constexpr int kMaxDevices = 64;
  static std::atomic<bool> attr_set[kMaxDevices];
  cudaError_t e;
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!attr_set[dev].load()) {
    e = cudaFuncSetAttribute(mkc_group_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(MkcSmem));
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true);
  }
  char* w = static_cast<char*>(a.workspace);
  const size_t lb = align256((size_t)(a.theta_len + 1) * sizeof(int32_t));
  MkcParams p;
  p.N = a.n_seqs;
  p.Hq = a.n_q_heads;
  p.R = a.n_rows;
  p.Nk = a.n_keys;
  p.Lmax = a.theta_len;
  p.n_k = a.n_k;
  p.mode = a.mode;
  p.ks = a.ks;
  p.row_len = a.row_len;
  p.len_cnt = reinterpret_cast<int32_t*>(w);
  p.len_start = reinterpret_cast<int32_t*>(w + lb);
  int32_t* cur = reinterpret_cast<int32_t*>(w + 2 * lb);
  p.order = reinterpret_cast<int32_t*>(w + 3 * lb);
  p.gval = reinterpret_cast<float*>(w + 3 * lb + align256((size_t)a.n_rows * sizeof(int32_t)));
  p.status = a.status;
  float* ws = reinterpret_cast<float*>(w + calibrate_multik_fixed_bytes(a));
  const size_t per_head = calibrate_multik_head_bytes(a);
  size_t fit = (a.workspace_bytes - calibrate_multik_fixed_bytes(a)) / per_head;
  const int Hp = fit < (size_t)a.n_q_heads ? (int)fit : a.n_q_heads;
  if (Hp < 1) return cudaErrorInvalidValue;
  p.ws = ws;

  mkc_index_kernel<<<1, kIdxThreads, 0, s>>>(p, cur);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  CalibParams cp;
  cp.N = a.n_seqs;
  cp.Hq = a.n_q_heads;
  cp.Hkv = a.n_kv_heads;
  cp.R = a.n_rows;
  cp.Nk = a.n_keys;
  cp.Lmax = a.theta_len;
  cp.mode = a.mode;
  cp.k = 1;
  cp.fit = 0;
  cp.alpha = 0.f;
  cp.sm_scale = 1.0f / sqrtf((float)a.head_dim);
  cp.q = a.q;
  cp.keys = a.keys;
  cp.row_len = a.row_len;
  cp.acc = nullptr;
  cp.count = nullptr;
  cp.theta = nullptr;
  cp.status = a.status;
  for (int h0 = 0; h0 < a.n_q_heads; h0 += Hp) {
    const int hp = (a.n_q_heads - h0) < Hp ? (a.n_q_heads - h0) : Hp;
    cp.h0 = p.h0 = h0;
    cp.Hp = p.Hp = hp;
    const long total = (long)a.n_seqs * hp * a.n_rows;
    if (a.dtype == TOPT_BF16) {
      e = a.head_dim == 128 ? mkc_scores<__nv_bfloat16, 128>(cp, total, ws, s)
                            : mkc_scores<__nv_bfloat16, 64>(cp, total, ws, s);
    } else {
      e = a.head_dim == 128 ? mkc_scores<float, 128>(cp, total, ws, s) : mkc_scores<float, 64>(cp, total, ws, s);
    }
    if (e != cudaSuccess) return e;
    if (a.mode == TOPT_POST) {
      mkc_softmax_kernel<<<(unsigned)total, kSelThreads, 0, s>>>(p);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    mkc_group_kernel<<<dim3((unsigned)a.theta_len, (unsigned)hp), kMkcThreads, sizeof(MkcSmem), s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  mkc_finalize_kernel<<<dim3((unsigned)a.n_q_heads, (unsigned)a.n_k), kFinThreads, 0, s>>>(p, a.theta);
  return cudaGetLastError();
}

cudaError_t select_kth_launch(const float* x, int32_t rows, int32_t stride, const int32_t* row_len,
                              int32_t k, float* out, int32_t* status, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  select_kth_kernel<<<rows, kSelThreads, 0, s>>>(x, stride, row_len, k, out, status);
  return cudaGetLastError();
}

}  // namespace topt

// Top-theta causal prefill: workspace layout and dispatch, and the CUDA-core
// variant (fp32 inputs) with the causal prefix means of V its VMC uses.  bf16
// inputs run on the tensor cores (prefill_tc.cu).
//
// [TopTheta] = "Top-Theta Attention: Sparsifying Transformers by Compensated
// Thresholding" (arXiv 2502.08363v2).  Row i of head h sees keys 0..i
// ([TopTheta §2.2, prefill phase]); every score is compared against the row's
// calibrated threshold theta[h][i] ([TopTheta §3, Fig. 1]).
//
// Two passes over the causal key tiles of a block of 16 query rows:
//   pass 1  row maximum m and Z = sum exp(a - m) (online);
//   pass 2  the threshold bound of each row (post-softmax needs m and Z),
//           P = exp(a - m) on kept elements, P.V only for tiles with at least
//           one kept element, then SDC [Eq. 4] and VMC [Eq. 5-7] with mu the
//           prefix mean of V rows 0..i.
// The prefix means come from prefix_mean_kernel (fp32, [B][Hkv][S][d]).
#include "common.cuh"
#include "internal.h"

namespace topt {
namespace {

constexpr int kRows = 16;     // query rows per CTA
constexpr int kKeys = 32;     // keys per tile
constexpr int kThreads = 128; // 8 threads per query row
constexpr int kMeanChunk = 64;

struct PrefillParams {
  int B, Hq, Hkv, S, Lmax, mode, sdc, vmc, mask_words;
  float gamma, sm_scale;
  const void* q;
  const void* k;
  const void* v;
  const float* theta;
  const float* e_tilde;  // offline E~ [Hq][Lmax] (pre-softmax, TOPT_SDC_OFFLINE)
  float* out;
  int32_t* kept;
  uint32_t* mask;
  unsigned long long* tiles;
  int32_t* status;
  float* mu;      // [B][Hkv][S][D] prefix means (when vmc)
  float* csum;    // [B][Hkv][nchunk][D] chunk sums
};

template <typename T, int D>
__global__ void __launch_bounds__(D) chunk_sum_kernel(const PrefillParams p) {
  const int c = blockIdx.x, bh = blockIdx.y, dd = threadIdx.x;
  const T* V = static_cast<const T*>(p.v) + (size_t)bh * p.S * D;
  const int lo = c * kMeanChunk, hi = min(lo + kMeanChunk, p.S);
  float s = 0.f;
  for (int i = lo; i < hi; ++i) s += to_f32<T>(V[(size_t)i * D + dd]);
  const int nchunk = (p.S + kMeanChunk - 1) / kMeanChunk;
  p.csum[((size_t)bh * nchunk + c) * D + dd] = s;
}

template <typename T, int D>
__global__ void __launch_bounds__(D) prefix_mean_kernel(const PrefillParams p) {
  const int c = blockIdx.x, bh = blockIdx.y, dd = threadIdx.x;
  const int nchunk = (p.S + kMeanChunk - 1) / kMeanChunk;
  const T* V = static_cast<const T*>(p.v) + (size_t)bh * p.S * D;
  float s = 0.f;
  for (int u = 0; u < c; ++u) s += p.csum[((size_t)bh * nchunk + u) * D + dd];
  const int lo = c * kMeanChunk, hi = min(lo + kMeanChunk, p.S);
  for (int i = lo; i < hi; ++i) {
    s += to_f32<T>(V[(size_t)i * D + dd]);
    p.mu[((size_t)bh * p.S + i) * D + dd] = s / (float)(i + 1);
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) prefill_simt_kernel(const PrefillParams p) {
  constexpr int NE = D / 8;  // output columns per thread
  __shared__ float Qs[kRows][D + 1];  // padded: 4 rows per warp read distinct banks
  __shared__ float Ks[kKeys][D + 1];
  __shared__ float Vs[kKeys][D];
  __shared__ float Ps[kRows][kKeys];
  __shared__ unsigned char Kf[kRows][kKeys];

  const int rb = blockIdx.x * kRows;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int G = p.Hq / p.Hkv;
  const int kvh = h / G;
  const int tid = threadIdx.x;
  const int r = tid >> 3;        // query row within the block
  const int cl = tid & 7;        // column lane within the row
  const int i_row = rb + r;
  const bool row_ok = i_row < p.S;
  const int last_row = min(rb + kRows, p.S) - 1;
  const int ntiles = last_row / kKeys + 1;

  const T* Q = static_cast<const T*>(p.q) + (((size_t)b * p.Hq + h) * p.S) * D;
  const T* K = static_cast<const T*>(p.k) + (((size_t)b * p.Hkv + kvh) * p.S) * D;
  const T* V = static_cast<const T*>(p.v) + (((size_t)b * p.Hkv + kvh) * p.S) * D;

  for (int idx = tid; idx < kRows * D; idx += kThreads) {
    const int rr = idx / D, dd = idx - rr * D;
    Qs[rr][dd] = (rb + rr < p.S) ? to_f32<T>(Q[(size_t)(rb + rr) * D + dd]) : 0.f;
  }

  auto load_tile = [&](int kt, bool with_v) {
    for (int idx = tid; idx < kKeys * D; idx += kThreads) {
      const int c = idx / D, dd = idx - c * D;
      const int j = kt * kKeys + c;
      const bool ok = j < p.S;
      Ks[c][dd] = ok ? to_f32<T>(K[(size_t)j * D + dd]) : 0.f;
      if (with_v) Vs[c][dd] = ok ? to_f32<T>(V[(size_t)j * D + dd]) : 0.f;
    }
  };
  auto score = [&](int c) {
    float acc = 0.f;
#pragma unroll 8
    for (int dd = 0; dd < D; ++dd) acc = fmaf(Qs[r][dd], Ks[c][dd], acc);
    return acc * p.sm_scale;
  };

  // ---- pass 1: row max and sum
  float m = -CUDART_INF_F, z = 0.f;
  for (int kt = 0; kt < ntiles; ++kt) {
    __syncthreads();
    load_tile(kt, false);
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kKeys / 8; ++u) {
      const int c = cl + 8 * u;
      const int j = kt * kKeys + c;
      if (row_ok && j <= i_row) ms_merge(m, z, score(c), 1.f);
    }
  }
#pragma unroll
  for (int off = 1; off < 8; off <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const float z2 = __shfl_xor_sync(0xffffffffu, z, off);
    ms_merge(m, z, m2, z2);
  }
  const int L = i_row + 1;
  const float th = row_ok ? p.theta[(size_t)h * p.Lmax + (min(L, p.Lmax) - 1)] : 0.f;
  const float bound = score_bound(p.mode, th, m, z);

  // ---- pass 2: threshold, P.V on tiles with survivors
  float acc[NE];
#pragma unroll
  for (int e = 0; e < NE; ++e) acc[e] = 0.f;
  float R = 0.f;
  int kt_cnt = 0;
  unsigned long long executed = 0;
  uint32_t* mrow = (p.mask && row_ok) ? p.mask + (((size_t)b * p.Hq + h) * p.S + i_row) * p.mask_words : nullptr;
  for (int kt = 0; kt < ntiles; ++kt) {
    __syncthreads();
    load_tile(kt, true);
    __syncthreads();
    bool any = false;
#pragma unroll
    for (int u = 0; u < kKeys / 8; ++u) {
      const int c = cl + 8 * u;
      const int j = kt * kKeys + c;
      float w = 0.f;
      bool keep = false;
      if (row_ok && j <= i_row) {
        const float a = score(c);
        keep = a >= bound;
        if (keep) w = __expf(a - m);
      }
      Ps[r][c] = w;
      Kf[r][c] = keep ? 1 : 0;
      R += w;
      kt_cnt += keep ? 1 : 0;
      any |= keep;
    }
    const int tile_any = __syncthreads_or(any);
    if (mrow && cl == 0) {
      uint32_t word = 0u;
      for (int c = 0; c < kKeys; ++c) word |= (uint32_t)Kf[r][c] << c;
      mrow[kt] = word;
    }
    if (tile_any) {
      ++executed;
      for (int c = 0; c < kKeys; ++c) {
        const float w = Ps[r][c];
#pragma unroll
        for (int e = 0; e < NE; ++e) acc[e] = fmaf(w, Vs[c][cl + 8 * e], acc[e]);
      }
    }
  }
  // mask words after the last causal tile
  if (mrow && cl == 0)
    for (int w = ntiles; w < p.mask_words; ++w) mrow[w] = 0u;

#pragma unroll
  for (int off = 1; off < 8; off <<= 1) {
    R += __shfl_xor_sync(0xffffffffu, R, off);
    kt_cnt += __shfl_xor_sync(0xffffffffu, kt_cnt, off);
  }
  if (row_ok) {
    float sc, beta;
    const float e_off = (p.mode == TOPT_PRE && p.sdc == TOPT_SDC_OFFLINE)
                            ? p.e_tilde[(size_t)h * p.Lmax + (min(L, p.Lmax) - 1)]
                            : 0.f;
    out_scale_beta(p.mode, p.sdc, p.gamma, th, m, z, R, L, kt_cnt, e_off, sc, beta);
    const size_t orow = ((size_t)b * p.Hq + h) * p.S + i_row;
    const float* mu = p.vmc ? p.mu + (((size_t)b * p.Hkv + kvh) * p.S + i_row) * D : nullptr;
#pragma unroll
    for (int e = 0; e < NE; ++e) {
      const int dd = cl + 8 * e;
      float o = acc[e] * sc;
      if (mu) o = fmaf(beta, mu[dd], o);
      p.out[orow * D + dd] = o;
    }
    if (p.kept && cl == 0) p.kept[orow] = kt_cnt;
  }
  if (p.tiles && tid == 0) {
    atomicAdd(p.tiles + 0, executed);
    atomicAdd(p.tiles + 1, (unsigned long long)ntiles);
  }
}

// Causal prefix means mu_i = mean(V_0..V_i) into p.mu.
template <typename T, int D>
cudaError_t launch_means(const PrefillParams& p, cudaStream_t s) {
  cudaError_t e;
  const int nchunk = (p.S + kMeanChunk - 1) / kMeanChunk;
  chunk_sum_kernel<T, D><<<dim3(nchunk, p.B * p.Hkv), D, 0, s>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  prefix_mean_kernel<T, D><<<dim3(nchunk, p.B * p.Hkv), D, 0, s>>>(p);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_td(const PrefillParams& p, void* const events[2], cudaStream_t s) {
  cudaError_t e;
  if (p.vmc && (e = launch_means<T, D>(p, s)) != cudaSuccess) return e;
  if ((e = record_event(events[0], s)) != cudaSuccess) return e;
  prefill_simt_kernel<T, D><<<dim3((p.S + kRows - 1) / kRows, p.Hq, p.B), kThreads, 0, s>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return record_event(events[1], s);
}

struct PrefillLayout {
  size_t mu, csum, v16, vmax, vexp, bsum, total;
};

PrefillLayout prefill_layout(const topt_prefill_args& a) {
  PrefillLayout l;
  const size_t bh = (size_t)a.batch * a.n_kv_heads;
  const size_t nchunk = (a.seq + kMeanChunk - 1) / kMeanChunk;
  const bool tc = a.dtype == TOPT_BF16;
  size_t off = 0;
  // CUDA-core path: prefix means and chunk sums (VMC)
  l.mu = off;   off += (!tc && a.vmc) ? align256(bh * a.seq * (size_t)a.head_dim * sizeof(float)) : 0;
  l.csum = off; off += (!tc && a.vmc) ? align256(bh * nchunk * (size_t)a.head_dim * sizeof(float)) : 0;
  // tensor-core path: fp16 copy of V, its per-head scale, block column sums (VMC)
  l.v16 = off;  off += tc ? align256(prefill_tc_v16_bytes(a)) : 0;
  l.vmax = off; off += tc ? align256(bh * sizeof(uint32_t)) : 0;
  l.vexp = off; off += tc ? align256(bh * sizeof(int32_t)) : 0;
  l.bsum = off; off += (tc && a.vmc) ? align256(prefill_tc_bsum_bytes(a)) : 0;
  l.total = off;
  return l;
}

}  // namespace

size_t prefill_workspace_bytes(const topt_prefill_args& a) { return prefill_layout(a).total; }

void prefill_tile_shape(const topt_prefill_args& a, int32_t* rows, int32_t* keys) {
  const bool tc = a.dtype == TOPT_BF16;
  *rows = tc ? prefill_tc_rows() : kRows;
  *keys = tc ? prefill_tc_keys(a.mode) : kKeys;
}

cudaError_t prefill_launch(const topt_prefill_args& a, cudaStream_t s, int withhold_k) {
  const PrefillLayout l = prefill_layout(a);
  char* ws = static_cast<char*>(a.workspace);
  PrefillParams p;
  p.B = a.batch;
  p.Hq = a.n_q_heads;
  p.Hkv = a.n_kv_heads;
  p.S = a.seq;
  p.Lmax = a.theta_len;
  p.mode = a.mode;
  p.sdc = a.sdc;
  p.vmc = a.vmc;
  p.mask_words = (a.seq + 31) / 32;
  p.gamma = a.gamma;
  p.sm_scale = 1.0f / sqrtf((float)a.head_dim);
  p.q = a.q;
  p.k = a.k;
  p.v = a.v;
  p.theta = a.theta;
  p.e_tilde = a.e_tilde;
  p.out = a.out;
  p.kept = a.kept;
  p.mask = a.mask;
  p.tiles = a.tiles;
  p.status = a.status;
  p.mu = (a.vmc && a.dtype != TOPT_BF16) ? reinterpret_cast<float*>(ws + l.mu) : nullptr;
  p.csum = (a.vmc && a.dtype != TOPT_BF16) ? reinterpret_cast<float*>(ws + l.csum) : nullptr;
  if (a.dtype == TOPT_BF16)
    return prefill_tc_run(a, ws + l.v16, reinterpret_cast<uint32_t*>(ws + l.vmax),
                          reinterpret_cast<int32_t*>(ws + l.vexp),
                          reinterpret_cast<float*>(ws + l.bsum), s, withhold_k);
  return a.head_dim == 128 ? launch_td<float, 128>(p, a.events, s) : launch_td<float, 64>(p, a.events, s);
}

}  // namespace topt

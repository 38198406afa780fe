// Top-theta GQA decode: one query token per sequence against its KV cache.
//
// [TopTheta] = "Top-Theta Attention: Sparsifying Transformers by Compensated
// Thresholding" (arXiv 2502.08363v2).  Decode is bound by reading the K cache
// ([TopTheta §2.2, generative decoding]); Top-theta's saving is that only the
// V rows that survive the threshold are read ([TopTheta §1, §4.6]).
//
// Two kernels per call, one (batch, KV head) "pair" = the G = Hq/Hkv query
// heads of a GQA group ([TopTheta §2.2, GQA]):
//
//  1. decode_scores_kernel: streams the pair's K rows once with 16-byte
//     loads (L2 evict-first) and computes the G x n score block
//     a = q K^T / sqrt(d) [Eq. 1] with one m16n8k16 bf16 MMA per 16 keys and
//     16 d (keys are the M side, the G query heads the N side).  Scores go
//     to a workspace array that stays L2-resident (G x 4 bytes per key, vs
//     2 d bytes of K), and each CTA writes per-head softmax partials (m, Z).
//  2. decode_select_kernel: merges the (m, Z) partials of the pair, turns
//     theta into a bound on the score (post-softmax: s >= theta <=>
//     a >= m + ln theta + ln Z), thresholds 32 keys per warp in registers,
//     ballots the per-head masks, ORs them into the group union, compacts
//     the union with a popcount prefix into shared memory, gathers only those
//     V rows and accumulates sum exp(a - m) V per head.  The last CTA of a
//     pair (atomic ticket, no waiting) combines the partial sums and applies
//     SDC [Eq. 4] and VMC [Eq. 5-7].
#include "common.cuh"
#include "internal.h"

namespace topt {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * kWarp;
constexpr int kCh1 = 512;                       // keys per score CTA
constexpr int kKeysPerWarp1 = kCh1 / kWarps;    // 128 = 8 MMA tiles of 16 keys
constexpr int kCh2 = 1024;                      // keys per select CTA
constexpr int kGatherUnroll = 8;                // V rows in flight per thread slot
constexpr int kMaxDevices = 64;

struct DecodeParams {
  int B, Hq, Hkv, Nmax, Lmax, mode, sdc, vmc;
  float gamma, sm_scale;
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const int32_t* seq_len;
  const float* theta;
  const float* mu;
  float* out;
  int32_t* kept;
  int32_t* vrows;
  uint32_t* mask;
  int32_t* status;
  int mask_words, nch1, nch2;
  // workspace
  float* logits;      // [pairs][G][Nmax]
  float2* stats;      // [pairs][nch1][G]
  float* part_num;    // [pairs][nch2][G][D]
  float* part_r;      // [pairs][nch2][G]
  int* part_kt;       // [pairs][nch2][G]
  int* part_nu;       // [pairs][nch2]
  unsigned* counter;  // [pairs]
};

struct DecodeLayout {
  size_t logits, stats, part_num, part_r, part_kt, part_nu, counter, total;
};

DecodeLayout decode_layout(const topt_decode_args& a) {
  const size_t pairs = (size_t)a.batch * a.n_kv_heads;
  const int G = a.n_q_heads / a.n_kv_heads;
  const size_t nch1 = (a.cache_len + kCh1 - 1) / kCh1;
  const size_t nch2 = (a.cache_len + kCh2 - 1) / kCh2;
  DecodeLayout l;
  size_t off = 0;
  l.logits = off;   off += align256(pairs * G * (size_t)a.cache_len * sizeof(float));
  l.stats = off;    off += align256(pairs * nch1 * G * sizeof(float2));
  l.part_num = off; off += align256(pairs * nch2 * G * (size_t)a.head_dim * sizeof(float));
  l.part_r = off;   off += align256(pairs * nch2 * G * sizeof(float));
  l.part_kt = off;  off += align256(pairs * nch2 * G * sizeof(int));
  l.part_nu = off;  off += align256(pairs * nch2 * sizeof(int));
  l.counter = off;  off += align256(pairs * sizeof(unsigned));
  l.total = off;
  return l;
}

// Online (max, sum) update with two new scores (either may be -inf).
__device__ __forceinline__ void ms_add2(float& m, float& z, float x0, float x1) {
  const float mt = fmaxf(x0, x1);
  if (mt == -CUDART_INF_F) return;
  const float mn = fmaxf(m, mt);
  z = z * __expf(m - mn) + __expf(x0 - mn) + __expf(x1 - mn);
  m = mn;
}

// ----------------------------------------------------------------------------
// Pass 1: scores and softmax partials.
// MMA fragment mapping.  Thread (g = lane/4, t = lane%4) loads, for key rows
// g and g+8 of a 16-key tile, the 16 bytes at d = 32p + 8t .. 32p + 8t + 7
// (p = 0 .. D/32-1), i.e. words w0..w3 of two bf16 each.  Because a dot
// product may visit d in any order, k-step s (0, 1) of slab p uses
//   A row g:   {w[2s], w[2s+1]} of row g      (columns 2t,2t+1 and 2t+8,2t+9)
//   A row g+8: {w[2s], w[2s+1]} of row g+8
//   B col g:   {w[2s], w[2s+1]} of the q row of head g
// which assigns the same 4 d values to the same k slots of A and B, so each
// MMA adds an exact partial dot product.  C then holds (key g, heads 2t, 2t+1)
// and (key g+8, heads 2t, 2t+1).
// ----------------------------------------------------------------------------
template <int D, int G>
__global__ void __launch_bounds__(kThreads) decode_scores_kernel(const DecodeParams p) {
  static_assert(D % 32 == 0 && G >= 1 && G <= 8, "shape");
  constexpr int NP = D / 32;
  const int pair = blockIdx.y;
  const int chunk = blockIdx.x;
  const int b = pair / p.Hkv;
  const int kvh = pair - b * p.Hkv;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int t = lane & 3;
  __shared__ float s_m[kWarps][8], s_z[kWarps][8];

  if (chunk == 0 && threadIdx.x == 0) p.counter[pair] = 0u;
  float2* st = p.stats + ((size_t)pair * p.nch1 + chunk) * G;
  const int L = p.seq_len[b];
  const int key_begin = chunk * kCh1;
  if (L < 1 || L > p.Nmax || key_begin >= L) {
    if ((L < 1 || L > p.Nmax) && chunk == 0 && threadIdx.x == 0) set_status(p.status, TOPT_EINVAL);
    if (threadIdx.x < G) st[threadIdx.x] = make_float2(-CUDART_INF_F, 0.f);
    return;
  }

  uint32_t qf[NP][4];
  if (g < G) {
    const __nv_bfloat16* qrow = p.q + ((size_t)b * p.Hq + kvh * G + g) * D;
#pragma unroll
    for (int pp = 0; pp < NP; ++pp) {
      const uint4 w = *reinterpret_cast<const uint4*>(qrow + 32 * pp + 8 * t);
      qf[pp][0] = w.x; qf[pp][1] = w.y; qf[pp][2] = w.z; qf[pp][3] = w.w;
    }
  } else {
#pragma unroll
    for (int pp = 0; pp < NP; ++pp) qf[pp][0] = qf[pp][1] = qf[pp][2] = qf[pp][3] = 0u;
  }

  const __nv_bfloat16* kbase = p.k + (size_t)pair * p.Nmax * D;
  float* lbase = p.logits + (size_t)pair * G * p.Nmax;
  const uint64_t pol = l2_evict_first_policy();
  const uint64_t keep_pol = l2_evict_last_policy();
  const float scale = p.sm_scale;
  const int h0 = 2 * t, h1 = 2 * t + 1;
  float m0 = -CUDART_INF_F, z0 = 0.f, m1 = -CUDART_INF_F, z1 = 0.f;

  const int wbeg = key_begin + warp * kKeysPerWarp1;
  const int wend = min(wbeg + kKeysPerWarp1, L);
  for (int tile = wbeg; tile < wend; tile += 32) {
    uint4 ka[2][NP], kb[2][NP];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int r0 = min(tile + 16 * u + g, L - 1);
      const int r1 = min(tile + 16 * u + g + 8, L - 1);
#pragma unroll
      for (int pp = 0; pp < NP; ++pp) {
        ka[u][pp] = ld_stream16(kbase + (size_t)r0 * D + 32 * pp + 8 * t, pol);
        kb[u][pp] = ld_stream16(kbase + (size_t)r1 * D + 32 * pp + 8 * t, pol);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int key0 = tile + 16 * u;
      if (key0 >= wend) break;
      float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int pp = 0; pp < NP; ++pp) {
        const uint32_t wa[4] = {ka[u][pp].x, ka[u][pp].y, ka[u][pp].z, ka[u][pp].w};
        const uint32_t wb[4] = {kb[u][pp].x, kb[u][pp].y, kb[u][pp].z, kb[u][pp].w};
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          const uint32_t af[4] = {wa[2 * s], wb[2 * s], wa[2 * s + 1], wb[2 * s + 1]};
          const uint32_t bf[2] = {qf[pp][2 * s], qf[pp][2 * s + 1]};
          mma_16816_bf16(c, af, bf);
        }
      }
      const int j0 = key0 + g;
      const int j1 = key0 + g + 8;
      const float a00 = j0 < wend ? c[0] * scale : -CUDART_INF_F;
      const float a01 = j0 < wend ? c[1] * scale : -CUDART_INF_F;
      const float a10 = j1 < wend ? c[2] * scale : -CUDART_INF_F;
      const float a11 = j1 < wend ? c[3] * scale : -CUDART_INF_F;
      if (h0 < G) {
        if (j0 < wend) st_hint_f32(lbase + (size_t)h0 * p.Nmax + j0, a00, keep_pol);
        if (j1 < wend) st_hint_f32(lbase + (size_t)h0 * p.Nmax + j1, a10, keep_pol);
        ms_add2(m0, z0, a00, a10);
      }
      if (h1 < G) {
        if (j0 < wend) st_hint_f32(lbase + (size_t)h1 * p.Nmax + j0, a01, keep_pol);
        if (j1 < wend) st_hint_f32(lbase + (size_t)h1 * p.Nmax + j1, a11, keep_pol);
        ms_add2(m1, z1, a01, a11);
      }
    }
  }

  // Merge over the 8 key rows (lane bits 2..4), then over warps.
  ms_warp_merge(m0, z0, 4);
  ms_warp_merge(m1, z1, 4);
  if (g == 0) {
    s_m[warp][h0] = m0; s_z[warp][h0] = z0;
    s_m[warp][h1] = m1; s_z[warp][h1] = z1;
  }
  __syncthreads();
  if (threadIdx.x < G) {
    float m = -CUDART_INF_F, z = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) ms_merge(m, z, s_m[w][threadIdx.x], s_z[w][threadIdx.x]);
    st[threadIdx.x] = make_float2(m, z);
  }
}

// ----------------------------------------------------------------------------
// Pass 2: threshold, compaction of the group union, V gather, SDC/VMC.
// Phase A: every warp loads the scores of its 8 groups of 32 keys at once,
// ballots the per-head masks, ORs them into the group union and writes the
// union's (key, weights) entries into a CTA-wide list at positions given by a
// popcount prefix (deterministic order).  Phase B: all threads gather the
// listed V rows, 16 bytes per lane, several rows in flight per thread.
// ----------------------------------------------------------------------------
constexpr int kGroupsPerWarp = kCh2 / (kWarps * kWarp);   // 8

template <int D, int G>
struct SelectSmem {
  int j[kCh2];                       // union keys of the CTA, in key order
  float w[kCh2][G];                  // exp(a - m) per head (0 if the head drops it)
  float acc[kWarps][G][D];           // per-warp partial sums (phase B reduction)
  float M[G], Z[G], T[G], th[G];
  float r[kWarps][G];
  int kt[kWarps][G];
  int cnt[kWarps];
  int last;
};

template <int D, int G>
__global__ void __launch_bounds__(kThreads) decode_select_kernel(const DecodeParams p) {
  constexpr int LPR = D / 8;           // lanes per V row (16 bytes each)
  constexpr int SLOTS = kThreads / LPR;  // V rows per CTA instruction
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SelectSmem<D, G>& sm = *reinterpret_cast<SelectSmem<D, G>*>(smem_raw);
  const int pair = blockIdx.y;
  const int chunk = blockIdx.x;
  const int b = pair / p.Hkv;
  const int kvh = pair - b * p.Hkv;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int L = p.seq_len[b];
  if (L < 1 || L > p.Nmax) return;  // reported by pass 1

  // Softmax statistics of the whole row, per head of the group.
  for (int h = warp; h < G; h += kWarps) {
    float m = -CUDART_INF_F, z = 0.f;
    for (int c = lane; c < p.nch1; c += kWarp) {
      const float2 v = p.stats[((size_t)pair * p.nch1 + c) * G + h];
      ms_merge(m, z, v.x, v.y);
    }
    ms_warp_merge(m, z, 1);
    if (lane == 0) {
      const float th = p.theta[(size_t)(kvh * G + h) * p.Lmax + (min(L, p.Lmax) - 1)];
      sm.M[h] = m;
      sm.Z[h] = z;
      sm.th[h] = th;
      sm.T[h] = score_bound(p.mode, th, m, z);
    }
  }
  __syncthreads();

  // ---- phase A: thresholds and union list
  const int c_begin = chunk * kCh2;
  const int c_end = min(c_begin + kCh2, L);
  const int w_begin = c_begin + warp * kGroupsPerWarp * kWarp;
  const float* lbase = p.logits + (size_t)pair * G * p.Nmax;
  const uint64_t pol = l2_evict_first_policy();
  float wv[kGroupsPerWarp][G];
#pragma unroll
  for (int gi = 0; gi < kGroupsPerWarp; ++gi) {
    const int j = w_begin + gi * kWarp + lane;
#pragma unroll
    for (int h = 0; h < G; ++h)
      wv[gi][h] = j < c_end ? ld_hint_f32(lbase + (size_t)h * p.Nmax + j, pol) : -CUDART_INF_F;
  }
  float Rl[G];
  int kt[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    Rl[h] = 0.f;
    kt[h] = 0;
  }
  unsigned uni[kGroupsPerWarp];
  int wcount = 0;
  uint32_t* mrow = p.mask ? p.mask + ((size_t)b * p.Hq + kvh * G) * p.mask_words : nullptr;
#pragma unroll
  for (int gi = 0; gi < kGroupsPerWarp; ++gi) {
    const int j0 = w_begin + gi * kWarp;
    const bool valid = j0 + lane < c_end;
    unsigned u = 0u;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float a = wv[gi][h];
      const bool keep = valid && (a >= sm.T[h]);
      wv[gi][h] = keep ? __expf(a - sm.M[h]) : 0.f;
      Rl[h] += wv[gi][h];
      const unsigned bal = __ballot_sync(0xffffffffu, keep);
      kt[h] += __popc(bal);
      u |= bal;
      if (mrow && lane == 0 && j0 < p.mask_words * 32)
        mrow[(size_t)h * p.mask_words + (j0 >> 5)] = bal;
    }
    uni[gi] = u;
    wcount += __popc(u);
  }
  if (lane == 0) sm.cnt[warp] = wcount;
  __syncthreads();
  int base = 0, total = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    base += (w < warp) ? sm.cnt[w] : 0;
    total += sm.cnt[w];
  }
#pragma unroll
  for (int gi = 0; gi < kGroupsPerWarp; ++gi) {
    if ((uni[gi] >> lane) & 1u) {
      const int pos = base + __popc(uni[gi] & ((1u << lane) - 1u));
      sm.j[pos] = w_begin + gi * kWarp + lane;
#pragma unroll
      for (int h = 0; h < G; ++h) sm.w[pos][h] = wv[gi][h];
    }
    base += __popc(uni[gi]);
  }
  __syncthreads();

  // ---- phase B: gather the listed V rows
  const int slot = threadIdx.x / LPR;
  const int dl = threadIdx.x % LPR;
  const __nv_bfloat16* vbase = p.v + (size_t)pair * p.Nmax * D + dl * 8;
  float acc[G][8];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[h][e] = 0.f;
  for (int r0 = 0; r0 < total; r0 += SLOTS * kGatherUnroll) {
    uint4 vv[kGatherUnroll];
#pragma unroll
    for (int u = 0; u < kGatherUnroll; ++u) {
      const int r = r0 + u * SLOTS + slot;
      if (r < total) vv[u] = ld_nc16(vbase + (size_t)sm.j[r] * D);
    }
#pragma unroll
    for (int u = 0; u < kGatherUnroll; ++u) {
      const int r = r0 + u * SLOTS + slot;
      if (r < total) {
        const float vf[8] = {bf16lo(vv[u].x), bf16hi(vv[u].x), bf16lo(vv[u].y), bf16hi(vv[u].y),
                             bf16lo(vv[u].z), bf16hi(vv[u].z), bf16lo(vv[u].w), bf16hi(vv[u].w)};
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float wh = sm.w[r][h];
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[h][e] = fmaf(wh, vf[e], acc[h][e]);
        }
      }
    }
  }

  // Reduce over the rows of a warp instruction, then over warps.
#pragma unroll
  for (int h = 0; h < G; ++h) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
#pragma unroll
      for (int off = LPR; off < kWarp; off <<= 1) acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], off);
    }
    Rl[h] = warp_sum(Rl[h]);
  }
  if (lane < LPR) {
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < 8; ++e) sm.acc[warp][h][dl * 8 + e] = acc[h][e];
  }
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      sm.r[warp][h] = Rl[h];
      sm.kt[warp][h] = kt[h];
    }
  }
  __syncthreads();

  const size_t pc = (size_t)pair * p.nch2 + chunk;
  if (total > 0) {
    for (int idx = threadIdx.x; idx < G * D; idx += kThreads) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) s += sm.acc[w][idx / D][idx % D];
      p.part_num[pc * G * D + idx] = s;
    }
  }
  if (threadIdx.x < G) {
    float r = 0.f;
    int k = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      r += sm.r[w][threadIdx.x];
      k += sm.kt[w][threadIdx.x];
    }
    p.part_r[pc * G + threadIdx.x] = r;
    p.part_kt[pc * G + threadIdx.x] = k;
  }
  if (threadIdx.x == 0) p.part_nu[pc] = total;

  // The last CTA of the pair to arrive combines (no CTA ever waits).
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(&p.counter[pair], 1u);
    sm.last = (prev == (unsigned)gridDim.x - 1u);
  }
  __syncthreads();
  if (!sm.last) return;
  __threadfence();

  for (int idx = threadIdx.x; idx < G * D; idx += kThreads) {
    const int h = idx / D;
    const int dd = idx - h * D;
    float num = 0.f, R = 0.f;
    int ktot = 0;
    for (int c = 0; c < p.nch2; ++c) {
      const size_t q = (size_t)pair * p.nch2 + c;
      if (__ldcg(p.part_nu + q) > 0) num += __ldcg(p.part_num + q * G * D + idx);
      R += __ldcg(p.part_r + q * G + h);
      ktot += __ldcg(p.part_kt + q * G + h);
    }
    float sc, beta;
    out_scale_beta(p.mode, p.sdc, p.gamma, sm.th[h], sm.M[h], sm.Z[h], R, L, ktot, sc, beta);
    float o = num * sc;
    if (p.vmc) o = fmaf(beta, p.mu[(size_t)pair * D + dd], o);
    const size_t row = (size_t)b * p.Hq + kvh * G + h;
    p.out[row * D + dd] = o;
    if (dd == 0 && p.kept) p.kept[row] = ktot;
  }
  if (threadIdx.x == 0) {
    int tot = 0;
    for (int c = 0; c < p.nch2; ++c) tot += __ldcg(p.part_nu + (size_t)pair * p.nch2 + c);
    if (p.vrows) p.vrows[pair] = tot;
    p.counter[pair] = 0u;
  }
}

template <int D, int G>
constexpr size_t select_smem_bytes() {
  return sizeof(SelectSmem<D, G>);
}

cudaError_t record(void* ev, cudaStream_t s) {
  return ev ? cudaEventRecord(static_cast<cudaEvent_t>(ev), s) : cudaSuccess;
}

template <int D, int G>
cudaError_t launch_dg(const DecodeParams& p, void* const* ev, cudaStream_t s) {
  const unsigned pairs = (unsigned)(p.B * p.Hkv);
  cudaError_t e;
  if ((e = record(ev[0], s)) != cudaSuccess) return e;
  decode_scores_kernel<D, G><<<dim3(p.nch1, pairs), kThreads, 0, s>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = record(ev[1], s)) != cudaSuccess) return e;
  constexpr size_t smem = select_smem_bytes<D, G>();
  static bool attr_set[kMaxDevices] = {};  // per device, per (D, G) instantiation
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    if ((e = cudaFuncSetAttribute(decode_select_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem)) != cudaSuccess)
      return e;
    attr_set[dev] = true;
  }
  decode_select_kernel<D, G><<<dim3(p.nch2, pairs), kThreads, smem, s>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return record(ev[2], s);
}

template <int D>
cudaError_t launch_d(const DecodeParams& p, int G, void* const* ev, cudaStream_t s) {
  switch (G) {
    case 1: return launch_dg<D, 1>(p, ev, s);
    case 2: return launch_dg<D, 2>(p, ev, s);
    case 3: return launch_dg<D, 3>(p, ev, s);
    case 4: return launch_dg<D, 4>(p, ev, s);
    case 5: return launch_dg<D, 5>(p, ev, s);
    case 6: return launch_dg<D, 6>(p, ev, s);
    case 7: return launch_dg<D, 7>(p, ev, s);
    case 8: return launch_dg<D, 8>(p, ev, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

size_t decode_workspace_bytes(const topt_decode_args& a) { return decode_layout(a).total; }

cudaError_t decode_launch(const topt_decode_args& a, cudaStream_t s) {
  const DecodeLayout l = decode_layout(a);
  char* ws = static_cast<char*>(a.workspace);
  DecodeParams p;
  p.B = a.batch;
  p.Hq = a.n_q_heads;
  p.Hkv = a.n_kv_heads;
  p.Nmax = a.cache_len;
  p.Lmax = a.theta_len;
  p.mode = a.mode;
  p.sdc = a.sdc;
  p.vmc = a.vmc;
  p.gamma = a.gamma;
  p.sm_scale = 1.0f / sqrtf((float)a.head_dim);
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.k = static_cast<const __nv_bfloat16*>(a.k_cache);
  p.v = static_cast<const __nv_bfloat16*>(a.v_cache);
  p.seq_len = a.seq_len;
  p.theta = a.theta;
  p.mu = a.mu;
  p.out = a.out;
  p.kept = a.kept;
  p.vrows = a.vrows;
  p.mask = a.mask;
  p.status = a.status;
  p.mask_words = (a.cache_len + 31) / 32;
  p.nch1 = (a.cache_len + kCh1 - 1) / kCh1;
  p.nch2 = (a.cache_len + kCh2 - 1) / kCh2;
  p.logits = reinterpret_cast<float*>(ws + l.logits);
  p.stats = reinterpret_cast<float2*>(ws + l.stats);
  p.part_num = reinterpret_cast<float*>(ws + l.part_num);
  p.part_r = reinterpret_cast<float*>(ws + l.part_r);
  p.part_kt = reinterpret_cast<int*>(ws + l.part_kt);
  p.part_nu = reinterpret_cast<int*>(ws + l.part_nu);
  p.counter = reinterpret_cast<unsigned*>(ws + l.counter);
  const int G = a.n_q_heads / a.n_kv_heads;
  if (a.head_dim == 128) return launch_d<128>(p, G, a.events, s);
  if (a.head_dim == 64) return launch_d<64>(p, G, a.events, s);
  return cudaErrorInvalidValue;
}

}  // namespace topt

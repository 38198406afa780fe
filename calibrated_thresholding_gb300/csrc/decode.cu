// Top-theta GQA decode: one query token per sequence against its KV cache.
//
// [TopTheta] = "Top-Theta Attention: Sparsifying Transformers by Compensated
// Thresholding" (arXiv 2502.08363v2).  Decode is bound by reading the K cache
// ([TopTheta §2.2, generative decoding]); Top-theta's saving is that only the
// V rows that survive the threshold are read ([TopTheta §1, §4.6]).  A "pair"
// is one (sequence, KV head) and its G = Hq/Hkv query heads ([TopTheta §2.2,
// GQA]).
//
// Two kernels per call, the second launched as a programmatic dependent of
// the first (it is scheduled while the first drains and waits for its data):
//
//  decode_scores_kernel (one resident wave, 4 warps per CTA).  Every pair's
//   valid keys form 16-key tiles, numbered pair after pair; warp w of the W
//   warps takes the contiguous tile range [T*w/W, T*(w+1)/W), so every warp
//   streams the same number of bytes.  Each warp stages its tiles in a
//   private shared-memory ring with cp.async (16 bytes per lane, 3 tiles in
//   flight), computes each 16-key x G-head score block with m16n8k16 bf16
//   MMAs (keys on the M side, query heads on the N side, one accumulator
//   chain per 32-wide d slab), writes a = q K^T / sqrt(d) [Eq. 1] to an
//   L2-resident workspace laid out [key][head] (one 8-byte store per lane and
//   key), and keeps a running softmax partial (m, Z) per head that it writes
//   once per run of tiles of one pair.
//  decode_select_kernel (one CTA per (pair, slice)).  Loads the slice's
//   scores (one vector load per key) while it merges the pair's (m, Z)
//   partials, turns theta into a bound on the score (post-softmax:
//   s >= theta <=> a >= m + ln theta + ln Z), ballots per-head masks of 32
//   keys per warp, ORs them into the group union, compacts the union into a
//   shared list by popcount prefix, gathers only those V rows (16-byte loads,
//   many rows in flight) and accumulates sum exp(a - m) V per head.  The last
//   slice of a pair to finish (atomic ticket, nothing waits) combines the
//   slices and applies SDC [Eq. 4] and VMC [Eq. 5-7].
//
// The workspace starts with a block of counters; the last user of a counter
// puts it back to zero, so a zero-filled workspace serves every later call.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace topt {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * kWarp;
constexpr int kTile = 16;                          // keys per MMA tile
constexpr int kStages = 3;                         // cp.async ring slots per warp
constexpr int kMaxBatch = 256;
constexpr int kMaxDevices = 64;

// V rows in flight per thread slot of the gather (register budget).
template <int G>
__host__ __device__ constexpr int gather_unroll() { return G <= 2 ? 8 : 4; }

// Most keys per select slice: 128-key groups, at most 40 staged scores and
// 24 groups per thread.  Calls use balanced slices of at most this length.
template <int G>
__host__ __device__ constexpr int slice_keys() { return kThreads * (40 / G < 24 ? 40 / G : 24); }

// Resident select CTAs per SM the register budget is sized for: 6 (80
// registers) keeps the short per-CTA latency chains overlapped; from G = 6 on
// the eight-head state spills at 80 registers, and 4 CTAs with 128 registers
// measured faster (G = 8: 229 against 258 us per decode call of the
// 70B-shaped workload; G = 4: 87.4 against 84.4 us, so it stays at 6).
template <int G>
__host__ __device__ constexpr int select_min_blocks() { return G >= 6 ? 4 : 6; }

// Score columns per key in the workspace: G rounded up to even (8-byte stores).
__host__ __device__ constexpr int score_cols(int G) { return G == 1 ? 1 : (G + 1) / 2 * 2; }

struct DecodeParams {
  int B, Hq, Hkv, Nmax, Lmax, mode, sdc, vmc;
  float gamma, sm_scale;
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const int32_t* seq_len;
  const float* theta;
  const float* e_tilde;  // offline E~ [Hq][Lmax] (pre-softmax, TOPT_SDC_OFFLINE)
  const float* mu;
  float* out;
  int32_t* kept;
  int32_t* vrows;
  uint32_t* mask;
  int32_t* status;
  int mask_words, spp, ipp, slice_len, lstride, score_warps;
  int gqa_min;        // TOPT_GQA_VOTE: heads of the group that must keep a key
  // workspace
  float* logits;      // [pairs][lstride][score_cols(G)]
  float2* stats;      // [pairs][spp][G]: a warp run's partial at the run's first tile
  float* part_num;    // [pairs][ipp][G][D]
  float* part_r;      // [pairs][ipp][G]
  int* part_kt;       // [pairs][ipp][G]
  int* part_nu;       // [pairs][ipp]
  unsigned* ticket;   // [pairs]: select slices finished (zero between calls)
  int* tstart;        // [B + 1]: first tile of each sequence, total (written each call)
};

// The workspace starts with a fixed-size block of counters, so a workspace
// reused across shapes keeps them in one place: zero before the first call,
// and every call leaves the ones it used at zero again.
constexpr size_t kCounterBytes = 128 * 1024;
constexpr int kMaxPairs = (int)(kCounterBytes / sizeof(unsigned)) - 2 * (kMaxBatch + 1);

struct DecodeLayout {
  size_t counters, logits, stats, part_num, part_r, part_kt, part_nu, total;
};

int logit_stride(int cache_len) { return (cache_len + 31) / 32 * 32; }

DecodeLayout decode_layout(const topt_decode_args& a, int ipp) {
  const size_t pairs = (size_t)a.batch * a.n_kv_heads;
  const int G = a.n_q_heads / a.n_kv_heads;
  const size_t spp = (a.cache_len + kTile - 1) / kTile + 1;
  DecodeLayout l;
  size_t off = 0;
  l.counters = off; off += kCounterBytes;
  l.logits = off;   off += align256(pairs * score_cols(G) * (size_t)logit_stride(a.cache_len) * sizeof(float));
  l.stats = off;    off += align256(pairs * spp * G * sizeof(float2));
  l.part_num = off; off += align256(pairs * ipp * G * (size_t)a.head_dim * sizeof(float));
  l.part_r = off;   off += align256(pairs * ipp * G * sizeof(float));
  l.part_kt = off;  off += align256(pairs * ipp * G * sizeof(int));
  l.part_nu = off;  off += align256(pairs * ipp * sizeof(int));
  l.total = off;
  return l;
}

// ------------------------------------------------------------ PTX helpers --
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
// 16-byte async copy global -> shared; src_bytes = 0 fills zeros and reads nothing.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, unsigned src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Online (max, sum) update with two new scores (either may be -inf).
__device__ __forceinline__ void ms_add2(float& m, float& z, float x0, float x1) {
  const float mt = fmaxf(x0, x1);
  if (mt == -CUDART_INF_F) return;
  const float mn = fmaxf(m, mt);
  z = z * __expf(m - mn) + __expf(x0 - mn) + __expf(x1 - mn);
  m = mn;
}

// Warp w's first tile in a split of T tiles over W warps, and the warp that
// owns tile tau in that split.
__device__ __forceinline__ int split_start(long T, long W, long w) { return (int)(T * w / W); }
__device__ __forceinline__ int split_owner(long T, long W, long tau) { return (int)(((tau + 1) * W - 1) / T); }

// ----------------------------------------------------------------------------
// Shared memory
// ----------------------------------------------------------------------------
template <int D>
struct ScoreSmem {
  int tstart[kMaxBatch + 1];  // first tile of each sequence; [B] = total
  int ntile[kMaxBatch];       // tiles per KV head of each sequence (0: invalid)
  int len[kMaxBatch];
  __align__(128) unsigned char slot[kWarps][kStages][kTile * D * 2];
};

template <int D, int G>
struct SelectSmem {
  float M[G], Z[G], T[G], th[G];
  int last;
  int cnt[kWarps];
  float m[kWarps][G], z[kWarps][G];
  float r[kWarps][G];
  int kt[kWarps][G];
  int j[slice_keys<G>()];  // union keys of the slice
  union {
    alignas(16) float sc[slice_keys<G>() * score_cols(G)];  // the slice's scores, [key][column]
    alignas(16) float w[slice_keys<G>()][G];                // then: exp(a - m) of the union
    float acc[kWarps][G][D];                                // then: per-warp sums
  } u;
};

// Tile bookkeeping shared by the producer and consumer of a warp's run.
struct TileCursor {
  int b, kvh, tile, nt, L;
  __device__ __forceinline__ int pair(int Hkv) const { return b * Hkv + kvh; }
};

template <int D>
__device__ __forceinline__ TileCursor cursor_at(const ScoreSmem<D>& sm, int B, int Hkv, int tau) {
  int lo = 0, hi = B - 1;  // last b with tstart[b] <= tau and tiles
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (sm.tstart[mid] <= tau) lo = mid;
    else hi = mid - 1;
  }
  while (lo < B - 1 && sm.ntile[lo] == 0) ++lo;  // sequences without tiles share tstart
  TileCursor c;
  c.b = lo;
  c.nt = sm.ntile[lo];
  const int rem = tau - sm.tstart[lo];
  c.kvh = rem / c.nt;
  c.tile = rem - c.kvh * c.nt;
  c.L = sm.len[lo];
  return c;
}

template <int D>
__device__ __forceinline__ void cursor_next(const ScoreSmem<D>& sm, int B, int Hkv, TileCursor& c) {
  if (++c.tile < c.nt) return;
  c.tile = 0;
  if (++c.kvh < Hkv) return;
  c.kvh = 0;
  do {
    ++c.b;
  } while (c.b < B && sm.ntile[c.b] == 0);
  if (c.b < B) {
    c.nt = sm.ntile[c.b];
    c.L = sm.len[c.b];
  }
}

// ----------------------------------------------------------------------------
// Scores.  MMA fragment mapping: thread (g = lane/4, t = lane%4) uses, for
// key rows g and g+8 of a tile, the 16 bytes at d = 32p + 8t .. +7
// (p = 0 .. D/32-1) as words w0..w3 (two bf16 each).  A dot product may visit
// d in any order, so k-step s (0, 1) of slab p uses
//   A row g:   {w[2s], w[2s+1]} of row g      (k = 2t,2t+1 and 2t+8,2t+9)
//   A row g+8: {w[2s], w[2s+1]} of row g+8
//   B col g:   {w[2s], w[2s+1]} of the q row of head g
// so every MMA adds an exact partial dot product; C then holds (key g, heads
// 2t, 2t+1) and (key g+8, heads 2t, 2t+1).
// ----------------------------------------------------------------------------
template <int D, int G>
__global__ void __launch_bounds__(kThreads, 4) decode_scores_kernel(const DecodeParams p) {
  constexpr int NP = D / 32;
  constexpr int GC = score_cols(G);
  constexpr unsigned kTileBytes = kTile * D * 2;
  constexpr int kChunks = kTileBytes / 16 / kWarp;  // 16-byte copies per lane per tile
  extern __shared__ __align__(128) unsigned char smem_raw[];
  ScoreSmem<D>& sm = *reinterpret_cast<ScoreSmem<D>*>(smem_raw);
  // The select kernel may be scheduled now; it waits for this grid's data.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // Tiles per sequence (every KV head of a sequence has the same length).
  if (threadIdx.x < kWarp) {
    const int lane = threadIdx.x;
    const int per = (p.B + kWarp - 1) / kWarp;
    int run = 0;
    for (int i = 0; i < per; ++i) {
      const int b = lane * per + i;
      if (b < p.B) {
        const int L = p.seq_len[b];
        sm.len[b] = L;
        int nt = 0;
        if (L >= 1 && L <= p.Nmax) nt = (L + kTile - 1) / kTile;
        else if (blockIdx.x == 0) set_status(p.status, TOPT_EINVAL);
        sm.ntile[b] = nt;
        run += nt * p.Hkv;
      }
    }
    int incl = run;
#pragma unroll
    for (int off = 1; off < kWarp; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    int acc = incl - run;
    for (int i = 0; i < per; ++i) {
      const int b = lane * per + i;
      if (b < p.B) {
        sm.tstart[b] = acc;
        acc += sm.ntile[b] * p.Hkv;
      }
    }
    if (lane == kWarp - 1) sm.tstart[p.B] = incl;
  }
  __syncthreads();
  if (blockIdx.x == 0)  // for the select kernel
    for (int i = threadIdx.x; i <= p.B; i += kThreads) p.tstart[i] = sm.tstart[i];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int t = lane & 3;
  const long T = sm.tstart[p.B];
  const long W = (long)gridDim.x * kWarps;
  const long gw = (long)blockIdx.x * kWarps + warp;
  const int t_begin = split_start(T, W, gw);
  const int t_end = split_start(T, W, gw + 1);
  if (t_begin >= t_end) return;

  unsigned char* ring = &sm.slot[warp][0][0];
  const uint32_t ring_s = smem_u32(ring);
  auto issue = [&](const TileCursor& c, int slot) {
    const char* src = reinterpret_cast<const char*>(p.k + ((size_t)c.pair(p.Hkv) * p.Nmax + c.tile * kTile) * D);
    const int rows = min(kTile, c.L - c.tile * kTile);
#pragma unroll
    for (int i = 0; i < kChunks; ++i) {
      const int off = (i * kWarp + lane) * 16;
      const int row = off / (D * 2);
      const bool ok = row < rows;
      cp_async16(ring_s + slot * kTileBytes + off, src + (ok ? off : 0), ok ? 16u : 0u);
    }
    cp_async_commit();
  };

  // Prologue: kStages-1 tiles in flight.
  TileCursor prod = cursor_at(sm, p.B, p.Hkv, t_begin);
  int issued = t_begin;
#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (issued < t_end) {
      issue(prod, s);
      cursor_next(sm, p.B, p.Hkv, prod);
      ++issued;
    } else {
      cp_async_commit();
    }
  }

  const float scale = p.sm_scale;
  const int h0 = 2 * t, h1 = 2 * t + 1;
  TileCursor c = cursor_at(sm, p.B, p.Hkv, t_begin);
  int cur_pair = -1;
  int run_first = 0;  // first global tile of the current pair
  int run_slot = 0;   // this warp's first tile of that pair, relative to run_first
  uint32_t qf[NP][4];
  float m0 = -CUDART_INF_F, z0 = 0.f, m1 = -CUDART_INF_F, z1 = 0.f;
  auto flush = [&](int pair) {  // this warp's partial of `pair`
    ms_warp_merge(m0, z0, 4);
    ms_warp_merge(m1, z1, 4);
    if (g == 0) {
      float2* st = p.stats + ((size_t)pair * p.spp + run_slot) * G;
      if (h0 < G) st[h0] = make_float2(m0, z0);
      if (h1 < G) st[h1] = make_float2(m1, z1);
    }
    m0 = -CUDART_INF_F;
    z0 = 0.f;
    m1 = -CUDART_INF_F;
    z1 = 0.f;
  };

  int slot = 0;
  for (int tau = t_begin; tau < t_end; ++tau) {
    // Keep kStages-1 copies ahead: refill the slot consumed last iteration.
    if (issued < t_end) {
      issue(prod, (slot + kStages - 1) % kStages);
      cursor_next(sm, p.B, p.Hkv, prod);
      ++issued;
    } else {
      cp_async_commit();
    }
    const int pair = c.pair(p.Hkv);
    if (pair != cur_pair) {
      if (cur_pair >= 0) flush(cur_pair);
      cur_pair = pair;
      run_first = sm.tstart[c.b] + c.kvh * c.nt;
      run_slot = tau - run_first;  // this warp's run of the pair starts at tau
      if (g < G) {
        const __nv_bfloat16* qrow = p.q + ((size_t)c.b * p.Hq + c.kvh * G + g) * D;
#pragma unroll
        for (int pp = 0; pp < NP; ++pp) {
          const uint4 w = *reinterpret_cast<const uint4*>(qrow + 32 * pp + 8 * t);
          qf[pp][0] = w.x; qf[pp][1] = w.y; qf[pp][2] = w.z; qf[pp][3] = w.w;
        }
      } else {
#pragma unroll
        for (int pp = 0; pp < NP; ++pp) qf[pp][0] = qf[pp][1] = qf[pp][2] = qf[pp][3] = 0u;
      }
    }
    cp_async_wait<kStages - 1>();
    __syncwarp();
    const unsigned char* tb = ring + slot * kTileBytes;
    uint4 ka[NP], kb[NP];
#pragma unroll
    for (int pp = 0; pp < NP; ++pp) {
      ka[pp] = *reinterpret_cast<const uint4*>(tb + (size_t)g * D * 2 + (32 * pp + 8 * t) * 2);
      kb[pp] = *reinterpret_cast<const uint4*>(tb + (size_t)(g + 8) * D * 2 + (32 * pp + 8 * t) * 2);
    }
    __syncwarp();  // the slot may be refilled from here on
    float cs[NP][4];
#pragma unroll
    for (int pp = 0; pp < NP; ++pp) {
      cs[pp][0] = cs[pp][1] = cs[pp][2] = cs[pp][3] = 0.f;
      const uint32_t wa[4] = {ka[pp].x, ka[pp].y, ka[pp].z, ka[pp].w};
      const uint32_t wb[4] = {kb[pp].x, kb[pp].y, kb[pp].z, kb[pp].w};
#pragma unroll
      for (int ss = 0; ss < 2; ++ss) {
        const uint32_t af[4] = {wa[2 * ss], wb[2 * ss], wa[2 * ss + 1], wb[2 * ss + 1]};
        const uint32_t bf[2] = {qf[pp][2 * ss], qf[pp][2 * ss + 1]};
        mma_16816_bf16(cs[pp], af, bf);
      }
    }
    float cc[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float v = cs[0][e];
#pragma unroll
      for (int pp = 1; pp < NP; ++pp) v += cs[pp][e];
      cc[e] = v;
    }
    const int key0 = c.tile * kTile;
    const int j0 = key0 + g;
    const int j1 = key0 + g + 8;
    const int L = c.L;
    const float a00 = j0 < L ? cc[0] * scale : -CUDART_INF_F;
    const float a01 = j0 < L ? cc[1] * scale : -CUDART_INF_F;
    const float a10 = j1 < L ? cc[2] * scale : -CUDART_INF_F;
    const float a11 = j1 < L ? cc[3] * scale : -CUDART_INF_F;
    float* lrow = p.logits + (size_t)pair * p.lstride * GC;
    if (G == 1) {
      if (t == 0) {
        if (j0 < L) lrow[j0] = a00;
        if (j1 < L) lrow[j1] = a10;
      }
    } else if (h0 < G) {
      if (j0 < L) *reinterpret_cast<float2*>(lrow + (size_t)j0 * GC + h0) = make_float2(a00, a01);
      if (j1 < L) *reinterpret_cast<float2*>(lrow + (size_t)j1 * GC + h0) = make_float2(a10, a11);
    }
    if (h0 < G) ms_add2(m0, z0, a00, a10);
    if (h1 < G) ms_add2(m1, z1, a01, a11);
    cursor_next(sm, p.B, p.Hkv, c);
    slot = (slot + 1) % kStages;
  }
  flush(cur_pair);
  cp_async_wait<0>();
}

// ----------------------------------------------------------------------------
// Select: one slice of one pair per CTA.
// ----------------------------------------------------------------------------
// POL is the GQA group policy [TopTheta §4.6]: TOPT_GQA_OWN (each head its own
// selection), TOPT_GQA_UNION (every head the group's union) or TOPT_GQA_VOTE
// (a key survives for a head that keeps it only if p.gqa_min heads keep it).
template <int D, int G, int POL>
__global__ void __launch_bounds__(kThreads, select_min_blocks<G>()) decode_select_kernel(const DecodeParams p) {
  constexpr int SK = slice_keys<G>();
  constexpr int NGRP = SK / kThreads;     // 32-key groups per warp
  constexpr int GC = score_cols(G);
  constexpr int kGatherUnroll = gather_unroll<G>();
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SelectSmem<D, G>& sm = *reinterpret_cast<SelectSmem<D, G>*>(smem_raw);
  const int item = blockIdx.x;
  const int pair = item / p.ipp;
  const int slice = item - pair * p.ipp;
  const int b = pair / p.Hkv;
  const int kvh = pair - b * p.Hkv;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Inputs of the call can be read before the score kernel has finished.
  const int L = p.seq_len[b];
  float th_pre = 0.f;
  if (L >= 1 && L <= p.Nmax && threadIdx.x < G)
    th_pre = p.theta[(size_t)(kvh * G + threadIdx.x) * p.Lmax + (min(L, p.Lmax) - 1)];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (L < 1 || L > p.Nmax) return;  // reported by the score kernel

  // Stage the slice's scores in shared memory (keys beyond the stride are
  // never copied; keys beyond L are ignored below).
  const int SL = p.slice_len;  // keys in every slice, a multiple of 128, <= SK
  const int s0 = slice * SL;
  {
    const char* src = reinterpret_cast<const char*>(p.logits + ((size_t)pair * p.lstride + s0) * GC);
    const int limit = (min(s0 + SL, p.lstride) - s0) * GC * 4;  // bytes inside the pair's row
    const uint32_t dst = smem_u32(sm.u.sc);
    for (int i = threadIdx.x; i * 16 < limit; i += kThreads) cp_async16(dst + i * 16, src + i * 16, 16u);
    cp_async_commit();
  }

  // Softmax statistics of the whole row, per head, from the warp partials.
  {
    const long T = p.tstart[p.B];
    const long W = p.score_warps;
    const int nt = (L + kTile - 1) / kTile;
    const long first = p.tstart[b] + (long)kvh * nt;
    const int w_first = split_owner(T, W, first);
    const int nslots = split_owner(T, W, first + nt - 1) - w_first + 1;
    float m[G], z[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m[h] = -CUDART_INF_F;
      z[h] = 0.f;
    }
    for (int c = threadIdx.x; c < nslots; c += kThreads) {
      // each warp covering the pair wrote one partial at its run's first tile;
      // warps with an empty range (more warps than tiles) wrote none
      const long ws = split_start(T, W, w_first + c);
      if (ws == split_start(T, W, w_first + c + 1)) continue;
      const int slot = (int)((ws > first ? ws : first) - first);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float2 v = __ldcg(p.stats + ((size_t)pair * p.spp + slot) * G + h);
        ms_merge(m[h], z[h], v.x, v.y);
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      ms_warp_merge(m[h], z[h], 1);
      if (lane == 0) {
        sm.m[warp][h] = m[h];
        sm.z[warp][h] = z[h];
      }
    }
    cp_async_wait<0>();
    __syncthreads();
    if (threadIdx.x < G) {
      const int h = threadIdx.x;
      float mm = -CUDART_INF_F, zz = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) ms_merge(mm, zz, sm.m[w][h], sm.z[w][h]);
      sm.M[h] = mm;
      sm.Z[h] = zz;
      sm.th[h] = th_pre;
      sm.T[h] = score_bound(p.mode, th_pre, mm, zz);
    }
    __syncthreads();
  }
  float T[G], M[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    T[h] = sm.T[h];
    M[h] = sm.M[h];
  }

  // Thresholds, masks and the union of the group: group gi of warp w is keys
  // s0 + gi*128 + w*32 + lane.
  uint32_t* mrow = p.mask ? p.mask + ((size_t)b * p.Hq + kvh * G) * p.mask_words : nullptr;
  float Rl[G];
  int kt[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    Rl[h] = 0.f;
    kt[h] = 0;
  }
  unsigned uni[NGRP];
  float wv[NGRP][G];
  int wcount = 0;
#pragma unroll
  for (int gi = 0; gi < NGRP; ++gi) {
    const int jl = gi * kThreads + warp * kWarp + lane;  // key within the slice
    const int j0 = s0 + gi * kThreads + warp * kWarp;
    const bool in_slice = gi * kThreads < SL;  // warp-uniform
    const bool valid = in_slice && s0 + jl < L;
    unsigned un = 0u;
    if constexpr (POL == TOPT_GQA_OWN) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float a = valid ? sm.u.sc[jl * GC + h] : -CUDART_INF_F;
        const bool keep = valid && (a >= T[h]);
        wv[gi][h] = keep ? __expf(a - M[h]) : 0.f;
        Rl[h] += wv[gi][h];
        const unsigned bal = __ballot_sync(0xffffffffu, keep);
        kt[h] += __popc(bal);
        un |= bal;
        if (mrow && lane == 0 && in_slice && j0 < p.mask_words * 32) mrow[(size_t)h * p.mask_words + (j0 >> 5)] = bal;
      }
    } else {
      // the heads' own decisions for this lane's key, then the group policy
      unsigned kb = 0u;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float a = valid ? sm.u.sc[jl * GC + h] : -CUDART_INF_F;
        if (valid && a >= T[h]) kb |= 1u << h;
      }
      if constexpr (POL == TOPT_GQA_UNION) {
        if (kb) kb = (1u << G) - 1u;
      } else {
        if (__popc(kb) < p.gqa_min) kb = 0u;
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const bool keep = (kb >> h) & 1u;
        const float a = keep ? sm.u.sc[jl * GC + h] : 0.f;
        wv[gi][h] = keep ? __expf(a - M[h]) : 0.f;
        Rl[h] += wv[gi][h];
        const unsigned bal = __ballot_sync(0xffffffffu, keep);
        kt[h] += __popc(bal);
        un |= bal;
        if (mrow && lane == 0 && in_slice && j0 < p.mask_words * 32) mrow[(size_t)h * p.mask_words + (j0 >> 5)] = bal;
      }
    }
    uni[gi] = un;
    wcount += __popc(un);
  }
  if (lane == 0) sm.cnt[warp] = wcount;
  __syncthreads();  // every score is in registers: the weights may overwrite them
  int base = 0, total = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    base += (w < warp) ? sm.cnt[w] : 0;
    total += sm.cnt[w];
  }
#pragma unroll
  for (int gi = 0; gi < NGRP; ++gi) {
    if ((uni[gi] >> lane) & 1u) {
      const int pos = base + __popc(uni[gi] & ((1u << lane) - 1u));
      sm.j[pos] = gi * kThreads + warp * kWarp + lane;
#pragma unroll
      for (int h = 0; h < G; ++h) sm.u.w[pos][h] = wv[gi][h];
    }
    base += __popc(uni[gi]);
  }
  __syncthreads();

  // Gather the union's V rows: LPR lanes per row, 16 bytes (8 d values) each.
  constexpr int LPR = D / 8;
  constexpr int RPI = kThreads / LPR;  // rows per CTA instruction
  const int rsub = threadIdx.x / LPR;
  const int dl = threadIdx.x % LPR;
  const __nv_bfloat16* vbase = p.v + ((size_t)pair * p.Nmax + s0) * D + dl * 8;
  float acc[G][8];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[h][e] = 0.f;
  for (int r0 = 0; r0 < total; r0 += RPI * kGatherUnroll) {
    uint4 vv[kGatherUnroll];
#pragma unroll
    for (int u = 0; u < kGatherUnroll; ++u) {
      const int r = r0 + u * RPI + rsub;
      if (r < total) vv[u] = ld_nc16(vbase + (size_t)sm.j[r] * D);
    }
#pragma unroll
    for (int u = 0; u < kGatherUnroll; ++u) {
      const int r = r0 + u * RPI + rsub;
      if (r < total) {
        const float vf[8] = {bf16lo(vv[u].x), bf16hi(vv[u].x), bf16lo(vv[u].y), bf16hi(vv[u].y),
                             bf16lo(vv[u].z), bf16hi(vv[u].z), bf16lo(vv[u].w), bf16hi(vv[u].w)};
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float wh = sm.u.w[r][h];
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
  __syncthreads();  // the weights are no longer read: acc may reuse them
  if (lane < LPR) {
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < 8; ++e) sm.u.acc[warp][h][dl * 8 + e] = acc[h][e];
  }
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      sm.r[warp][h] = Rl[h];
      sm.kt[warp][h] = kt[h];
    }
  }
  __syncthreads();

  const size_t pc = (size_t)pair * p.ipp + slice;
  if (total > 0) {
    for (int idx = threadIdx.x; idx < G * D; idx += kThreads) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) s += sm.u.acc[w][idx / D][idx % D];
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

  // The last slice of the pair to arrive combines (nothing waits).
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(&p.ticket[pair], 1u);
    sm.last = (prev == (unsigned)p.ipp - 1u);
  }
  __syncthreads();
  if (!sm.last) return;
  __threadfence();
  if (threadIdx.x == 0) p.ticket[pair] = 0u;  // every slice has arrived
  for (int idx = threadIdx.x; idx < G * D; idx += kThreads) {
    const int h = idx / D;
    const int dd = idx - h * D;
    float num = 0.f, R = 0.f;
    int ktot = 0;
    // independent L2 loads of several slices in flight
#pragma unroll 4
    for (int c = 0; c < p.ipp; ++c) {
      const size_t q = (size_t)pair * p.ipp + c;
      const int nu = __ldcg(p.part_nu + q);
      const float nv = __ldcg(p.part_num + q * G * D + idx);  // stale when nu == 0
      num += nu > 0 ? nv : 0.f;
      R += __ldcg(p.part_r + q * G + h);
      ktot += __ldcg(p.part_kt + q * G + h);
    }
    float scl, beta;
    const float e_off = (p.mode == TOPT_PRE && p.sdc == TOPT_SDC_OFFLINE)
                            ? p.e_tilde[(size_t)(kvh * G + h) * p.Lmax + (min(L, p.Lmax) - 1)]
                            : 0.f;
    out_scale_beta(p.mode, p.sdc, p.gamma, sm.th[h], sm.M[h], sm.Z[h], R, L, ktot, e_off, scl, beta);
    float o = num * scl;
    if (p.vmc) o = fmaf(beta, p.mu[(size_t)pair * D + dd], o);
    const size_t row = (size_t)b * p.Hq + kvh * G + h;
    p.out[row * D + dd] = o;
    if (dd == 0 && p.kept) p.kept[row] = ktot;
  }
  if (threadIdx.x == 0) {
    int tot = 0;
    for (int c = 0; c < p.ipp; ++c) tot += __ldcg(p.part_nu + (size_t)pair * p.ipp + c);
    if (p.vrows) p.vrows[pair] = tot;
  }
}

// Resident CTAs of the score grid, per device and instantiation (also sets
// both kernels' shared-memory limits once).
template <int D, int G>
cudaError_t grid_of(int& grid) {
  static int cached[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (cached[dev] == 0) {
    const size_t smem = sizeof(ScoreSmem<D>);
    if ((e = cudaFuncSetAttribute(decode_scores_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem)) != cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(decode_select_kernel<D, G, TOPT_GQA_OWN>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(SelectSmem<D, G>))) !=
        cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(decode_select_kernel<D, G, TOPT_GQA_UNION>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(SelectSmem<D, G>))) !=
        cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(decode_select_kernel<D, G, TOPT_GQA_VOTE>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(SelectSmem<D, G>))) !=
        cudaSuccess)
      return e;
    int per_sm = 0, sms = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_scores_kernel<D, G>, kThreads, smem)) !=
        cudaSuccess)
      return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    cached[dev] = per_sm * sms;
  }
  grid = cached[dev];
  return cudaSuccess;
}

// Fewest balanced slices of at most slice_keys<G>() keys.
int slices_per_pair(int cache_len, int G) {
  int sk = 0;
  switch (G) {
    case 1: sk = slice_keys<1>(); break;
    case 2: sk = slice_keys<2>(); break;
    case 3: sk = slice_keys<3>(); break;
    case 4: sk = slice_keys<4>(); break;
    case 5: sk = slice_keys<5>(); break;
    case 6: sk = slice_keys<6>(); break;
    case 7: sk = slice_keys<7>(); break;
    default: sk = slice_keys<8>(); break;
  }
  return (cache_len + sk - 1) / sk;
}

// Profiling events; under stream capture they become timing nodes of the graph.
template <int D, int G>
cudaError_t launch_dg(DecodeParams p, const topt_decode_args& a, cudaStream_t s) {
  int grid = 0;
  cudaError_t e;
  if ((e = grid_of<D, G>(grid)) != cudaSuccess) return e;
  const int pairs = p.B * p.Hkv;
  p.ipp = slices_per_pair(p.Nmax, G);
  p.slice_len = ((p.Nmax + p.ipp - 1) / p.ipp + kThreads - 1) / kThreads * kThreads;
  p.score_warps = grid * kWarps;
  const DecodeLayout l = decode_layout(a, p.ipp);
  if (a.workspace_bytes < l.total) return cudaErrorInvalidValue;
  char* ws = static_cast<char*>(a.workspace);
  p.logits = reinterpret_cast<float*>(ws + l.logits);
  p.stats = reinterpret_cast<float2*>(ws + l.stats);
  p.part_num = reinterpret_cast<float*>(ws + l.part_num);
  p.part_r = reinterpret_cast<float*>(ws + l.part_r);
  p.part_kt = reinterpret_cast<int*>(ws + l.part_kt);
  p.part_nu = reinterpret_cast<int*>(ws + l.part_nu);
  unsigned* counters = reinterpret_cast<unsigned*>(ws + l.counters);
  p.tstart = reinterpret_cast<int*>(counters);
  p.ticket = counters + 2 * (kMaxBatch + 1);
  if ((e = record_event(a.events[0], s)) != cudaSuccess) return e;
  decode_scores_kernel<D, G><<<grid, kThreads, sizeof(ScoreSmem<D>), s>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(pairs * p.ipp));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = sizeof(SelectSmem<D, G>);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if ((e = record_event(a.events[1], s)) != cudaSuccess) return e;
  if (a.gqa_policy == TOPT_GQA_UNION) e = cudaLaunchKernelEx(&cfg, decode_select_kernel<D, G, TOPT_GQA_UNION>, p);
  else if (a.gqa_policy == TOPT_GQA_VOTE) e = cudaLaunchKernelEx(&cfg, decode_select_kernel<D, G, TOPT_GQA_VOTE>, p);
  else e = cudaLaunchKernelEx(&cfg, decode_select_kernel<D, G, TOPT_GQA_OWN>, p);
  if (e != cudaSuccess) return e;
  return record_event(a.events[2], s);
}

template <int D>
cudaError_t launch_d(const DecodeParams& p, int G, const topt_decode_args& a, cudaStream_t s) {
  switch (G) {
    case 1: return launch_dg<D, 1>(p, a, s);
    case 2: return launch_dg<D, 2>(p, a, s);
    case 3: return launch_dg<D, 3>(p, a, s);
    case 4: return launch_dg<D, 4>(p, a, s);
    case 5: return launch_dg<D, 5>(p, a, s);
    case 6: return launch_dg<D, 6>(p, a, s);
    case 7: return launch_dg<D, 7>(p, a, s);
    case 8: return launch_dg<D, 8>(p, a, s);
  }
  return cudaErrorInvalidValue;
}

// Fixed scratch for topt_decode_noalloc: one file-scope device array (every
// GPU that loads the library holds it until exit).  Host code must not use the
// symbol as a device address; the address comes from cudaGetSymbolAddress.
constexpr size_t kNoAllocBytes = size_t(32) << 20;
__device__ __align__(256) unsigned char g_decode_scratch[kNoAllocBytes];

}  // namespace

size_t decode_noalloc_capacity() { return kNoAllocBytes; }

cudaError_t decode_noalloc_launch(const topt_decode_args& a, cudaStream_t s) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {  // once per device, with that device current
      void* ptr = nullptr;
      if ((e = cudaGetSymbolAddress(&ptr, g_decode_scratch)) != cudaSuccess) return e;
      addr[dev] = ptr;
    }
    base = addr[dev];
  }
  // The array keeps the previous call's contents: the counters must start at 0.
  if ((e = cudaMemsetAsync(base, 0, kCounterBytes, s)) != cudaSuccess) return e;
  topt_decode_args b = a;
  b.workspace = base;
  b.workspace_bytes = kNoAllocBytes;
  return decode_launch(b, s);
}

int decode_max_batch() { return kMaxBatch; }
int decode_max_pairs() { return kMaxPairs; }

size_t decode_workspace_bytes(const topt_decode_args& a) {
  const int G = a.n_q_heads / a.n_kv_heads;
  return decode_layout(a, slices_per_pair(a.cache_len, G)).total;
}

cudaError_t decode_launch(const topt_decode_args& a, cudaStream_t s) {
  if (a.batch > kMaxBatch || a.batch * a.n_kv_heads > kMaxPairs) return cudaErrorInvalidValue;
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
  p.e_tilde = a.e_tilde;
  p.mu = a.mu;
  p.out = a.out;
  p.kept = a.kept;
  p.vrows = a.vrows;
  p.mask = a.mask;
  p.status = a.status;
  p.mask_words = (a.cache_len + 31) / 32;
  p.gqa_min = a.gqa_min_heads;
  p.spp = (a.cache_len + kTile - 1) / kTile + 1;
  p.lstride = logit_stride(a.cache_len);
  p.ipp = 1;
  p.score_warps = 1;
  const int G = a.n_q_heads / a.n_kv_heads;
  if (a.head_dim == 128) return launch_d<128>(p, G, a, s);
  if (a.head_dim == 64) return launch_d<64>(p, G, a, s);
  return cudaErrorInvalidValue;
}

}  // namespace topt

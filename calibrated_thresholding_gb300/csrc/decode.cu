// Top-theta GQA decode: one query token per sequence against its KV cache.
//
// [TopTheta] = "Top-Theta Attention: Sparsifying Transformers by Compensated
// Thresholding" (arXiv 2502.08363v2).  Decode is bound by reading the K cache
// ([TopTheta §2.2, generative decoding]); Top-theta's saving is that only the
// V rows that survive the threshold are read ([TopTheta §1, §4.6]).  A "pair"
// is one (sequence, KV head) and its G = Hq/Hkv query heads ([TopTheta §2.2,
// GQA]).
//
// One kernel per call.  Every pair is served by one thread-block cluster of C
// CTAs (C = 1..16, chosen on the host so that the whole grid is resident at
// once); CTA c of the cluster owns 1/C of the pair's valid keys, in 32-key
// units (one mask word each), and each of its four warps owns a contiguous
// quarter of those units.  A CTA:
//
//  1. streams its K rows (cp.async ring per warp, 16 bytes per lane, evicted
//     first from L2), computes each 16-key x G-head score block with m16n8k16
//     bf16 MMAs (keys on M, query heads on N), writes a = q K^T / sqrt(d)
//     [Eq. 1] to an L2-resident scratch row and keeps a running softmax
//     partial (m, Z) per head;
//  2. publishes its (m, Z) in shared memory; after a cluster barrier every
//     CTA merges the C partials in rank order (identical bits everywhere) and
//     turns theta into a bound on the score (post-softmax:
//     s >= theta <=> a >= m + ln theta + ln Z);
//  3. per warp, re-reads its own units' scores, ballots the per-head masks,
//     applies the GQA group policy, compacts the group's union into a list
//     with each kept key's weights exp(a - m), gathers only those V rows and
//     accumulates sum exp(a - m) v per head; the score lines are dropped from
//     L2 once read (never written back);
//  4. reduces its warps' sums; after a second cluster barrier every CTA reads
//     the C partials of its share of the outputs through distributed shared
//     memory (summed in rank order), applies SDC [Eq. 4] and VMC [Eq. 5-7]
//     and writes them; a third barrier keeps every CTA's shared memory alive
//     until its peers have read it.
//
// Nothing waits on another grid or on a flag: the only waits are cp.async
// groups and cluster barriers that every CTA of a cluster reaches through the
// same control flow.  The kernel starts with griddepcontrol.wait (it may be
// launched before the previous kernel of the stream has finished) and lets
// the next kernel of the stream be scheduled once its K stream is done.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace topt {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * kWarp;
constexpr int kTile = 16;         // keys per MMA tile
constexpr int kUnit = 32;         // keys per unit: one mask word, one ballot
constexpr int kMaxDevices = 64;
constexpr int kMinUnitsPerCta = 8;  // a CTA of a cluster gets at least 256 keys
constexpr int kMaxCluster = 16;

// Score columns per key in the scratch: G rounded up to even (8-byte stores).
__host__ __device__ constexpr int score_cols(int G) { return G == 1 ? 1 : (G + 1) / 2 * 2; }
// Shared memory of one warp: its K ring while streaming (3 tiles of 16 keys
// at d = 128, 6 at d = 64), then, in the same bytes, its select state.
constexpr int kWarpSmem = 12288;
template <int D>
__host__ __device__ constexpr int ring_stages() { return kWarpSmem / (kTile * D * 2); }
// Select state: a ring of kBatches score batches (kBatches - 1 in flight) and
// the union list (key, G weights).  A batch is batch_units 32-key units.
constexpr int kBatches = 4;
template <int G>
__host__ __device__ constexpr int batch_units() { return score_cols(G) <= 2 ? 8 : (score_cols(G) <= 4 ? 4 : 2); }
template <int G>
__host__ __device__ constexpr int batch_floats() { return batch_units<G>() * kUnit * score_cols(G); }
template <int G>
__host__ __device__ constexpr int list_cap() {
  return (kWarpSmem - kBatches * batch_floats<G>() * 4) / (4 + 4 * G) / 32 * 32;
}
// Gather layout: VEC d-values (VEC * 2 bytes) per lane, G * VEC accumulators,
// 16 V rows in flight per warp.
template <int G>
__host__ __device__ constexpr int gather_vec() { return G <= 4 ? 8 : 4; }
template <int G>
__host__ __device__ constexpr int gather_unroll() { return G <= 4 ? 8 : 16; }

struct DecodeParams {
  int B, Hq, Hkv, Nmax, Lmax, mode, sdc, vmc, mask_words, gqa_min, nstride;
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
  float* scores;         // scratch [pairs][nstride][score_cols(G)]
};

size_t scratch_bytes(const topt_decode_args& a) {
  const size_t pairs = (size_t)a.batch * a.n_kv_heads;
  const int G = a.n_q_heads / a.n_kv_heads;
  const size_t nstride = (size_t)(a.cache_len + kUnit - 1) / kUnit * kUnit;
  return align256(pairs * nstride * score_cols(G) * sizeof(float));
}

// ------------------------------------------------------------ PTX helpers --
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
// 16-byte async copy global -> shared with an L2 eviction policy; src_bytes = 0
// fills zeros and reads nothing.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, unsigned src_bytes, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(dst), "l"(src),
               "r"(src_bytes), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void st_hint_v2(float* p, float a, float b, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v2.f32 [%0], {%1, %2}, %3;" ::"l"(p), "f"(a), "f"(b), "l"(pol)
               : "memory");
}
// Drops one 128-byte line of scratch from L2 without writing it back.
__device__ __forceinline__ void discard_line(const void* p) {
  asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster arrives; orders shared and global
// memory writes before the barrier with reads after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_peer_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ int ld_peer_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Online (max, sum) update with two new scores (either may be -inf).
__device__ __forceinline__ void ms_add2(float& m, float& z, float x0, float x1) {
  const float mt = fmaxf(x0, x1);
  if (mt == -CUDART_INF_F) return;
  const float mn = fmaxf(m, mt);
  z = z * __expf(m - mn) + __expf(x0 - mn) + __expf(x1 - mn);
  m = mn;
}

// VEC consecutive bf16 of a V row as floats (VEC = 8: 16 bytes, 4: 8 bytes).
template <int VEC>
__device__ __forceinline__ void ld_vrow(const __nv_bfloat16* p, uint32_t (&w)[VEC / 2]) {
  if constexpr (VEC == 8) {
    const uint4 v = ld_nc16(p);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else {
    uint2 v;
    asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    w[0] = v.x; w[1] = v.y;
  }
}

// ----------------------------------------------------------------------------
// Shared memory
// ----------------------------------------------------------------------------
template <int G>
union WarpSel {
  struct {
    float sc[kBatches][batch_floats<G>()];  // score batches [key][column]
    int j[list_cap<G>()];                   // union keys
    float w[list_cap<G>()][G];              // their weights exp(a - m), 0 for a head that drops the key
  } s;
  unsigned char raw[kWarpSmem];             // exactly one warp's ring
};

template <int D, int G>
struct DecodeSmem {
  union {
    unsigned char ring[kWarps][ring_stages<D>()][kTile * D * 2];  // K stream
    WarpSel<G> sel[kWarps];                                       // then, in each warp's own ring
    float acc[kWarps][G][D];                                      // then per-warp sums; acc[0] the CTA's
  } u;
  float wm[kWarps][G], wz[kWarps][G];  // per-warp softmax partials
  float cm[G], cz[G];                  // this CTA's partial, read by the cluster
  float M[G], Z[G], T[G], th[G];       // the row's statistics, bounds, thresholds
  float wr[kWarps][G];
  int wk[kWarps][G], wn[kWarps];
  float R[G];                          // this CTA's sums, read by the leader
  int KT[G], NU;
  float Rt[G];                         // the leader's totals
  int Kt[G];
};

// ----------------------------------------------------------------------------
// The kernel.  MMA fragment mapping of the score step: thread (g = lane/4,
// t = lane%4) uses, for key rows g and g+8 of a tile, the 16 bytes at
// d = 32p + 8t .. +7 (p = 0 .. D/32-1) as words w0..w3 (two bf16 each).  A dot
// product may visit d in any order, so k-step s (0, 1) of slab p uses
//   A row g:   {w[2s], w[2s+1]} of row g      (k = 2t,2t+1 and 2t+8,2t+9)
//   A row g+8: {w[2s], w[2s+1]} of row g+8
//   B col g:   {w[2s], w[2s+1]} of the q row of head g
// so every MMA adds an exact partial dot product; C then holds (key g, heads
// 2t, 2t+1) and (key g+8, heads 2t, 2t+1).
//
// POL is the GQA group policy [TopTheta §4.6]: TOPT_GQA_OWN (each head its own
// selection), TOPT_GQA_UNION (every head the group's union) or TOPT_GQA_VOTE
// (a key survives for a head that keeps it only if p.gqa_min heads keep it).
// ----------------------------------------------------------------------------
template <int D, int G, int POL>
__global__ void __launch_bounds__(kThreads, 4) decode_kernel(const DecodeParams p) {
  constexpr int NP = D / 32;
  constexpr int GC = score_cols(G);
  constexpr unsigned kTileBytes = kTile * D * 2;
  constexpr int kChunks = kTileBytes / 16 / kWarp;  // 16-byte copies per lane per tile
  constexpr int NS = ring_stages<D>();
  constexpr int BU = batch_units<G>();
  constexpr int BF = batch_floats<G>();
  constexpr int kChunksB = BF * 4 / 16 / kWarp;     // 16-byte copies per lane per score batch
  constexpr int UNR = gather_unroll<G>();
  constexpr int VEC = gather_vec<G>();
  constexpr int LPR = D / VEC;                      // lanes per V row
  constexpr int RPI = kWarp / LPR;                  // rows per warp instruction
  static_assert(sizeof(WarpSel<G>) == kWarpSmem && NS * kTileBytes == kWarpSmem, "one warp's shared memory");
  static_assert(BF * 4 % (16 * kWarp) == 0, "score batches copy in whole lane rounds");
  extern __shared__ __align__(128) unsigned char smem_raw[];
  DecodeSmem<D, G>& sm = *reinterpret_cast<DecodeSmem<D, G>*>(smem_raw);

  const uint32_t crank = cluster_rank();
  const uint32_t csize = cluster_size();
  const int pair = blockIdx.x / csize;
  const int b = pair / p.Hkv;
  const int kvh = pair - b * p.Hkv;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  grid_dep_wait();  // inputs may be written by the previous kernel of the stream
  const int L = p.seq_len[b];
  if (L < 1 || L > p.Nmax) {  // the whole cluster (same sequence) leaves together
    if (crank == 0 && threadIdx.x == 0) set_status(p.status, TOPT_EINVAL);
    return;
  }
  if (threadIdx.x < G) sm.th[threadIdx.x] = p.theta[(size_t)(kvh * G + threadIdx.x) * p.Lmax + (min(L, p.Lmax) - 1)];

  // Units of the row, of this CTA and of this warp.
  const int nunits = (L + kUnit - 1) / kUnit;
  const int u0 = (int)((long)nunits * crank / csize);
  const int u1 = (int)((long)nunits * (crank + 1) / csize);
  const int wu0 = u0 + (u1 - u0) * warp / kWarps;
  const int wu1 = u0 + (u1 - u0) * (warp + 1) / kWarps;

  uint32_t* mrow = p.mask ? p.mask + ((size_t)b * p.Hq + kvh * G) * p.mask_words : nullptr;
  if (mrow)  // words beyond the row: zero, shared out over the cluster
    for (int w = nunits + (int)crank * kThreads + threadIdx.x; w < p.mask_words; w += (int)csize * kThreads)
#pragma unroll
      for (int h = 0; h < G; ++h) mrow[(size_t)h * p.mask_words + w] = 0u;

  // ---------------------------------------------------------------- stream
  const int g = lane >> 2;
  const int t = lane & 3;
  const int h0 = 2 * t, h1 = 2 * t + 1;
  float* srow = p.scores + (size_t)pair * p.nstride * GC;
  {
    const __nv_bfloat16* kbase = p.k + (size_t)pair * p.Nmax * D;
    const uint64_t pol_k = l2_evict_first_policy();
    const uint64_t pol_s = l2_evict_last_policy();
    const int t0 = 2 * wu0;
    const int t1 = min(2 * wu1, (L + kTile - 1) / kTile);  // this warp's 16-key tiles
    const uint32_t ring_s = smem_u32(&sm.u.ring[warp][0][0]);
    auto issue = [&](int tile, int slot) {
      const char* src = reinterpret_cast<const char*>(kbase + (size_t)tile * kTile * D);
      const int rows = min(kTile, L - tile * kTile);
#pragma unroll
      for (int i = 0; i < kChunks; ++i) {
        const int off = (i * kWarp + lane) * 16;
        const bool ok = off / (D * 2) < rows;
        cp_async16(ring_s + slot * kTileBytes + off, src + (ok ? off : 0), ok ? 16u : 0u, pol_k);
      }
      cp_async_commit();
    };
#pragma unroll
    for (int s = 0; s < NS - 1; ++s) {
      if (t0 + s < t1) issue(t0 + s, s);
      else cp_async_commit();
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
    const float scale = p.sm_scale;
    float m0 = -CUDART_INF_F, z0 = 0.f, m1 = -CUDART_INF_F, z1 = 0.f;
    int slot = 0;
    for (int tile = t0; tile < t1; ++tile) {
      // keep NS-1 copies ahead: refill the slot consumed last iteration
      if (tile + NS - 1 < t1) issue(tile + NS - 1, (slot + NS - 1) % NS);
      else cp_async_commit();
      cp_async_wait<NS - 1>();
      __syncwarp();
      const unsigned char* tb = &sm.u.ring[warp][slot][0];
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
      const int j0 = tile * kTile + g;
      const int j1 = j0 + 8;
      const float a00 = j0 < L ? cc[0] * scale : -CUDART_INF_F;
      const float a01 = j0 < L ? cc[1] * scale : -CUDART_INF_F;
      const float a10 = j1 < L ? cc[2] * scale : -CUDART_INF_F;
      const float a11 = j1 < L ? cc[3] * scale : -CUDART_INF_F;
      if constexpr (G == 1) {
        if (t == 0) {
          if (j0 < L) st_hint_f32(srow + j0, a00, pol_s);
          if (j1 < L) st_hint_f32(srow + j1, a10, pol_s);
        }
      } else if (h0 < G) {
        if (j0 < L) st_hint_v2(srow + (size_t)j0 * GC + h0, a00, a01, pol_s);
        if (j1 < L) st_hint_v2(srow + (size_t)j1 * GC + h0, a10, a11, pol_s);
      }
      if (h0 < G) ms_add2(m0, z0, a00, a10);
      if (h1 < G) ms_add2(m1, z1, a01, a11);
      slot = (slot + 1) % NS;
    }
    cp_async_wait<0>();
    // this warp's partial per head: lanes with the same t hold the same heads
    ms_warp_merge(m0, z0, 4);
    ms_warp_merge(m1, z1, 4);
    if (g == 0) {
      if (h0 < G) { sm.wm[warp][h0] = m0; sm.wz[warp][h0] = z0; }
      if (h1 < G) { sm.wm[warp][h1] = m1; sm.wz[warp][h1] = z1; }
    }
  }
  // This warp's ring is drained: its first score batches go into the same
  // bytes now and travel while the cluster exchanges the row statistics.
  const int nbatch = (wu1 - wu0 + BU - 1) / BU;
  WarpSel<G>& ws = sm.u.sel[warp];
  const uint64_t pol_b = l2_evict_first_policy();
  auto fetch = [&](int bi) {  // batch bi of this warp's units into slot bi % kBatches
    const int bu = wu0 + bi * BU;
    const int bytes = min(BU, wu1 - bu) * kUnit * GC * 4;
    const char* src = reinterpret_cast<const char*>(srow + (size_t)bu * kUnit * GC);
    const uint32_t dst = smem_u32(&ws.s.sc[bi % kBatches][0]);
#pragma unroll
    for (int i = 0; i < kChunksB; ++i) {
      const int off = (i * kWarp + lane) * 16;
      const bool ok = off < bytes;
      cp_async16(dst + off, src + (ok ? off : 0), ok ? 16u : 0u, pol_b);
    }
  };
  __syncwarp();  // every lane's score stores come before any lane's copy of them
#pragma unroll
  for (int bi = 0; bi < kBatches - 1; ++bi) {
    if (bi < nbatch) fetch(bi);
    cp_async_commit();
  }
  grid_dep_launch();  // the K stream is done: the next kernel may be scheduled
  __syncthreads();
  if (threadIdx.x < G) {
    const int h = threadIdx.x;
    float mm = -CUDART_INF_F, zz = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) ms_merge(mm, zz, sm.wm[w][h], sm.wz[w][h]);
    sm.cm[h] = mm;
    sm.cz[h] = zz;
  }
  cluster_sync();  // #1: every CTA's partial is published

  // ---------------------------------------------------- row statistics
  if (threadIdx.x < G) {
    const int h = threadIdx.x;
    float pm[kMaxCluster], pz[kMaxCluster];
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r) {  // every load in flight before the first use
      if (r < (int)csize) {
        pm[r] = ld_peer_f32(peer_addr(&sm.cm[h], r));
        pz[r] = ld_peer_f32(peer_addr(&sm.cz[h], r));
      }
    }
    float mm = -CUDART_INF_F, zz = 0.f;
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r)  // rank order: the same bits in every CTA
      if (r < (int)csize) ms_merge(mm, zz, pm[r], pz[r]);
    sm.M[h] = mm;
    sm.Z[h] = zz;
    sm.T[h] = score_bound(p.mode, sm.th[h], mm, zz);
  }
  __syncthreads();

  // ------------------------------------------- threshold, union, V gather
  float acc[G][VEC];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[h][e] = 0.f;
  float Rl[G], Th[G], Mh[G];
  int kt[G];  // per lane: keys of its own that each head keeps
#pragma unroll
  for (int h = 0; h < G; ++h) {
    Rl[h] = 0.f;
    kt[h] = 0;
    Th[h] = sm.T[h];
    Mh[h] = sm.M[h];
  }
  int nsel = 0;
  int cnt = 0;  // entries in this warp's union list
  const int rsub = lane / LPR;
  const int dl = lane % LPR;
  const __nv_bfloat16* vbase = p.v + (size_t)pair * p.Nmax * D + dl * VEC;
  int* jl = ws.s.j;
  float (*wl)[G] = ws.s.w;
  auto gather = [&]() {  // accumulate the listed V rows, then empty the list
    __syncwarp();
    for (int r0 = 0; r0 < cnt; r0 += RPI * UNR) {
      uint32_t vv[UNR][VEC / 2];
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        const int r = r0 + u * RPI + rsub;
        if (r < cnt) ld_vrow<VEC>(vbase + (size_t)jl[r] * D, vv[u]);
      }
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        const int r = r0 + u * RPI + rsub;
        if (r < cnt) {
          float vf[VEC];
#pragma unroll
          for (int e = 0; e < VEC / 2; ++e) {
            vf[2 * e] = bf16lo(vv[u][e]);
            vf[2 * e + 1] = bf16hi(vv[u][e]);
          }
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float wh = wl[r][h];
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[h][e] = fmaf(wh, vf[e], acc[h][e]);
          }
        }
      }
    }
    nsel += cnt;
    cnt = 0;
    __syncwarp();
  };
  for (int bi = 0; bi < nbatch; ++bi) {
    if (bi + kBatches - 1 < nbatch) fetch(bi + kBatches - 1);  // into the slot consumed last
    cp_async_commit();
    cp_async_wait<kBatches - 1>();
    __syncwarp();
    const int bu = wu0 + bi * BU;
    const int nr = min(BU, wu1 - bu);
    // the batch is in shared memory: drop its scratch lines from L2
    for (int x = lane; x < nr * GC; x += kWarp) discard_line(srow + (size_t)bu * kUnit * GC + (size_t)x * 32);
    if (cnt + nr * kUnit > list_cap<G>()) gather();
    const float* sb = ws.s.sc[bi % kBatches];
    // The batch's decisions first (independent units), then the list.
    unsigned kb[BU], un[BU];
#pragma unroll
    for (int i = 0; i < BU; ++i) {
      const int j = (bu + i) * kUnit + lane;
      unsigned bits = 0u;
      if (i < nr && j < L) {
#pragma unroll
        for (int h = 0; h < G; ++h)
          if (sb[(i * kUnit + lane) * GC + h] >= Th[h]) bits |= 1u << h;
      }
      if constexpr (POL == TOPT_GQA_UNION) {
        if (bits) bits = (1u << G) - 1u;
      } else if constexpr (POL == TOPT_GQA_VOTE) {
        if (__popc(bits) < p.gqa_min) bits = 0u;
      }
      kb[i] = bits;
      un[i] = __ballot_sync(0xffffffffu, bits != 0u);
    }
    if (mrow) {  // per-head mask words
#pragma unroll
      for (int i = 0; i < BU; ++i) {
        if (i < nr) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const unsigned bal = __ballot_sync(0xffffffffu, (kb[i] >> h) & 1u);
            if (lane == 0) mrow[(size_t)h * p.mask_words + bu + i] = bal;
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < BU; ++i) {
      const unsigned bits = kb[i];
      if (bits) {
        const int pos = cnt + __popc(un[i] & ((1u << lane) - 1u));
        jl[pos] = (bu + i) * kUnit + lane;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const bool keep = (bits >> h) & 1u;
          const float w = keep ? __expf(sb[(i * kUnit + lane) * GC + h] - Mh[h]) : 0.f;
          kt[h] += keep ? 1 : 0;
          Rl[h] += w;
          wl[pos][h] = w;
        }
      }
      cnt += __popc(un[i]);
    }
    __syncwarp();  // the slot may be refilled from here on
  }
  cp_async_wait<0>();
  gather();

  // -------------------------------------------------- CTA partial sums
#pragma unroll
  for (int h = 0; h < G; ++h) {
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
#pragma unroll
      for (int off = LPR; off < kWarp; off <<= 1) acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], off);
    }
    Rl[h] = warp_sum(Rl[h]);
    kt[h] = warp_sum_int(kt[h]);
  }
  __syncthreads();  // every warp's list is consumed: acc may overwrite it
  if (lane < LPR) {
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < VEC; ++e) sm.u.acc[warp][h][dl * VEC + e] = acc[h][e];
  }
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      sm.wr[warp][h] = Rl[h];
      sm.wk[warp][h] = kt[h];
    }
    sm.wn[warp] = nsel;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * D; idx += kThreads) {
    const int h = idx / D, dd = idx - h * D;
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s += sm.u.acc[w][h][dd];
    sm.u.acc[0][h][dd] = s;  // read and written by this thread only
  }
  if (threadIdx.x < G) {
    float r = 0.f;
    int k = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      r += sm.wr[w][threadIdx.x];
      k += sm.wk[w][threadIdx.x];
    }
    sm.R[threadIdx.x] = r;
    sm.KT[threadIdx.x] = k;
  }
  if (threadIdx.x == 0) {
    int n = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) n += sm.wn[w];
    sm.NU = n;
  }
  cluster_sync();  // #2: the partials are visible to the leader

  // ------------------------- combine, SDC and VMC (shared out over the cluster)
  if (threadIdx.x < G) {
    const int h = threadIdx.x;
    float pr[kMaxCluster];
    int pk[kMaxCluster];
#pragma unroll
    for (int c = 0; c < kMaxCluster; ++c) {
      if (c < (int)csize) {
        pr[c] = ld_peer_f32(peer_addr(&sm.R[h], c));
        pk[c] = ld_peer_s32(peer_addr(&sm.KT[h], c));
      }
    }
    float r = 0.f;
    int k = 0;
#pragma unroll
    for (int c = 0; c < kMaxCluster; ++c) {
      if (c < (int)csize) {
        r += pr[c];
        k += pk[c];
      }
    }
    sm.Rt[h] = r;
    sm.Kt[h] = k;
  }
  if (crank == 0 && threadIdx.x == kWarp && p.vrows) {
    int n = 0;
    for (uint32_t c = 0; c < csize; ++c) n += ld_peer_s32(peer_addr(&sm.NU, c));
    p.vrows[pair] = n;
  }
  __syncthreads();
  {
    const int o0 = G * D * (int)crank / (int)csize;  // this CTA's share of the G x D outputs
    const int o1 = G * D * ((int)crank + 1) / (int)csize;
    for (int idx = o0 + threadIdx.x; idx < o1; idx += kThreads) {
      const int h = idx / D, dd = idx - h * D;
      float pn[kMaxCluster];
#pragma unroll
      for (int c = 0; c < kMaxCluster; ++c)
        if (c < (int)csize) pn[c] = ld_peer_f32(peer_addr(&sm.u.acc[0][h][dd], c));
      float num = 0.f;
#pragma unroll
      for (int c = 0; c < kMaxCluster; ++c)  // rank order
        if (c < (int)csize) num += pn[c];
      const float e_off = (p.mode == TOPT_PRE && p.sdc == TOPT_SDC_OFFLINE)
                              ? p.e_tilde[(size_t)(kvh * G + h) * p.Lmax + (min(L, p.Lmax) - 1)]
                              : 0.f;
      float scl, beta;
      out_scale_beta(p.mode, p.sdc, p.gamma, sm.th[h], sm.M[h], sm.Z[h], sm.Rt[h], L, sm.Kt[h], e_off, scl,
                     beta);
      float o = num * scl;
      if (p.vmc) o = fmaf(beta, p.mu[(size_t)pair * D + dd], o);
      const size_t row = (size_t)b * p.Hq + kvh * G + h;
      p.out[row * D + dd] = o;
      if (dd == 0 && p.kept) p.kept[row] = sm.Kt[h];
    }
  }
  cluster_sync();  // #3: shared memory stays alive until every peer has read it
}

// ----------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------
constexpr int kClusterSizes[] = {16, 8, 4, 2};

// Clusters of each size (16, 8, 4, 2) that can be resident at once, per
// device and instantiation (also sets the kernel's attributes once).
template <int D, int G, int POL>
cudaError_t cluster_capacity(const int*& cap) {
  static int cached[kMaxDevices][4] = {};
  static bool done[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!done[dev]) {
    auto kern = decode_kernel<D, G, POL>;
    const int smem = (int)sizeof(DecodeSmem<D, G>);
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
      return e;
    for (int i = 0; i < 4; ++i) {
      const int C = kClusterSizes[i];
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)(C * 64));
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = (unsigned)C;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, (const void*)kern, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();  // a size this device cannot schedule: not used
        n = 0;
      }
      cached[dev][i] = n;
    }
    done[dev] = true;
  }
  cap = cached[dev];
  return cudaSuccess;
}

// The largest cluster size whose clusters all fit at once, one per pair, with
// at least kMinUnitsPerCta units per CTA; 1 (plain CTAs, any number of waves)
// if none does.
int choose_cluster(const int* cap, long pairs, int Nmax) {
  const int units = (Nmax + kUnit - 1) / kUnit;
  for (int i = 0; i < 4; ++i) {
    const int C = kClusterSizes[i];
    if (units >= C * kMinUnitsPerCta && pairs <= cap[i]) return C;
  }
  return 1;
}

template <int D, int G, int POL>
cudaError_t launch_dgp(const DecodeParams& p, const topt_decode_args& a, cudaStream_t s) {
  const int* cap = nullptr;
  cudaError_t e;
  if ((e = cluster_capacity<D, G, POL>(cap)) != cudaSuccess) return e;
  const long pairs = (long)p.B * p.Hkv;
  const int C = choose_cluster(cap, pairs, p.Nmax);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(pairs * C));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = sizeof(DecodeSmem<D, G>);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if ((e = record_event(a.events[0], s)) != cudaSuccess) return e;
  if ((e = cudaLaunchKernelEx(&cfg, decode_kernel<D, G, POL>, p)) != cudaSuccess) return e;
  return record_event(a.events[1], s);
}

template <int D, int G>
cudaError_t launch_dg(const DecodeParams& p, const topt_decode_args& a, cudaStream_t s) {
  if (a.gqa_policy == TOPT_GQA_UNION) return launch_dgp<D, G, TOPT_GQA_UNION>(p, a, s);
  if (a.gqa_policy == TOPT_GQA_VOTE) return launch_dgp<D, G, TOPT_GQA_VOTE>(p, a, s);
  return launch_dgp<D, G, TOPT_GQA_OWN>(p, a, s);
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
long decode_max_pairs() { return 1L << 26; }

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
  // The kernel writes every scratch score before reading it: nothing in the
  // array has to be cleared between calls.
  topt_decode_args b = a;
  b.workspace = base;
  b.workspace_bytes = kNoAllocBytes;
  return decode_launch(b, s);
}

size_t decode_workspace_bytes(const topt_decode_args& a) { return scratch_bytes(a); }

cudaError_t decode_launch(const topt_decode_args& a, cudaStream_t s) {
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
  p.nstride = (a.cache_len + kUnit - 1) / kUnit * kUnit;
  if (a.workspace_bytes < scratch_bytes(a)) return cudaErrorInvalidValue;
  p.scores = static_cast<float*>(a.workspace);
  const int G = a.n_q_heads / a.n_kv_heads;
  if (a.head_dim == 128) return launch_d<128>(p, G, a, s);
  if (a.head_dim == 64) return launch_d<64>(p, G, a, s);
  return cudaErrorInvalidValue;
}

}  // namespace topt

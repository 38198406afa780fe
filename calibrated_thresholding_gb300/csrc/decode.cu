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
//  2. writes its (m, Z) into every CTA's shared memory; after a cluster
//     barrier every CTA merges the C partials in rank order (identical bits
//     everywhere) and turns theta into a bound on the score (post-softmax:
//     s >= theta <=> a >= m + ln theta + ln Z);
//  3. per warp, re-reads its own units' scores, ballots the per-head masks,
//     applies the GQA group policy, compacts the group's union into a list
//     with each kept key's weights exp(a - m), gathers only those V rows and
//     accumulates sum exp(a - m) v per head; the score lines are dropped from
//     L2 once read (never written back);
//  4. reduces its warps' sums and writes each slice of them into the shared
//     memory of the CTA that owns that slice of the outputs; after a second
//     cluster barrier every CTA sums the C partials of its slice (rank
//     order), applies SDC [Eq. 4] and VMC [Eq. 5-7] and writes the outputs.
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
// A union list entry packs the key (below 2^24) with its per-head keep bits.
constexpr int kKeyBits = 24;
constexpr unsigned kKeyMask = (1u << kKeyBits) - 1u;

// Score columns per key in the scratch: G rounded up to even (8-byte stores).
__host__ __device__ constexpr int score_cols(int G) { return G == 1 ? 1 : (G + 1) / 2 * 2; }
// Shared memory of one warp: its K ring while streaming (3 tiles of 16 keys
// at d = 128, 6 at d = 64), then, in the same bytes, its select state.
constexpr int kWarpSmem = 12288;
template <int D>
__host__ __device__ constexpr int ring_stages() { return kWarpSmem / (kTile * D * 2); }
// Select state: a ring of kBatches candidate batches (all in flight before the
// cluster barrier, each refilled once consumed) and the union list (key, G
// weights).  A batch holds batch_units * 32 candidates.
constexpr int kBatches = 3;
template <int G>
__host__ __device__ constexpr int batch_units() { return score_cols(G) <= 2 ? 8 : (score_cols(G) <= 4 ? 4 : 2); }
template <int G>
__host__ __device__ constexpr int batch_floats() { return batch_units<G>() * kUnit * score_cols(G); }
template <int G>
__host__ __device__ constexpr int list_cap() {
  return (kWarpSmem - kBatches * (batch_floats<G>() + batch_units<G>() * kUnit) * 4) / (4 + 4 * G) / 32 * 32;
}
// A post-softmax candidate needs a >= lse + ln theta - kLogSlack for the largest
// log-sum-exp that a warp of the cluster had reached over its keys so far; the
// slack keeps rounding from dropping a key the exact test keeps.
constexpr float kLogSlack = 1.0f / 1024.0f;
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
  float* scores;         // scratch [pairs][nstride][score_cols(G)]: each warp's candidates, compacted
  int32_t* cidx;         // scratch [pairs][nstride]: their key indices
};

size_t scores_bytes(const topt_decode_args& a) {
  const size_t pairs = (size_t)a.batch * a.n_kv_heads;
  const int G = a.n_q_heads / a.n_kv_heads;
  const size_t nstride = (size_t)(a.cache_len + kUnit - 1) / kUnit * kUnit;
  return align256(pairs * nstride * score_cols(G) * sizeof(float));
}
size_t scratch_bytes(const topt_decode_args& a) {
  const size_t pairs = (size_t)a.batch * a.n_kv_heads;
  const size_t nstride = (size_t)(a.cache_len + kUnit - 1) / kUnit * kUnit;
  return scores_bytes(a) + align256(pairs * nstride * sizeof(int32_t));
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
__device__ __forceinline__ void cp_async16_full(uint32_t dst, const void* src, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(pol)
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
__device__ __forceinline__ void st_peer_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void st_peer_s32(uint32_t addr, int v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_peer_v2(uint32_t addr, float a, float b) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
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

// Order-preserving map of floats to unsigned ints (for an integer max).
__device__ __forceinline__ unsigned fkey(float f) {
  const unsigned u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float funkey(unsigned k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
__device__ __forceinline__ void red_max_peer(uint32_t addr, unsigned v) {
  asm volatile("red.shared::cluster.max.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_peer_u32(uint32_t addr) {
  unsigned v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Bit g (g = 0..7) set iff any of bits 4g .. 4g+3 of b is set: from a ballot
// over lanes 4g + t to one bit per key row g of an MMA tile.
__device__ __forceinline__ unsigned quad_any(unsigned b) {
  b |= b >> 1;
  b |= b >> 2;
  b &= 0x11111111u;
  b = (b | (b >> 3)) & 0x03030303u;
  b = (b | (b >> 6)) & 0x000F000Fu;
  return (b | (b >> 12)) & 0xFFu;
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
    float sc[kBatches][batch_floats<G>()];          // candidate scores [entry][column]
    int ci[kBatches][batch_units<G>() * kUnit];     // candidate keys
    int j[list_cap<G>()];                           // union keys
    float w[list_cap<G>()][G];                      // their weights exp(a - m), 0 for a head that drops the key
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
  float M[G], Z[G], T[G], th[G];       // the row's statistics, bounds, thresholds
  float wr[kWarps][G];
  int wk[kWarps][G], wn[kWarps];
  float Rt[G];                         // the row's totals
  int Kt[G];
  unsigned clse[G];                    // leader only: the largest warp log-sum-exp so far (fkey)
  // written by the cluster's CTAs into each other's shared memory:
  float2 pstat[kMaxCluster][G];        // (m, Z) per head of every CTA
  float rnum[G * D];                   // partial sums of this CTA's share of the outputs, by source CTA
  float rR[kMaxCluster][G];            // R per head of every CTA
  int rK[kMaxCluster][G];              // kept keys per head of every CTA
  int rN[kMaxCluster];                 // (rank 0) union rows of every CTA
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
  constexpr int BK = BU * kUnit;                    // candidates per batch
  constexpr int kChunksB = BF * 4 / 16 / kWarp;     // 16-byte copies per lane per score batch
  constexpr int kChunksI = (BK * 4 / 16 + kWarp - 1) / kWarp;  // ... per index batch
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
  if (threadIdx.x < G) {
    sm.th[threadIdx.x] = p.theta[(size_t)(kvh * G + threadIdx.x) * p.Lmax + (min(L, p.Lmax) - 1)];
    sm.clse[threadIdx.x] = fkey(-CUDART_INF_F);
  }
  // the leader's bound slots are initialised before any CTA of the cluster
  // touches them (waited for after the first tile)
  cluster_arrive();

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
  // this warp's candidate region of the scratch: one entry per key it streams
  float* cscore = p.scores + ((size_t)pair * p.nstride + (size_t)wu0 * kUnit) * GC;
  int32_t* ckey = p.cidx + (size_t)pair * p.nstride + (size_t)wu0 * kUnit;
  int ncand = 0;  // candidates of this warp (warp-uniform)
  {
    const __nv_bfloat16* kbase = p.k + (size_t)pair * p.Nmax * D;
    const uint64_t pol_k = l2_evict_first_policy();
    const uint64_t pol_s = l2_evict_last_policy();
    const int t0 = 2 * wu0;
    const int t1 = min(2 * wu1, (L + kTile - 1) / kTile);  // this warp's 16-key tiles
    const uint32_t ring_s = smem_u32(&sm.u.ring[warp][0][0]);
    auto issue = [&](int tile, int slot) {
      const char* src = reinterpret_cast<const char*>(kbase + (size_t)tile * kTile * D) + lane * 16;
      const uint32_t dst = ring_s + slot * kTileBytes + lane * 16;
      const int rows = min(kTile, L - tile * kTile);
      if (rows == kTile) {  // a whole tile: no per-chunk size
#pragma unroll
        for (int i = 0; i < kChunks; ++i) cp_async16_full(dst + i * kWarp * 16, src + i * kWarp * 16, pol_k);
      } else {
#pragma unroll
        for (int i = 0; i < kChunks; ++i) {
          const int off = (i * kWarp + lane) * 16;
          const bool ok = off / (D * 2) < rows;
          cp_async16(dst + i * kWarp * 16, src - lane * 16 + (ok ? off : 0), ok ? 16u : 0u, pol_k);
        }
      }
      cp_async_commit();
    };
#pragma unroll
    for (int s = 0; s < NS; ++s) {  // every slot in flight
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
    const bool pre = p.mode == TOPT_PRE;
    const float th0 = h0 < G ? sm.th[h0] : 0.f;
    const float th1 = h1 < G ? sm.th[h1] : 0.f;
    // every key is a candidate of a post-softmax head whose threshold is <= 0
    const bool all0 = !pre && !(th0 > 0.f), all1 = !pre && !(th1 > 0.f);
    const float lth0 = all0 ? 0.f : __logf(th0) - kLogSlack, lth1 = all1 ? 0.f : __logf(th1) - kLogSlack;
    // cluster-wide bound: slots of heads h0, h1 in the leader CTA
    const uint32_t slot0 = peer_addr(&sm.clse[h0 < G ? h0 : 0], 0);
    const uint32_t slot1 = peer_addr(&sm.clse[h1 < G ? h1 : 0], 0);
    float bl0 = -CUDART_INF_F, bl1 = -CUDART_INF_F;        // candidate bounds on a (post-softmax)
    unsigned pend0 = fkey(-CUDART_INF_F), pend1 = pend0;  // the cluster's largest lse, last read
    bool waited = false;
    float m0 = -CUDART_INF_F, z0 = 0.f, m1 = -CUDART_INF_F, z1 = 0.f;
    int slot = 0;
    for (int tile = t0; tile < t1; ++tile) {
      cp_async_wait<NS - 1>();  // this tile has landed
      __syncwarp();
      const unsigned char* tb = &sm.u.ring[warp][slot][0];
      uint4 ka[NP], kb[NP];
#pragma unroll
      for (int pp = 0; pp < NP; ++pp) {
        ka[pp] = *reinterpret_cast<const uint4*>(tb + (size_t)g * D * 2 + (32 * pp + 8 * t) * 2);
        kb[pp] = *reinterpret_cast<const uint4*>(tb + (size_t)(g + 8) * D * 2 + (32 * pp + 8 * t) * 2);
      }
      __syncwarp();  // the tile is in registers: refill its slot before the math
      if (tile + NS < t1) issue(tile + NS, slot);
      else cp_async_commit();
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
      ms_add2(m0, z0, a00, a10);  // this lane's partial of heads h0, h1
      ms_add2(m1, z1, a01, a11);
      // Candidates: a key some head may keep.  The log-sum-exp of any subset
      // of the row's keys is at most the row's, so a key below such a bound
      // [post: s >= theta <=> a >= m + ln Z + ln theta] fails the row's bound
      // too; pre-softmax compares with theta itself.
      bool c0 = false, c1 = false;
      if (h0 < G) {
        c0 = pre ? a00 >= th0 : a00 >= bl0;
        c1 = pre ? a10 >= th0 : a10 >= bl0;
      }
      if (h1 < G) {
        c0 = c0 || (pre ? a01 >= th1 : a01 >= bl1);
        c1 = c1 || (pre ? a11 >= th1 : a11 >= bl1);
      }
      const int done = tile - t0 + 1;
      if (!pre && (done <= 2 || (done & 3) == 0)) {
        // Refresh the bound from this warp's log-sum-exp so far and the largest
        // one the cluster had published at the previous refresh; publish ours.
        if (!waited) {
          cluster_wait();
          waited = true;
        }
        float wm0 = m0, wz0 = z0, wm1 = m1, wz1 = z1;
        ms_warp_merge(wm0, wz0, 4);
        ms_warp_merge(wm1, wz1, 4);
        const float own0 = wm0 + __logf(wz0), own1 = wm1 + __logf(wz1);
        const float cl0 = __shfl_sync(0xffffffffu, funkey(pend0), t);
        const float cl1 = __shfl_sync(0xffffffffu, funkey(pend1), t);
        bl0 = all0 ? -CUDART_INF_F : fmaxf(own0, cl0) + lth0;
        bl1 = all1 ? -CUDART_INF_F : fmaxf(own1, cl1) + lth1;
        if (g == 0) {
          if (h0 < G) {
            red_max_peer(slot0, fkey(own0));
            pend0 = ld_peer_u32(slot0);
          }
          if (h1 < G) {
            red_max_peer(slot1, fkey(own1));
            pend1 = ld_peer_u32(slot1);
          }
        }
      }
      const unsigned tmask = quad_any(__ballot_sync(0xffffffffu, c0 && j0 < L)) |
                             (quad_any(__ballot_sync(0xffffffffu, c1 && j1 < L)) << 8);
      if (tmask) {  // warp-uniform: store the tile's candidates, compacted in key order
        const bool k0 = (tmask >> g) & 1u, k1 = (tmask >> (g + 8)) & 1u;
        const int r0 = ncand + __popc(tmask & ((1u << g) - 1u));
        const int r1 = ncand + __popc(tmask & ((1u << (g + 8)) - 1u));
        if constexpr (G == 1) {
          if (t == 0) {
            if (k0) st_hint_f32(cscore + r0, a00, pol_s);
            if (k1) st_hint_f32(cscore + r1, a10, pol_s);
          }
        } else if (h0 < G) {
          if (k0) st_hint_v2(cscore + (size_t)r0 * GC + h0, a00, a01, pol_s);
          if (k1) st_hint_v2(cscore + (size_t)r1 * GC + h0, a10, a11, pol_s);
        }
        if (t == 0) {
          if (k0) ckey[r0] = j0;
          if (k1) ckey[r1] = j1;
        }
        ncand += __popc(tmask);
      }
      slot = (slot + 1) % NS;
    }
    cp_async_wait<0>();
    if (!waited) cluster_wait();  // pairs the arrive at the start
    ms_warp_merge(m0, z0, 4);     // this warp's partial per head: lanes with the same t
    ms_warp_merge(m1, z1, 4);
    if (g == 0) {
      if (h0 < G) { sm.wm[warp][h0] = m0; sm.wz[warp][h0] = z0; }
      if (h1 < G) { sm.wm[warp][h1] = m1; sm.wz[warp][h1] = z1; }
    }
  }
  // This warp's ring is drained: its first candidate batches go into the same
  // bytes now and travel while the cluster exchanges the row statistics.
  const int nbatch = (ncand + BK - 1) / BK;
  WarpSel<G>& ws = sm.u.sel[warp];
  const uint64_t pol_b = l2_evict_first_policy();
  auto fetch = [&](int bi) {  // candidates [bi * BK, ..) into slot bi % kBatches
    const int n = min(BK, ncand - bi * BK);
    const int sbytes = n * GC * 4, ibytes = n * 4;
    const char* src = reinterpret_cast<const char*>(cscore + (size_t)bi * BK * GC);
    const uint32_t dst = smem_u32(&ws.s.sc[bi % kBatches][0]);
#pragma unroll
    for (int i = 0; i < kChunksB; ++i) {
      const int off = (i * kWarp + lane) * 16;
      const int nb = min(max(sbytes - off, 0), 16);  // the rest of the 16 bytes reads as 0
      cp_async16(dst + off, src + (nb ? off : 0), (unsigned)nb, pol_b);
    }
    const char* isrc = reinterpret_cast<const char*>(ckey + (size_t)bi * BK);
    const uint32_t idst = smem_u32(&ws.s.ci[bi % kBatches][0]);
#pragma unroll
    for (int i = 0; i < kChunksI; ++i) {
      const int off = (i * kWarp + lane) * 16;
      if (off < BK * 4) {
        const int nb = min(max(ibytes - off, 0), 16);
        cp_async16(idst + off, isrc + (nb ? off : 0), (unsigned)nb, pol_b);
      }
    }
  };
  __syncwarp();  // every lane's candidate stores come before any lane's copy of them
#pragma unroll
  for (int bi = 0; bi < kBatches; ++bi) {
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
    for (uint32_t r = 0; r < csize; ++r) st_peer_v2(peer_addr(&sm.pstat[crank][h], r), mm, zz);
  }
  cluster_sync();  // #1: every CTA's partial is in every CTA's shared memory

  // ---------------------------------------------------- row statistics
  if (threadIdx.x < G) {
    const int h = threadIdx.x;
    float mm = -CUDART_INF_F, zz = 0.f;
    for (uint32_t r = 0; r < csize; ++r)  // rank order: the same bits in every CTA
      ms_merge(mm, zz, sm.pstat[r][h].x, sm.pstat[r][h].y);
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
  // Accumulates union list entry r of warp w: its V row times each head's
  // weight; with a mask, one lane of the row sets the row's kept bits.
  auto gather_rows = [&](int w, int r0, int n) {  // entries [r0, r0 + RPI * UNR) below n
    const int* jw = sm.u.sel[w].s.j;
    const float (*ww)[G] = sm.u.sel[w].s.w;
    uint32_t vv[UNR][VEC / 2];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int r = r0 + u * RPI + rsub;
      if (r < n) ld_vrow<VEC>(vbase + (size_t)(jw[r] & kKeyMask) * D, vv[u]);
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int r = r0 + u * RPI + rsub;
      if (r < n) {
        float vf[VEC];
#pragma unroll
        for (int e = 0; e < VEC / 2; ++e) {
          vf[2 * e] = bf16lo(vv[u][e]);
          vf[2 * e + 1] = bf16hi(vv[u][e]);
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float wh = ww[r][h];
#pragma unroll
          for (int e = 0; e < VEC; ++e) acc[h][e] = fmaf(wh, vf[e], acc[h][e]);
        }
        if (mrow && dl == 0) {
          const unsigned jj = (unsigned)jw[r];
          const unsigned key = jj & kKeyMask;
#pragma unroll
          for (int h = 0; h < G; ++h)
            if ((jj >> (kKeyBits + h)) & 1u) atomicOr(&mrow[(size_t)h * p.mask_words + (key >> 5)], 1u << (key & 31));
        }
      }
    }
  };
  auto gather = [&]() {  // this warp's own list, when it is full
    __syncwarp();
    for (int r0 = 0; r0 < cnt; r0 += RPI * UNR) gather_rows(warp, r0, cnt);
    nsel += cnt;
    cnt = 0;
    __syncwarp();
  };
  if (mrow) {  // this warp's mask words: zero, then the kept bits of its candidates
    for (int x = lane; x < (wu1 - wu0) * G; x += kWarp)
      mrow[(size_t)(x / (wu1 - wu0)) * p.mask_words + wu0 + x % (wu1 - wu0)] = 0u;
    __syncwarp();
  }
  for (int bi = 0; bi < nbatch; ++bi) {
    cp_async_wait<kBatches - 1>();  // batches 0..bi have landed
    __syncwarp();
    const int n = min(BK, ncand - bi * BK);
    // the batch is in shared memory: drop its scratch lines from L2
    {
      const char* sb0 = reinterpret_cast<const char*>(cscore + (size_t)bi * BK * GC);
      const char* ib0 = reinterpret_cast<const char*>(ckey + (size_t)bi * BK);
      const int lines = (n * GC * 4) / 128;  // whole lines only (a partial one ends the candidates)
      const int ilines = (n * 4) / 128;
      for (int x = lane; x < lines + ilines; x += kWarp)
        discard_line(x < lines ? sb0 + (size_t)x * 128 : ib0 + (size_t)(x - lines) * 128);
    }
    if (cnt + n > list_cap<G>()) gather();
    const float* sb = ws.s.sc[bi % kBatches];
    const int* kb_j = ws.s.ci[bi % kBatches];
    // The batch's decisions first (independent rounds of 32), then the list.
    unsigned kb[BU], un[BU];
#pragma unroll
    for (int i = 0; i < BU; ++i) {
      const int e = i * kUnit + lane;
      unsigned bits = 0u;
      if (e < n) {
#pragma unroll
        for (int h = 0; h < G; ++h)
          if (sb[e * GC + h] >= Th[h]) bits |= 1u << h;
      }
      if constexpr (POL == TOPT_GQA_UNION) {
        if (bits) bits = (1u << G) - 1u;
      } else if constexpr (POL == TOPT_GQA_VOTE) {
        if (__popc(bits) < p.gqa_min) bits = 0u;
      }
      kb[i] = bits;
      un[i] = __ballot_sync(0xffffffffu, bits != 0u);
    }
#pragma unroll
    for (int i = 0; i < BU; ++i) {
      const unsigned bits = kb[i];
      if (bits) {
        const int e = i * kUnit + lane;
        const int j = kb_j[e];
        const int pos = cnt + __popc(un[i] & ((1u << lane) - 1u));
        jl[pos] = j | (int)(bits << kKeyBits);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const bool keep = (bits >> h) & 1u;
          const float w = keep ? __expf(sb[e * GC + h] - Mh[h]) : 0.f;
          kt[h] += keep ? 1 : 0;
          Rl[h] += w;
          wl[pos][h] = w;
        }
      }
      cnt += __popc(un[i]);
    }
    __syncwarp();  // the slot is consumed: refill it with a later batch
    if (bi + kBatches < nbatch) fetch(bi + kBatches);
    cp_async_commit();
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
  // This CTA's partial sums go to the CTA that combines them: output idx
  // belongs to CTA idx / slice, which keeps one slice per source CTA.
  const int slice = G * D / (int)csize;
  for (int idx = threadIdx.x; idx < G * D; idx += kThreads) {
    const int h = idx / D, dd = idx - h * D;
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s += sm.u.acc[w][h][dd];
    const int c = idx / slice;
    st_peer_f32(peer_addr(&sm.rnum[(int)crank * slice + (idx - c * slice)], (uint32_t)c), s);
  }
  if (threadIdx.x < G) {
    float r = 0.f;
    int k = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      r += sm.wr[w][threadIdx.x];
      k += sm.wk[w][threadIdx.x];
    }
    for (uint32_t c = 0; c < csize; ++c) {
      st_peer_f32(peer_addr(&sm.rR[crank][threadIdx.x], c), r);
      st_peer_s32(peer_addr(&sm.rK[crank][threadIdx.x], c), k);
    }
  }
  if (threadIdx.x == 0) {
    int n = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) n += sm.wn[w];
    st_peer_s32(peer_addr(&sm.rN[crank], 0), n);
  }
  cluster_sync();  // #2: every partial is in its combining CTA's shared memory

  // ----------------------------- combine, SDC and VMC (shared out over the cluster)
  if (threadIdx.x < G) {
    const int h = threadIdx.x;
    float r = 0.f;
    int k = 0;
    for (uint32_t c = 0; c < csize; ++c) {  // rank order
      r += sm.rR[c][h];
      k += sm.rK[c][h];
    }
    sm.Rt[h] = r;
    sm.Kt[h] = k;
  }
  if (crank == 0 && threadIdx.x == kWarp && p.vrows) {
    int n = 0;
    for (uint32_t c = 0; c < csize; ++c) n += sm.rN[c];
    p.vrows[pair] = n;
  }
  __syncthreads();
  {
    const int o0 = slice * (int)crank;  // this CTA's share of the G x D outputs
    for (int k = threadIdx.x; k < slice; k += kThreads) {
      const int idx = o0 + k;
      const int h = idx / D, dd = idx - h * D;
      float num = 0.f;
      for (uint32_t c = 0; c < csize; ++c) num += sm.rnum[c * slice + k];  // rank order
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
  // The CTA leaves: nothing reads its shared memory after the second barrier.
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
int decode_max_cache() { return (int)kKeyMask; }

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
  p.cidx = reinterpret_cast<int32_t*>(static_cast<char*>(a.workspace) + scores_bytes(a));
  const int G = a.n_q_heads / a.n_kv_heads;
  if (a.head_dim == 128) return launch_d<128>(p, G, a, s);
  if (a.head_dim == 64) return launch_d<64>(p, G, a, s);
  return cudaErrorInvalidValue;
}

}  // namespace topt

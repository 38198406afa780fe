// Top-theta causal prefill on the tensor cores (tcgen05), bf16 q/k/v.
//
// [TopTheta] = "Top-Theta Attention: Sparsifying Transformers by Compensated
// Thresholding" (arXiv 2502.08363v2).  Row i of head h sees keys 0..i
// ([TopTheta §2.2, prefill phase]); each score is compared against the row's
// calibrated threshold theta[h][i] ([TopTheta §3, Fig. 1]), SDC [Eq. 4] and
// VMC [Eq. 5-7] normalise the output as in the CUDA-core variant.
//
// One CTA = the same 128-row block of NQ query heads (NQ = 2 when the GQA
// group size is even: two heads of one KV head, so every K and V tile loaded
// serves both; else 1).  Each head's block is a "group": four warps, one
// thread per query row (the row is its TMEM lane), two score buffers S (64
// keys each) and an output accumulator O in TMEM, and its own MMA-issuing
// thread.  While a group's rows turn one S into P, the tensor core computes
// its next S and the other group's P.V and QK^T.
//
// Eleven warps:
//   warps 0-3   rows of group 0; warps 4-7 rows of group 1
//   warp 8      TMA producer: the Q blocks, then K and V tiles through one
//               ring of shared-memory slots, in the order they are consumed
//   warp 9      TMEM allocation; lane 0 issues the MMAs of group 0
//   warp 10     lane 0 issues the MMAs of group 1
//
// A row thread holds its 64 scores of a tile in registers (one 64-column TMEM
// load), so its row maximum and sums need no exchange.  It writes
// P = 2^(a log2(e) / sqrt(d) - m2ref) of kept elements (0 elsewhere) as fp16
// pairs over the first 32 columns of S, and O += P V takes P straight from
// TMEM; it is issued only when some row of the group kept an element.
// 64-key tiles make QK^T an N = 64 MMA (two thirds of the N = 128 rate, by
// measurement) but give each group two S buffers within the 512 TMEM columns,
// so the next QK^T never waits for the rows.
//
// This kernel serves pre-softmax thresholds (keep a >= theta), which need no
// row statistic before the decision, so one pass does S, P and P.V together.
// m2ref is a running reference per row that is raised only when the row
// maximum passes it by more than 15 (log2 units, so P < 2^15 stays finite in
// fp16); then O, R and the row sum are rescaled by 2^(old - new).  Post-softmax
// thresholds need the row maximum and sum first: prefill_tc_post.cu runs them
// in two passes on the buffers prepared here.
//
// P is fp16: rounding it to bf16 costs up to ~2e-3 relative output error on
// peaked rows, fp16 ~3e-4.  One MMA takes A and B in the same 16-bit type, so
// V is read from an fp16 copy scaled per (batch, kv head) by 2^-e with e set
// so that max|V| 2^-e lies in [2^14, 2^15): the scaling is exact and every
// bf16 value above 2^-17 max|V| converts exactly; O is multiplied by 2^e.
#include <cuda_fp16.h>

#include <algorithm>
#include <cfloat>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace topt {
namespace {

using namespace tc;

constexpr int BM = 128;          // query rows per head block = TMEM lanes
constexpr int BN = 64;           // keys per tile
constexpr int kGroups = 2;       // head blocks per CTA (at most)
constexpr int kRowThreads = 128 * kGroups;
constexpr int kProducerWarp = 8;
constexpr int kIssueWarp = 9;    // + group; warp 9 also allocates TMEM
constexpr int kTcThreads = 32 * 11;
constexpr uint32_t kTmemCols = 512;  // S buffer b of group g at 128 g + 64 b; O of group g at 256 + 128 g
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLazy = 15.f;        // headroom of the running reference (log2 units; P < 2^15 fits fp16)

// Shared-memory layout (byte offsets from a 1024-aligned base).  Operand
// tiles are stored as the 128-byte-swizzle layout TMA writes: rows of 128
// bytes (64 16-bit elements), 16-byte chunk c of row r at chunk c ^ (r & 7).
template <int D>
struct TcLayout {
  static constexpr int NP = D / 64;          // 64-element panels along d
  static constexpr uint32_t QP = BM * 128;   // one Q panel
  static constexpr uint32_t KP = BN * 128;   // one K or V panel
  static constexpr uint32_t QT = NP * QP;    // one Q block
  static constexpr uint32_t TILE = NP * KP;  // one K or V tile = one ring slot
  static constexpr int NS = 8;               // ring slots
  static constexpr uint32_t Q = 0;
  static constexpr uint32_t RING = Q + kGroups * QT;
  static constexpr uint32_t BAR = RING + NS * TILE;
  // barriers: Q full [group]; slot full / empty (empty counts one arrival per
  // group); per group and S buffer ([2 g + b]): S full (its QK^T finished),
  // P full (the rows wrote P), P.V done (or skipped); per group: O final, MMA
  // drain
  static constexpr int B_Q = 0, B_FULL = B_Q + kGroups, B_EMPTY = B_FULL + NS,
                       B_SF = B_EMPTY + NS, B_PF = B_SF + 2 * kGroups,
                       B_PD = B_PF + 2 * kGroups, B_O = B_PD + 2 * kGroups, B_DRAIN = B_O + kGroups,
                       NBAR = B_DRAIN + kGroups;
  // misc words: abort flag, TMEM address, O written [group]; any-kept flags
  // [group][S buffer][4 warps]
  static constexpr uint32_t MISC = BAR + NBAR * 8;
  static constexpr uint32_t ANY = MISC + 16;
  static constexpr uint32_t BYTES = ANY + kGroups * 2 * 4;
  static constexpr uint32_t ALLOC = BYTES + 1024;  // room to align the base
  // epilogue: both output blocks staged in the ring (16-byte chunks swizzled
  // by row), the row betas and the VMC scan sums in the idle Q blocks
  static constexpr uint32_t STAGE = RING;
  static constexpr uint32_t BETAS = Q;
  static constexpr uint32_t SCAN = Q + kGroups * BM * 4;
  static_assert(kGroups * BM * D * 4 <= NS * TILE, "output staging fits in the ring");
  static_assert(SCAN + (1 + kRowThreads / (D / 4)) * D * 4 <= RING, "scan sums fit in the Q blocks");
  static_assert(ALLOC <= 227 * 1024, "shared memory");
  static_assert(MISC % 8 == 0 && ANY % 4 == 0, "alignment");
  static_assert(RING % 1024 == 0 && TILE % 1024 == 0 && QT % 1024 == 0, "128-byte-swizzle tiles");
};

struct TcParams {
  int B, Hq, Hkv, S, Lmax, mode, sdc, vmc, mask_words, nqb;
  float gamma, sm_scale;
  const float* theta;
  const float* e_tilde;  // offline E~ [Hq][Lmax] (pre-softmax, TOPT_SDC_OFFLINE)
  float* out;
  int32_t* kept;
  uint32_t* mask;
  unsigned long long* tiles;
  int32_t* status;
  const uint32_t* v;     // [B][Hkv][S][D] bf16 V (pairs), read by the epilogue when vmc
  const float* bsum;     // [B * Hkv][nqb][D] column sums of V rows before each 128-row block (vmc)
  const int32_t* vexp;   // [B * Hkv] exponent e of the fp16 V copy (V16 = V 2^-e)
  int withhold_k;        // test hook: never load the first K tile of a block
};

// Programmatic dependent launch: this grid lets the next one start / waits
// for the previous one to complete with its memory visible.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Barrier of the row threads of both groups.
__device__ __forceinline__ void rows_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kRowThreads) : "memory");
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Largest of the BN scores of a tile (three-input max, four chains).
__device__ __forceinline__ float row_max(const uint32_t (&v)[BN]) {
  float mx[4] = {__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]),
                 __uint_as_float(v[3])};
#pragma unroll
  for (int c = 4; c < BN; c += 8) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      mx[q] = fmax3(mx[q], __uint_as_float(v[c + 2 * q]), __uint_as_float(v[c + 2 * q + 1]));
  }
  return fmax3(mx[0], mx[1], fmaxf(mx[2], mx[3]));
}

// Weights of 32 scores v[c0 .. c0 + 31]: P = 2^(a c2 - m2ref) where a >= braw
// (0 elsewhere) packed as fp16 pairs into w[c0 / 2 ..], with the sums of P,
// of the kept indicator and of 2^(a c2 - m2ref) over every element.
// Hidden keys hold -inf: weight 0, never kept (braw is finite or -FLT_MAX).
__device__ __forceinline__ void chunk_weights(const uint32_t (&v)[BN], int c0, float2 cc, float2 mm,
                                              float braw, uint32_t (&w)[BN / 2], float2& tR,
                                              float2& tK, float2& tZ) {
#pragma unroll
  for (int c = 0; c < 32; c += 2) {
    const float a0 = __uint_as_float(v[c0 + c]), a1 = __uint_as_float(v[c0 + c + 1]);
    const float2 y = ffma2(make_float2(a0, a1), cc, mm);
    const float2 e = make_float2(ex2(y.x), ex2(y.y));
    tZ = fadd2(tZ, e);
    const float2 k = make_float2(setge(a0, braw), setge(a1, braw));
    const float2 pw = fmul2(e, k);
    tR = fadd2(tR, pw);
    tK = fadd2(tK, k);
    w[(c0 + c) >> 1] = pack_half2(pw.x, pw.y);
  }
}

// Key tiles are taken from the diagonal backwards (tile nt-1 first): in a
// causal row the largest scores tend to be near the diagonal, so the running
// reference of the pre-softmax pass is seldom raised after its first tile.
// Load sequence of one CTA (the order the MMAs consume tiles), with
// T_u = tile nt-1-u: K(T_0) V(T_0) K(T_1) V(T_1) ...  Load n goes to ring
// slot n % NS, its (n / NS)-th use.  Tile u of a group uses S buffer u % 2;
// the per-buffer barriers complete once per use of their buffer, so a use's
// parity is (u / 2) & 1.
template <int D, int NQ>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const TcParams p) {
  using L = TcLayout<D>;
  constexpr int NS = L::NS;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  unsigned char* gb = smem_raw + (sb - raw);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gb + L::MISC);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gb + L::MISC + 4);
  volatile int* o_written = reinterpret_cast<volatile int*>(gb + L::MISC + 8);  // [group]
  volatile uint8_t* anyf = reinterpret_cast<volatile uint8_t*>(gb + L::ANY);    // [group][4]
  auto bar = [sb](int i) -> uint32_t { return sb + L::BAR + 8u * (uint32_t)i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // heaviest row blocks (most causal key tiles) first
  const int hgroups = p.Hq / NQ;
  const int per = p.B * hgroups;
  const int qb = p.nqb - 1 - (int)(blockIdx.x / per);
  const int rem = (int)(blockIdx.x % per);
  const int h0 = (rem % hgroups) * NQ, b = rem / hgroups;
  const int kvh = h0 / (p.Hq / p.Hkv);
  const int row0 = qb * BM;
  const int nt = (min(row0 + BM, p.S) - 1) / BN + 1;  // causal key tiles
  const int bh_kv = b * p.Hkv + kvh;

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::NBAR; ++i) {
      uint32_t count = 1;
      if (i >= L::B_EMPTY && i < L::B_EMPTY + NS) count = NQ;
      if (i >= L::B_PF && i < L::B_PF + 2 * kGroups) count = 4;
      mbar_init(bar(i), count);
    }
    *abort_flag = 0;
    o_written[0] = o_written[1] = 0;
    mbar_init_fence();
  }
  if (warp == kIssueWarp) {
    tmem_alloc(smem_u32(gb + L::MISC + 4), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kProducerWarp) {
    // ------------------------------------------------ producer: Q, K, V
    if (lane == 0) {
      for (int g = 0; g < NQ; ++g) {
        mbar_expect_tx(bar(L::B_Q + g), L::QT);
        for (int pn = 0; pn < L::NP; ++pn)
          tma_load_3d(sb + L::Q + g * L::QT + pn * L::QP, &tmQ, bar(L::B_Q + g), 64 * pn, row0,
                      b * p.Hq + h0 + g);
      }
      const int nseq = 2 * nt;
      bool v_ready = false;
      int issued = 0;
      for (int n = 0; n < nseq; ++n) {
        const int s = n % NS;
        if (n >= NS && !mbar_wait(bar(L::B_EMPTY + s), ((n / NS) - 1) & 1, abort_flag)) break;
        const bool isv = n & 1;
        const int tile = nt - 1 - (n >> 1);
        if (isv && !v_ready) {
          pdl_wait();  // the fp16 copy of V is written by the previous grid
          v_ready = true;
        }
        issued = n + 1;
        if (p.withhold_k && n == 0) continue;  // the first wait on slot 0 must run out
        mbar_expect_tx(bar(L::B_FULL + s), L::TILE);
        for (int pn = 0; pn < L::NP; ++pn)
          tma_load_3d(sb + L::RING + s * L::TILE + pn * L::KP, isv ? &tmV : &tmK, bar(L::B_FULL + s),
                      64 * pn, tile * BN, bh_kv);
      }
      // every copy this thread issued lands before the CTA releases its memory
      bool drained = true;
      for (int g = 0; g < NQ; ++g) drained &= mbar_wait_drain(bar(L::B_Q + g), 0);
      for (int n = max(0, issued - NS); n < issued; ++n)
        if (!(p.withhold_k && n == 0)) drained &= mbar_wait_drain(bar(L::B_FULL + n % NS), (n / NS) & 1);
      if (!drained) set_status(p.status, TOPT_ETIMEOUT);
    }
    __syncwarp();
  } else if (warp >= kIssueWarp) {
    // ------------------------------------------- MMAs of one group (head)
    const int g = warp - kIssueWarp;
    if (lane == 0 && g < NQ) {
      constexpr uint32_t idS = idesc_f16(BN, 1, 1, 0);  // bf16 Q, bf16 K (K-major)
      constexpr uint32_t idO = idesc_f16(D, 0, 0, 1);   // fp16 P (TMEM), fp16 V (N-major)
      // descriptor words: every shared operand has 8-row groups 1024 bytes apart
      constexpr uint32_t hi = sdesc_hi(1024);
      const uint32_t q_lo = sdesc_lo(sb + L::Q + g * L::QT, 16);
      const uint32_t k_lo = sdesc_lo(sb + L::RING, 16);
      const uint32_t v_lo = sdesc_lo(sb + L::RING, L::KP);
      const uint32_t sO = tmem + 256u + 128u * g;
      bool ok = mbar_wait(bar(L::B_Q + g), 0, abort_flag);
      // QK^T of tile j into S buffer j % 2, once the buffer's previous tile
      // (j - 2) is done: its P.V finished (or was skipped)
      auto qk = [&](int j) -> bool {
        const int bb = j & 1;
        const int n = 2 * j;  // load holding K of tile j
        const int s = n % NS;
        if (!mbar_wait(bar(L::B_FULL + s), (n / NS) & 1, abort_flag)) return false;
        if (j >= 2 && !mbar_wait(bar(L::B_PD + 2 * g + bb), ((j - 2) >> 1) & 1, abort_flag)) return false;
        tc_fence_after();
        const uint32_t ka = k_lo + s * (L::TILE >> 4);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          tc_mma_f16_w(tmem + 128u * g + 64u * bb, q_lo + (k >> 2) * (L::QP >> 4) + 2 * (k & 3),
                       ka + (k >> 2) * (L::KP >> 4) + 2 * (k & 3), hi, idS, (uint32_t)k);
        tc_commit(bar(L::B_SF + 2 * g + bb));
        tc_commit(bar(L::B_EMPTY + s));
        return true;
      };
      uint32_t started = 0;
      unsigned long long executed = 0;
      // the first two QK^T, then per tile P.V and the QK^T two tiles on
      for (int j = 0; ok && j < min(nt, 2); ++j) ok = qk(j);
      for (int u = 0; ok && u < nt; ++u) {
        const int bb = u & 1;
        const int nv = 2 * u + 1, sv = nv % NS;  // load holding V of tile u
        if (!(ok = mbar_wait(bar(L::B_PF + 2 * g + bb), (u >> 1) & 1, abort_flag))) break;
        const bool any = *reinterpret_cast<volatile uint32_t*>(anyf + 8 * g + 4 * bb) != 0u;
        // the slot is released only after its bytes arrived, also when unused
        if (!(ok = mbar_wait(bar(L::B_FULL + sv), (nv / NS) & 1, abort_flag))) break;
        if (any) {
          tc_fence_after();
          // P of keys 2c, 2c + 1 sits in column c of S
          const uint32_t pa = tmem + 128u * g + 64u * bb;
          const uint32_t va = v_lo + sv * (L::TILE >> 4);
#pragma unroll
          for (int k = 0; k < BN / 16; ++k)
            tc_mma_f16_ts(sO, pa + 8 * k, va + 128 * k, hi, idO, started | (uint32_t)k);
          started = 1;
          ++executed;
          tc_commit(bar(L::B_PD + 2 * g + bb));
          tc_commit(bar(L::B_EMPTY + sv));
        } else {
          mbar_arrive(bar(L::B_PD + 2 * g + bb));
          mbar_arrive(bar(L::B_EMPTY + sv));
        }
        if (u + 2 < nt) ok = qk(u + 2);
      }
      tc_commit(bar(L::B_DRAIN + g));
      const bool drained = mbar_wait_drain(bar(L::B_DRAIN + g), 0);
      if (ok && drained) {
        o_written[g] = (int)started;
        mbar_arrive(bar(L::B_O + g));  // releases o_written and the finished O
      }
      if (!ok || !drained) set_status(p.status, TOPT_ETIMEOUT);
      if (p.tiles) {
        atomicAdd(p.tiles + 0, executed);
        atomicAdd(p.tiles + 1, (unsigned long long)nt);
      }
    }
    __syncwarp();
  } else {
    // --------------------------------------------------------- query rows
    // Thread = row r of group g's head block: TMEM lane r of S and O.
    const int g = warp >> 2, quad = warp & 3;
    const int r = quad * 32 + lane;
    const int i = row0 + r;
    const bool active = g < NQ;
    const bool row_ok = active && i < p.S;
    const int h = h0 + g, bh_q = b * p.Hq + h;
    const uint32_t lanes = (uint32_t)(quad * 32) << 16;
    const uint32_t sS = tmem + lanes + 128u * g, sO = tmem + lanes + 256u + 128u * g;
    const float c2 = p.sm_scale * kLog2e;
    const int Lrow = i + 1;
    const float th = row_ok ? p.theta[(size_t)h * p.Lmax + (min(Lrow, p.Lmax) - 1)] : 0.f;
    bool ok = active;
    uint32_t v[BN];
    // hidden keys of key tile t (beyond the row, or the whole row when
    // i >= S) -> -inf
    auto hide = [&](int t) {
      const int lim = row_ok ? i - t * BN : -1;  // columns c <= lim are visible
      if (!__all_sync(0xffffffffu, lim >= BN - 1)) {
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (c > lim) v[c] = __float_as_uint(-CUDART_INF_F);
      }
    };

    // keep iff the raw score a * sqrt(d) >= braw; a hidden key (-inf) never
    // passes the finite bound
    const float braw = fmaxf(th / p.sm_scale, -FLT_MAX);

    // The single pass: P where kept.  R sums the fp32 weights (P.V multiplies
    // them rounded to fp16: relative difference below 2^-11 per weight).
    // m2ref follows the row maximum, Z sums every weight (used by exact SDC;
    // one packed add per two keys, cheaper than a second code path), m2max is
    // the row maximum.
    float m2ref = -CUDART_INF_F, m2max = -CUDART_INF_F;
    float R = 0.f, KEPT = 0.f, Z = 0.f;
    uint32_t* mrow = (p.mask && row_ok) ? p.mask + ((size_t)bh_q * p.S + i) * p.mask_words : nullptr;
    for (int u = 0; ok && u < nt; ++u) {
      const int bb = u & 1;
      const uint32_t sSb = sS + 64u * bb;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::B_SF + 2 * g + bb), (u >> 1) & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
      tmem_ld<BN>(sSb, v);
      const int tile = nt - 1 - u;
      hide(tile);
      float factor = 1.f;
      bool rescale_o = false;
      {
        const float t2 = row_max(v) * c2;
        m2max = fmaxf(m2max, t2);
        if (t2 > m2ref + kLazy) {  // -inf + kLazy = -inf: the first visible tile
          rescale_o = m2ref != -CUDART_INF_F;
          factor = rescale_o ? ex2(m2ref - t2) : 0.f;
          m2ref = t2;
          R *= factor;
          Z *= factor;
        }
      }
      const float mref = m2ref == -CUDART_INF_F ? 0.f : m2ref;
      const float2 cc = make_float2(c2, c2), mm = make_float2(-mref, -mref);
      // all P words first, then one store: the scores of a chunk are dead
      // once its words and mask bits exist
      float2 tR = make_float2(0.f, 0.f), tK = make_float2(0.f, 0.f), tZ = make_float2(0.f, 0.f);
      uint32_t w[BN / 2];
#pragma unroll
      for (int q = 0; q < BN / 32; ++q) {
        chunk_weights(v, 32 * q, cc, mm, braw, w, tR, tK, tZ);
        if (mrow) {
          uint32_t k = 0u;
#pragma unroll
          for (int c = 0; c < 32; ++c) k |= (uint32_t)(__uint_as_float(v[32 * q + c]) >= braw) << c;
          const int wd = (BN / 32) * tile + q;
          if (wd < p.mask_words) mrow[wd] = k;
        }
      }
      tmem_st<BN / 2>(sSb, w);  // waits for the store
      const float tk = tK.x + tK.y;
      R += tR.x + tR.y;
      KEPT += tk;
      Z += tZ.x + tZ.y;
      if (__any_sync(0xffffffffu, rescale_o)) {
        // O += P V of the previous tile has finished; the next P.V of this
        // group starts only after this warp signals P full
        ok = __all_sync(0xffffffffu,
                        mbar_wait(bar(L::B_PD + 2 * g + (bb ^ 1)), ((u - 1) >> 1) & 1, abort_flag));
        if (ok) {
          // the whole O row in one load and one store (the score registers
          // are free by now)
          tc_fence_after();
          uint32_t o[D];
          tmem_ld<D>(sO, o);
#pragma unroll
          for (int k = 0; k < D; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * factor);
          tmem_st_full<D>(sO, o);
        }
      }
      tc_fence_before();
      const bool wany = __any_sync(0xffffffffu, tk > 0.f);
      if (lane == 0) anyf[8 * g + 4 * bb + quad] = wany ? 1 : 0;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::B_PF + 2 * g + bb));
    }
    if (mrow)
      for (int wd = (BN / 32) * nt; wd < p.mask_words; ++wd) mrow[wd] = 0u;
    const int cnt = (int)KEPT;

    // epilogue: out = O * scale 2^e + beta mu   [TopTheta Eq. 4-7].  Both
    // groups stage O * scale in shared memory (the ring is idle by now: every
    // load of this CTA was consumed), then all row threads stream the blocks
    // out with coalesced 16-byte stores, adding beta mu (prefix means of V,
    // the same for both heads) on the way.
    float* stage = reinterpret_cast<float*>(gb + L::STAGE);  // [group][BM][D], chunks swizzled by row
    float* betas = reinterpret_cast<float*>(gb + L::BETAS);  // [group][BM]
    auto chunk_at = [](int row, int c4) { return row * D + 4 * (c4 ^ (row & 7)); };
    pdl_wait();  // vexp and the block sums come from the preparation grids
    // the staging area is the ring and the Q blocks: every MMA of both groups
    // has finished reading them before any row writes there
#pragma unroll
    for (int gg = 0; gg < NQ; ++gg)
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(L::B_O + gg), 0, abort_flag));
    if (ok) {
      tc_fence_after();
      const bool have_o = o_written[g] != 0;
      float sc = 0.f, beta = 0.f;
      if (row_ok) {
        // the sums are relative to 2^m2ref; the offline E~ is relative to the
        // row maximum
        float e_off = 0.f;
        if (p.sdc == TOPT_SDC_OFFLINE)
          e_off = p.e_tilde[(size_t)h * p.Lmax + (min(Lrow, p.Lmax) - 1)] * ex2(m2max - m2ref);
        out_scale_beta(p.mode, p.sdc, p.gamma, th, m2ref * kLn2, Z, R, Lrow, cnt, e_off, sc, beta);
      }
      const float f = sc * __int_as_float((127 + p.vexp[bh_kv]) << 23);
      float* st = stage + g * BM * D;
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t o[32];
        tmem_ld32(sO + c, o);
#pragma unroll
        for (int k = 0; k < 32; k += 4) {
          float4 val;
          val.x = have_o ? __uint_as_float(o[k + 0]) * f : 0.f;
          val.y = have_o ? __uint_as_float(o[k + 1]) * f : 0.f;
          val.z = have_o ? __uint_as_float(o[k + 2]) * f : 0.f;
          val.w = have_o ? __uint_as_float(o[k + 3]) * f : 0.f;
          *reinterpret_cast<float4*>(st + chunk_at(r, (c + k) / 4)) = val;
        }
      }
      betas[g * BM + r] = beta;
      if (row_ok && p.kept) p.kept[(size_t)bh_q * p.S + i] = cnt;
    }
    rows_sync();  // every row thread reaches it, also after an abort
    const int rows_here = min(BM, p.S - row0);
    constexpr int QD = D / 4;  // 16-byte column chunks of a row
    if (!p.vmc) {
      if (!*abort_flag)
        for (int idx = threadIdx.x; idx < NQ * rows_here * QD; idx += kRowThreads) {
          const int gg = idx / (rows_here * QD), rr = (idx / QD) % rows_here, c4 = idx % QD;
          float* out_blk = p.out + ((size_t)(b * p.Hq + h0 + gg) * p.S + row0) * D;
          *reinterpret_cast<float4*>(out_blk + (size_t)rr * D + 4 * c4) =
              *reinterpret_cast<const float4*>(stage + gg * BM * D + chunk_at(rr, c4));
        }
    } else {
      // mu_i = (sum of V rows 0..i) / (i + 1): the column sums of the blocks
      // before this one plus a scan over this block's rows, by segments of
      // RPS rows (thread: 4 columns x RPS rows), in fp32 from the bf16 V.
      constexpr int NSEG = kRowThreads / QD, RPS = BM / NSEG;
      const int c4 = threadIdx.x % QD, seg = threadIdx.x / QD, c = 4 * c4;
      float* pre_sum = reinterpret_cast<float*>(gb + L::SCAN);  // [D]: sum of V rows 0 .. row0-1
      float* segsum = pre_sum + D;                               // [NSEG][D]: totals of the segments
      if (threadIdx.x < D) pre_sum[threadIdx.x] = p.bsum[((size_t)bh_kv * p.nqb + qb) * D + threadIdx.x];
      float4 run[RPS];
      float4 tot = make_float4(0.f, 0.f, 0.f, 0.f);
      const uint32_t* vblk = p.v + ((size_t)bh_kv * p.S + row0) * (D / 2);
#pragma unroll
      for (int k = 0; k < RPS; ++k) {
        const int rr = seg * RPS + k;
        if (rr < rows_here) {
          const uint2 x = *reinterpret_cast<const uint2*>(vblk + (size_t)rr * (D / 2) + c / 2);
          tot.x += bf16lo(x.x);
          tot.y += bf16hi(x.x);
          tot.z += bf16lo(x.y);
          tot.w += bf16hi(x.y);
        }
        run[k] = tot;
      }
      *reinterpret_cast<float4*>(segsum + seg * D + c) = tot;
      rows_sync();
      if (!*abort_flag) {
        float4 base = *reinterpret_cast<const float4*>(pre_sum + c);
        for (int q = 0; q < seg; ++q) {
          const float4 t4 = *reinterpret_cast<const float4*>(segsum + q * D + c);
          base.x += t4.x;
          base.y += t4.y;
          base.z += t4.z;
          base.w += t4.w;
        }
#pragma unroll
        for (int k = 0; k < RPS; ++k) {
          const int rr = seg * RPS + k;
          if (rr < rows_here) {
            const float inv = 1.f / (float)(row0 + rr + 1);
            const float4 mu = make_float4((base.x + run[k].x) * inv, (base.y + run[k].y) * inv,
                                          (base.z + run[k].z) * inv, (base.w + run[k].w) * inv);
#pragma unroll
            for (int gg = 0; gg < NQ; ++gg) {
              const float bt = betas[gg * BM + rr];
              float4 val = *reinterpret_cast<const float4*>(stage + gg * BM * D + chunk_at(rr, c4));
              val.x = fmaf(bt, mu.x, val.x);
              val.y = fmaf(bt, mu.y, val.y);
              val.z = fmaf(bt, mu.z, val.z);
              val.w = fmaf(bt, mu.w, val.w);
              float* out_blk = p.out + ((size_t)(b * p.Hq + h0 + gg) * p.S + row0) * D;
              *reinterpret_cast<float4*>(out_blk + (size_t)rr * D + c) = val;
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kIssueWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) set_status(p.status, TOPT_ETIMEOUT);
}

// ------------------------------------------------------ fp16 copy of V --
// One 128-row block of V per CTA: the largest |v| of each (batch, kv head)
// into vmax (float bits; zeroed first) and, when bsum is given, the column
// sums of the block into bsum[bh][block][D].
template <int D>
__global__ void __launch_bounds__(256) vstats_kernel(const uint4* __restrict__ v, int S,
                                                     uint32_t* __restrict__ vmax,
                                                     float* __restrict__ bsum) {
  constexpr int W = D / 8;  // 16-byte words per row; every thread keeps one word column
  pdl_launch_dependents();
  const int qb = blockIdx.x, bh = blockIdx.y;
  const int r0 = qb * BM, rows = min(BM, S - r0);
  const uint4* src = v + ((size_t)bh * S + r0) * W;
  float cs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float mx = 0.f;
  for (int w = threadIdx.x; w < rows * W; w += blockDim.x) {
    const uint4 x = ld_nc16(src + w);
    const float e[8] = {bf16lo(x.x), bf16hi(x.x), bf16lo(x.y), bf16hi(x.y),
                        bf16lo(x.z), bf16hi(x.z), bf16lo(x.w), bf16hi(x.w)};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      cs[k] += e[k];
      mx = fmaxf(mx, fabsf(e[k]));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  __shared__ float wmax[8];
  __shared__ float part[256][9];
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = mx;
#pragma unroll
  for (int k = 0; k < 8; ++k) part[threadIdx.x][k] = cs[k];
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) mx = fmaxf(mx, wmax[w]);
    atomicMax(vmax + bh, __float_as_uint(mx));  // mx >= 0: integer order = float order
  }
  if (bsum && threadIdx.x < D) {
    const int col = threadIdx.x, wc = col / 8, k = col % 8;
    float acc = 0.f;
    for (int t = wc; t < (int)blockDim.x; t += W) acc += part[t][k];
    bsum[((size_t)bh * gridDim.x + qb) * D + col] = acc;
  }
}

// e with max|v| 2^-e in [2^14, 2^15) (0 for an all-zero or non-finite head).
__device__ __forceinline__ int v16_exponent(uint32_t maxbits) {
  const float mx = __uint_as_float(maxbits);
  if (!(mx > 0.f) || !(mx <= 3.4e38f)) return 0;
  return min(max(ilogbf(mx) - 14, -110), 110);
}

template <int D>
__global__ void __launch_bounds__(256) v16_kernel(const uint4* __restrict__ v, int S,
                                                  const uint32_t* __restrict__ vmax,
                                                  uint4* __restrict__ v16, int32_t* __restrict__ vexp,
                                                  float* __restrict__ bsum, int nqb) {
  pdl_wait();  // vmax and the block sums are complete
  pdl_launch_dependents();
  const int bh = blockIdx.y;
  if (bsum && blockIdx.x == 0 && threadIdx.x < D) {
    // block column sums -> exclusive prefix sums over the blocks of this head
    float* col = bsum + (size_t)bh * nqb * D + threadIdx.x;
    float run = 0.f;
    for (int q = 0; q < nqb; ++q) {
      const float x = col[(size_t)q * D];
      col[(size_t)q * D] = run;
      run += x;
    }
  }
  const size_t n16 = (size_t)S * D / 8;
  const int e = v16_exponent(vmax[bh]);
  const float scale = __int_as_float((127 - e) << 23);
  const uint4* src = v + (size_t)bh * n16;
  uint4* dst = v16 + (size_t)bh * n16;
  for (size_t w = (size_t)blockIdx.x * blockDim.x + threadIdx.x; w < n16;
       w += (size_t)gridDim.x * blockDim.x) {
    const uint4 x = ld_nc16(src + w);
    uint4 y;
    y.x = pack_half2(bf16lo(x.x) * scale, bf16hi(x.x) * scale);
    y.y = pack_half2(bf16lo(x.y) * scale, bf16hi(x.y) * scale);
    y.z = pack_half2(bf16lo(x.z) * scale, bf16hi(x.z) * scale);
    y.w = pack_half2(bf16lo(x.w) * scale, bf16hi(x.w) * scale);
    dst[w] = y;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) vexp[bh] = e;
}

template <int D, int NQ>
cudaError_t launch_tc(const topt_prefill_args& a, const TcParams& p, void* v16, cudaStream_t s) {
  const int BHkv = a.batch * a.n_kv_heads;
  CUtensorMap tq, tk, tv;
  if (!tensor_map_3d(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q, D, a.seq, a.batch * a.n_q_heads, BM) ||
      !tensor_map_3d(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.k, D, a.seq, BHkv, BN) ||
      !tensor_map_3d(&tv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, v16, D, a.seq, BHkv, BN))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D, NQ>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TcLayout<D>::ALLOC);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  // programmatic launch: loads of Q and K overlap the preparation grids (a
  // profiling event in between serialises them, which only moves time
  // between them)
  cfg.gridDim = dim3((unsigned)((size_t)p.nqb * a.n_q_heads / NQ * a.batch));
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = TcLayout<D>::ALLOC;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_tc_kernel<D, NQ>, tq, tk, tv, p);
}

template <int D>
cudaError_t run_d(const topt_prefill_args& a, const TcParams& p, void* v16, uint32_t* vmax,
                  int32_t* vexp, cudaStream_t s) {
  const int BHkv = a.batch * a.n_kv_heads;
  // fp16 copy of V scaled per head
  cudaError_t e = cudaMemsetAsync(vmax, 0, sizeof(uint32_t) * BHkv, s);
  if (e != cudaSuccess) return e;
  const size_t n16 = (size_t)a.seq * D / 8;
  const int chunks = (int)std::min<size_t>(64, (n16 + 1023) / 1024);
  vstats_kernel<D><<<dim3(p.nqb, BHkv), 256, 0, s>>>(static_cast<const uint4*>(a.v), a.seq, vmax,
                                                     const_cast<float*>(p.bsum));
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(chunks, BHkv);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if ((e = cudaLaunchKernelEx(&cfg, v16_kernel<D>, static_cast<const uint4*>(a.v), a.seq,
                              (const uint32_t*)vmax, static_cast<uint4*>(v16), vexp,
                              const_cast<float*>(p.bsum), p.nqb)) != cudaSuccess)
    return e;
  if ((e = record_event(a.events[0], s)) != cudaSuccess) return e;
  if (a.mode == TOPT_POST)  // two passes: the kernel of prefill_tc_post.cu
    e = prefill_tc_post_launch(a, v16, vexp, p.bsum, s, p.withhold_k);
  else  // one pass, two heads per CTA when they share a KV head
    e = (a.n_q_heads / a.n_kv_heads) % 2 == 0 ? launch_tc<D, 2>(a, p, v16, s) : launch_tc<D, 1>(a, p, v16, s);
  if (e != cudaSuccess) return e;
  return record_event(a.events[1], s);
}

}  // namespace

size_t prefill_tc_bsum_bytes(const topt_prefill_args& a) {
  return (size_t)a.batch * a.n_kv_heads * ((a.seq + BM - 1) / BM) * a.head_dim * sizeof(float);
}

size_t prefill_tc_v16_bytes(const topt_prefill_args& a) {
  return (size_t)a.batch * a.n_kv_heads * a.seq * a.head_dim * 2;
}

int prefill_tc_rows() { return BM; }
int prefill_tc_keys(int mode) { return mode == TOPT_POST ? prefill_tc_post_keys() : BN; }

cudaError_t prefill_tc_run(const topt_prefill_args& a, void* v16, uint32_t* vmax, int32_t* vexp,
                           float* bsum, cudaStream_t s, int withhold_k) {
  TcParams p;
  p.B = a.batch;
  p.Hq = a.n_q_heads;
  p.Hkv = a.n_kv_heads;
  p.S = a.seq;
  p.Lmax = a.theta_len;
  p.mode = a.mode;
  p.sdc = a.sdc;
  p.vmc = a.vmc;
  p.mask_words = (a.seq + 31) / 32;
  p.nqb = (a.seq + BM - 1) / BM;
  p.gamma = a.gamma;
  p.sm_scale = 1.0f / sqrtf((float)a.head_dim);
  p.theta = a.theta;
  p.e_tilde = a.e_tilde;
  p.out = a.out;
  p.kept = a.kept;
  p.mask = a.mask;
  p.tiles = a.tiles;
  p.status = a.status;
  p.v = static_cast<const uint32_t*>(a.v);
  p.bsum = a.vmc ? bsum : nullptr;
  p.vexp = vexp;
  p.withhold_k = withhold_k;
  return a.head_dim == 128 ? run_d<128>(a, p, v16, vmax, vexp, s) : run_d<64>(a, p, v16, vmax, vexp, s);
}

}  // namespace topt

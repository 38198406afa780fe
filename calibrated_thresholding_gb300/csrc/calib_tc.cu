// Calibration scores on the tensor cores (tcgen05), bf16 q/k.
//
// [TopTheta] = "Top-Theta Attention: Sparsifying Transformers by Compensated
// Thresholding" (arXiv 2502.08363v2).  Algorithm 1 of [TopTheta §3.1] (and
// the multi-k calibration of App. D and the offline SDC estimate of §3.2.1)
// need every score a_ij = q_i . k_j / sqrt(d), j < L_i, of every calibration
// row: this kernel writes them to the workspace, row-major with n_keys floats
// per row, exactly where the CUDA-core score kernel of calibrate.cu puts them,
// and the select kernels read them from there.
//
// One CTA = 128 consecutive calibration rows of one (sequence, head); it
// computes 128 x 128 score tiles over the keys the longest of its rows needs.
// Six warps:
//   warps 0-3  writers: thread = row (its TMEM lane); per tile, four chunks of
//              32 columns go TMEM -> registers -> a per-warp staging tile in
//              shared memory -> the workspace, one 128-byte row segment per
//              store instruction
//   warp 4     TMA producer: the Q block once, K tiles through a 3-stage ring
//   warp 5     TMEM allocation; lane 0 issues QK^T (M = 128, N = 128 keys)
//              into two score buffers, so the next tile is computed while the
//              writers drain the last one
// The work is bound by the fp32 score writes (4 bytes per score against
// 4 d flops), not by the tensor core.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace topt {
namespace {

using namespace tc;

constexpr int BM = 128;             // rows per CTA = TMEM lanes
constexpr int BN = 128;             // keys per tile
constexpr int KST = 3;              // K ring stages
constexpr int kWriters = 4;         // warps 0-3
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreads = 32 * 6;
constexpr uint32_t kTmemCols = 256;  // score buffers at columns 0 and 128
// Staging tile of a writer warp: 32 rows x 32 floats, the 16-byte chunk c of
// row r at chunk c ^ (r & 7), so both the row-wise writes and the 4-row x
// 8-chunk reads of 16 bytes are free of bank conflicts.
constexpr int SS = 32;

template <int D>
struct CalLayout {
  static constexpr int NP = D / 64;
  static constexpr uint32_t QP = BM * 128;  // one 64-column panel of the Q block
  static constexpr uint32_t KP = BN * 128;  // one panel of a K tile
  static constexpr uint32_t Q = 0;
  static constexpr uint32_t K = Q + NP * QP;
  static constexpr uint32_t STAGE = K + KST * NP * KP;  // [kWriters][32][SS] floats
  static constexpr uint32_t BAR = (STAGE + kWriters * 32 * SS * 4 + 7) & ~7u;
  // Q full; K full / empty; S full (QK^T done) / S drained (writers done), per buffer
  static constexpr int B_Q = 0, B_FULL = 1, B_EMPTY = B_FULL + KST, B_SF = B_EMPTY + KST,
                       B_SD = B_SF + 2, B_DRAIN = B_SD + 2, NBAR = B_DRAIN + 1;
  static constexpr uint32_t MISC = BAR + NBAR * 8;  // abort flag, TMEM address, max row length
  static constexpr uint32_t ALLOC = MISC + 16 + 1024;
  static_assert(ALLOC <= 227 * 1024, "shared memory");
  static_assert(K % 1024 == 0 && (NP * KP) % 1024 == 0, "128-byte-swizzle tiles");
};

struct ScoreTcParams {
  int N, Hq, Hkv, R, Nk, h0, Hp;
  float scale;
  const int32_t* row_len;
  long it0;        // rows [it0, it0 + nrows) of the flattened (seq, head of the pass, row) index
  int nrows;
  float* ws;       // ws[(it - it0) * Nk + j]
  int nh0, nnh;    // (seq, head of the pass) blocks nh0 .. nh0 + nnh - 1 overlap the pass
  int ntile;       // 128-row tiles per block
  int32_t* status;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    calib_scores_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                           const ScoreTcParams p) {
  using L = CalLayout<D>;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  unsigned char* gb = smem_raw + (sb - raw);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gb + L::MISC);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gb + L::MISC + 4);
  volatile int* maxlen = reinterpret_cast<volatile int*>(gb + L::MISC + 8);
  auto bar = [sb](int i) -> uint32_t { return sb + L::BAR + 8u * (uint32_t)i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // longest tiles (largest row ids, usually the longest rows) first
  const int itile = p.ntile - 1 - (int)(blockIdx.x / p.nnh);
  const int nh = p.nh0 + (int)(blockIdx.x % p.nnh);  // flattened (seq, head of the pass)
  const int n = nh / p.Hp, h = p.h0 + nh % p.Hp;
  const int i0 = itile * BM;
  const long it_row0 = (long)nh * p.R + i0;  // flattened index of row i0

  // this writer's row: its length, 0 when outside the pass or invalid (the
  // select kernel reports an invalid length)
  int Lr = 0;
  if (warp < kWriters) {
    const int r = warp * 32 + lane;
    const long it = it_row0 + r;
    if (i0 + r < p.R && it >= p.it0 && it < p.it0 + p.nrows) {
      const int len = p.row_len[i0 + r];
      Lr = (len >= 1 && len <= p.Nk) ? len : 0;
    }
  }
  if (threadIdx.x == 0) *maxlen = 0;
  __syncthreads();
  if (warp < kWriters) {
    int m = Lr;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) atomicMax(const_cast<int*>(maxlen), m);
  }
  __syncthreads();
  const int nkt = (*maxlen + BN - 1) / BN;
  if (nkt == 0) return;  // the whole CTA: nothing of this tile is in the pass

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::NBAR; ++i) mbar_init(bar(i), (i >= L::B_SD && i < L::B_SD + 2) ? kWriters : 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(gb + L::MISC + 4), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      mbar_expect_tx(bar(L::B_Q), L::NP * L::QP);
      for (int pn = 0; pn < L::NP; ++pn)
        tma_load_3d(sb + L::Q + pn * L::QP, &tmQ, bar(L::B_Q), 64 * pn, i0, n * p.Hq + h);
      const int kz = n * p.Hkv + h / (p.Hq / p.Hkv);
      int issued = 0;
      for (int kt = 0; kt < nkt; ++kt) {
        const int s = kt % KST;
        if (kt >= KST && !mbar_wait(bar(L::B_EMPTY + s), ((kt / KST) - 1) & 1, abort_flag)) break;
        mbar_expect_tx(bar(L::B_FULL + s), L::NP * L::KP);
        for (int pn = 0; pn < L::NP; ++pn)
          tma_load_3d(sb + L::K + (s * L::NP + pn) * L::KP, &tmK, bar(L::B_FULL + s), 64 * pn, kt * BN, kz);
        issued = kt + 1;
      }
      // every copy this thread issued lands before the CTA releases its memory
      bool drained = mbar_wait_drain(bar(L::B_Q), 0);
      for (int kt = max(0, issued - KST); kt < issued; ++kt)
        drained &= mbar_wait_drain(bar(L::B_FULL + kt % KST), (kt / KST) & 1);
      if (!drained) set_status(p.status, TOPT_ETIMEOUT);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idS = idesc_f16(BN, 1, 1, 0);  // bf16 Q, bf16 K (K-major)
      constexpr uint32_t hi = sdesc_hi(1024);
      const uint32_t q_lo = sdesc_lo(sb + L::Q, 16);
      const uint32_t k_lo = sdesc_lo(sb + L::K, 16);
      bool ok = mbar_wait(bar(L::B_Q), 0, abort_flag);
      for (int kt = 0; ok && kt < nkt; ++kt) {
        const int s = kt % KST, bb = kt & 1;
        if (!(ok = mbar_wait(bar(L::B_FULL + s), (kt / KST) & 1, abort_flag))) break;
        // the writers drained this buffer's previous tile
        if (kt >= 2 && !(ok = mbar_wait(bar(L::B_SD + bb), ((kt >> 1) - 1) & 1, abort_flag))) break;
        tc_fence_after();
        const uint32_t ka = k_lo + s * (L::NP * L::KP >> 4);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          tc_mma_f16_w(tmem + 128u * bb, q_lo + (k >> 2) * (L::QP >> 4) + 2 * (k & 3),
                       ka + (k >> 2) * (L::KP >> 4) + 2 * (k & 3), hi, idS, (uint32_t)k);
        tc_commit(bar(L::B_SF + bb));
        tc_commit(bar(L::B_EMPTY + s));
      }
      tc_commit(bar(L::B_DRAIN));
      const bool drained = mbar_wait_drain(bar(L::B_DRAIN), 0);
      if (!ok || !drained) set_status(p.status, TOPT_ETIMEOUT);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ writers
    float* stage = reinterpret_cast<float*>(gb + L::STAGE) + warp * 32 * SS;  // this warp's [32][SS]
    const uint32_t lanes = (uint32_t)(warp * 32) << 16;
    const bool vec = (p.Nk & 3) == 0;  // 16-byte aligned rows of the workspace
    const int sub = lane >> 3, c4 = lane & 7;  // reads: row 4 i + sub, chunk c4
    for (int kt = 0; kt < nkt; ++kt) {
      const int bb = kt & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(L::B_SF + bb), (kt >> 1) & 1, abort_flag))) break;
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < BN; c += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lanes + 128u * bb + (uint32_t)c, v);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<float4*>(stage + lane * SS + 4 * (q ^ (lane & 7))) =
              make_float4(__uint_as_float(v[4 * q]) * p.scale, __uint_as_float(v[4 * q + 1]) * p.scale,
                          __uint_as_float(v[4 * q + 2]) * p.scale, __uint_as_float(v[4 * q + 3]) * p.scale);
        __syncwarp();
        // four rows of the warp per store instruction: 8 lanes x 16 bytes,
        // one 128-byte segment of each row
        const int col = kt * BN + c + 4 * c4;
#pragma unroll 2
        for (int i = 0; i < 8; ++i) {
          const int rr = 4 * i + sub;
          const int len = __shfl_sync(0xffffffffu, Lr, rr);
          if (col < len) {
            const float4 x = *reinterpret_cast<const float4*>(stage + rr * SS + 4 * (c4 ^ (rr & 7)));
            float* dst = p.ws + (it_row0 + warp * 32 + rr - p.it0) * (long)p.Nk + col;
            if (vec && col + 3 < len) {
              *reinterpret_cast<float4*>(dst) = x;
            } else {
              dst[0] = x.x;
              if (col + 1 < len) dst[1] = x.y;
              if (col + 2 < len) dst[2] = x.z;
              if (col + 3 < len) dst[3] = x.w;
            }
          }
        }
        __syncwarp();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::B_SD + bb));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) set_status(p.status, TOPT_ETIMEOUT);
}

template <int D>
cudaError_t run_d(const CalibScoreArgs& a, cudaStream_t s) {
  CUtensorMap tq, tk;
  if (!tensor_map_3d(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q, D, a.R, (long)a.N * a.Hq, BM) ||
      !tensor_map_3d(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.keys, D, a.Nk, (long)a.N * a.Hkv, BN))
    return cudaErrorInvalidValue;
  ScoreTcParams p;
  p.N = a.N;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.R = a.R;
  p.Nk = a.Nk;
  p.h0 = a.h0;
  p.Hp = a.Hp;
  p.scale = a.scale;
  p.row_len = a.row_len;
  p.it0 = a.it0;
  p.nrows = a.nrows;
  p.ws = a.ws;
  p.status = a.status;
  const long last = a.it0 + a.nrows - 1;
  p.nh0 = (int)(a.it0 / a.R);
  p.nnh = (int)(last / a.R) - p.nh0 + 1;
  p.ntile = (a.R + BM - 1) / BM;
  cudaError_t e = cudaFuncSetAttribute(calib_scores_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)CalLayout<D>::ALLOC);
  if (e != cudaSuccess) return e;
  const long grid = (long)p.nnh * p.ntile;
  calib_scores_tc_kernel<D><<<(unsigned)grid, kThreads, CalLayout<D>::ALLOC, s>>>(tq, tk, p);
  return cudaGetLastError();
}

}  // namespace

bool calib_scores_tc_ok(const CalibScoreArgs& a) {
  const auto aligned = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; };
  if (!(a.D == 64 || a.D == 128) || !aligned(a.q) || !aligned(a.keys) || a.R < 1 || a.Nk < 1 || a.nrows < 1)
    return false;
  const long blocks = (a.it0 + a.nrows - 1) / a.R - a.it0 / a.R + 1;
  return blocks * ((a.R + BM - 1) / BM) < (1L << 31) && encode_tiled() != nullptr;
}

cudaError_t calib_scores_tc(const CalibScoreArgs& a, cudaStream_t s) {
  return a.D == 128 ? run_d<128>(a, s) : run_d<64>(a, s);
}

}  // namespace topt

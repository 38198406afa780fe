/*
 * topt.h - C ABI of libtopt.so, Top-theta attention on one GB300 (sm_103a).
 *
 * Source of the method: "Top-Theta Attention: Sparsifying Transformers by
 * Compensated Thresholding" (arXiv 2502.08363v2), cited below as [TopTheta].
 *
 *   scores      a_j = q . k_j / sqrt(d)                 [TopTheta §2.2 Eq. 1]
 *   threshold   keep j iff x_j >= theta, x = a (pre-softmax) or
 *               x = softmax(a) (post-softmax)            [TopTheta §3, Fig. 1]
 *   calibration theta_r = mean + alpha*std of the per-sample k-th largest
 *               element of row r                         [TopTheta §3.1 Alg. 1]
 *   SDC         softmax over kept * R/(R + E~)           [TopTheta §3.2.1 Eq. 4]
 *   VMC         p = s~ V~ + beta * mu                    [TopTheta §3.2.2 Eq. 5-7]
 *
 * Conventions shared by every entry point
 *   - Every tensor pointer is a caller-owned DEVICE pointer to a dense,
 *     row-major (C-contiguous) array in the layout stated beside it.  bf16 is
 *     IEEE bfloat16 (2 bytes); fp32 is IEEE binary32.  16-byte alignment is
 *     required for q, k and v tensors.
 *   - A row with L visible keys uses theta table entry L-1; rows with
 *     L > theta_len use entry theta_len-1.  Entries of -INFINITY keep the
 *     whole row (dense attention).  Post-softmax entries <= 0 keep the row.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream).  Arguments are validated on the host before anything
 *     is launched; a failed validation returns an error and launches nothing.
 *   - Data that lives on the device (sequence lengths, row lengths) is checked
 *     by the kernels: a bad value makes the kernel store a nonzero
 *     topt_status into *status (when status is not NULL) and skip that unit.
 *     The caller zeroes *status and reads it after synchronising.
 *   - The library allocates no device memory.  Scratch memory is the
 *     caller's `workspace`; its size is returned by the *_workspace query.
 *   - Calls that share a workspace must not overlap on the GPU.
 */
#ifndef TOPT_H_
#define TOPT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* topt_stream; /* identical to cudaStream_t */

typedef enum {
  TOPT_OK = 0,
  TOPT_EINVAL = 1,     /* bad argument value, NULL pointer, or bad device-side length */
  TOPT_EDTYPE = 2,     /* unsupported dtype for this entry point */
  TOPT_ESHAPE = 3,     /* unsupported or inconsistent shape */
  TOPT_ECUDA = 4,      /* a CUDA launch or runtime call failed */
  TOPT_ETIMEOUT = 5,   /* reserved: a bounded device-side wait gave up */
  TOPT_EWORKSPACE = 6  /* workspace NULL or smaller than the query returned */
} topt_status;

typedef enum { TOPT_PRE = 0, TOPT_POST = 1 } topt_mode;

/* Estimators of the discarded exponent sum E~ [TopTheta §3.2.1]:
 *   EXACT    E~ = sum over discarded keys of exp(a_j - m)
 *   EXPTH    E~ = gamma * (L - k~) * exp(theta - m)   (gamma: 0.05 in the paper)
 *   OFFLINE  E~ = e_tilde[h][L-1], a static table calibrated beside theta by
 *            topt_calibrate_sdc (looked up like theta); used as it is,
 *            whatever the row itself keeps
 * m is the row maximum.  SDC applies to pre-softmax only; post-softmax ignores
 * the field. */
typedef enum {
  TOPT_SDC_NONE = 0,
  TOPT_SDC_EXACT = 1,
  TOPT_SDC_EXPTH = 2,
  TOPT_SDC_OFFLINE = 3
} topt_sdc;

typedef enum { TOPT_BF16 = 0, TOPT_F32 = 1 } topt_dtype;

/* GQA group policies of decode [TopTheta §4.6, the two alternatives to each
 * head using only its own selection]:
 *   OWN    each head keeps its own selection (the paper's experiments)
 *   UNION  every head of a group uses the union of the group's selections,
 *          which reads no extra V row
 *   VOTE   a key a head keeps survives only if at least gqa_min_heads heads
 *          of the group keep it; V rows requested by fewer heads are not read
 * Each head then normalises over its final set (R, k~, SDC, beta).  kept,
 * vrows and mask report the final sets. */
typedef enum { TOPT_GQA_OWN = 0, TOPT_GQA_UNION = 1, TOPT_GQA_VOTE = 2 } topt_gqa_policy;

/* ------------------------------------------------------------------------ */
/* Decode: one query token per sequence against its KV cache.               */
/* [TopTheta §2.2 (generative decoding), Fig. 1, §3.2, §4.6 (GQA)]          */
/* ------------------------------------------------------------------------ */
typedef struct {
  int32_t batch;        /* B >= 1 */
  int32_t n_q_heads;    /* Hq */
  int32_t n_kv_heads;   /* Hkv; Hq % Hkv == 0, Hq / Hkv <= 8, B * Hkv <= 2^26 */
  int32_t head_dim;     /* d: 64 or 128 */
  int32_t cache_len;    /* Nmax: token capacity of each cache, 1 .. 2^24 - 1 */
  int32_t theta_len;    /* Lmax >= 1: entries per head of `theta` */
  int32_t mode;         /* topt_mode */
  int32_t sdc;          /* topt_sdc */
  int32_t vmc;          /* nonzero: add beta * mu  [Eq. 7] */
  float gamma;          /* exp-threshold constant (TOPT_SDC_EXPTH) */
  const void* q;        /* [B][Hq][d] bf16 */
  const void* k_cache;  /* [B][Hkv][Nmax][d] bf16 */
  const void* v_cache;  /* [B][Hkv][Nmax][d] bf16 */
  const int32_t* seq_len; /* [B] keys per sequence incl. the current token, 1..Nmax */
  const float* theta;   /* [Hq][Lmax] fp32, the layer's slice of the table */
  const float* e_tilde; /* [Hq][Lmax] fp32 offline E~; required for TOPT_SDC_OFFLINE
                           with TOPT_PRE, else ignored (may be NULL) */
  const float* mu;      /* [B][Hkv][d] fp32 mean V row; required when vmc != 0 */
  float* out;           /* [B][Hq][d] fp32 */
  int32_t* kept;        /* [B][Hq] k~ per head, or NULL */
  int32_t* vrows;       /* [B][Hkv] V rows read (union over the group), or NULL */
  uint32_t* mask;       /* [B][Hq][ceil(Nmax/32)] kept bitmap (bit j%32 of word j/32), or NULL */
  int32_t* status;      /* device-side error word, or NULL */
  /* Scratch, >= topt_decode_workspace() bytes, 256-byte aligned: the fp32
   * scores of the call ([B][Hkv][Nmax rounded up to 32][G rounded up to
   * even]).  Every score is written before it is read, so the contents need
   * no initialisation and one workspace serves any number of calls. */
  void* workspace;
  size_t workspace_bytes;
  /* Optional profiling hook: cudaEvent_t handles (or NULL) recorded on
   * `stream` right before [0] and right after [1] the decode kernel; [2] is
   * not used.  The call is one kernel, launched so that it may start while
   * the previous kernel of the stream drains; an event in between removes
   * that overlap. */
  void* events[3];
  int32_t gqa_policy;     /* topt_gqa_policy; 0 (OWN) when zero-initialised */
  int32_t gqa_min_heads;  /* TOPT_GQA_VOTE: t >= 1 heads (t = 1 is OWN); else ignored */
} topt_decode_args;

/* Bytes of workspace topt_decode needs for these shapes (pointers unused). */
topt_status topt_decode_workspace(const topt_decode_args* args, size_t* bytes);

/* out[b][h] = Top-theta attention of q[b][h] over keys 0..seq_len[b]-1 of
 * KV head h / (Hq/Hkv).  The whole K row range is read; only V rows kept by
 * at least one head of the group are read.  Masked bits beyond seq_len[b]
 * are written as 0.  A sequence with seq_len[b] outside 1..Nmax sets *status
 * to TOPT_EINVAL and leaves its outputs untouched. */
topt_status topt_decode(const topt_decode_args* args, topt_stream stream);

/* Same operation as topt_decode, for callers that cannot allocate device
 * memory themselves (for example an application whose memory budget is fixed
 * at start-up, or code embedded in a framework whose allocator owns all device
 * memory).  This entry point has no counterpart in the paper; it only changes
 * where the scratch memory comes from.
 *   - args->workspace and args->workspace_bytes are ignored.  The scratch is
 *     one 32 MiB array that the library holds in device memory of every GPU
 *     that loads it, until the process exits.  Shapes that need more than
 *     32 MiB (topt_decode_workspace) return TOPT_EWORKSPACE and launch nothing.
 *   - Nothing is allocated: no cudaMalloc, no cudaFree, no allocating library
 *     call.  The first call on a device looks up the array's device address
 *     (with that device current) and keeps it for the life of the process;
 *     make that first call before any stream capture, and do not use this
 *     entry point across a cudaDeviceReset of that device.  The array keeps
 *     the previous call's contents; the kernel writes every value it reads,
 *     so nothing has to be cleared between calls.
 *   - Every call on a device shares the one array: calls that overlap on the
 *     GPU (other streams, other threads) race and corrupt each other's
 *     results.  Serialise them. */
topt_status topt_decode_noalloc(const topt_decode_args* args, topt_stream stream);

/* ------------------------------------------------------------------------ */
/* Prefill: causal attention of S query rows; row i sees keys 0..i.         */
/* [TopTheta §2.2 (prefill phase), §3, §3.2]                                 */
/* ------------------------------------------------------------------------ */
typedef struct {
  int32_t batch;        /* B */
  int32_t n_q_heads;    /* Hq */
  int32_t n_kv_heads;   /* Hkv; Hq % Hkv == 0 */
  int32_t head_dim;     /* d: 64 or 128 */
  int32_t seq;          /* S >= 1 */
  int32_t theta_len;    /* Lmax */
  int32_t dtype;        /* topt_dtype of q, k, v */
  int32_t mode, sdc, vmc;
  float gamma;
  const void* q;        /* [B][Hq][S][d] */
  const void* k;        /* [B][Hkv][S][d] */
  const void* v;        /* [B][Hkv][S][d] */
  const float* theta;   /* [Hq][Lmax] */
  const float* e_tilde; /* [Hq][Lmax] offline E~ (TOPT_SDC_OFFLINE with TOPT_PRE), else NULL */
  float* out;           /* [B][Hq][S][d] fp32, 16-byte aligned; VMC uses the prefix mean of
                           V rows 0..i.  q, k, v are 16-byte aligned too. */
  int32_t* kept;        /* [B][Hq][S] k~ per row, or NULL */
  uint32_t* mask;       /* [B][Hq][S][ceil(S/32)] kept bitmap, or NULL */
  unsigned long long* tiles; /* [2] += (P.V tiles executed, causal tiles), or NULL */
  int32_t* status;
  void* workspace;
  size_t workspace_bytes;
  /* Optional profiling hook: cudaEvent_t handles (or NULL) recorded on
   * `stream` right before [0] and right after [1] the attention kernel (after
   * the preparation kernels: prefix means, fp16 copy of V). */
  void* events[2];
} topt_prefill_args;

topt_status topt_prefill_workspace(const topt_prefill_args* args, size_t* bytes);
/* Row and key extent of the tiles counted in `tiles` for these arguments. */
topt_status topt_prefill_tile_shape(const topt_prefill_args* args, int32_t* tile_rows,
                                    int32_t* tile_keys);
topt_status topt_prefill(const topt_prefill_args* args, topt_stream stream);

/* Test hook of the bounded waits: topt_prefill (bf16 only, status required)
 * with the first K tile of every 128-row block never loaded, so a wait of the
 * tensor-core kernel runs out (1 s per block).  The kernel then stops every
 * role, drains its own copies and MMAs, frees its tensor memory and sets
 * *status = TOPT_ETIMEOUT; out is undefined.  Nothing faults and the CUDA
 * context stays usable.  Not part of the method. */
topt_status topt_prefill_test_timeout(const topt_prefill_args* args, topt_stream stream);

/* ------------------------------------------------------------------------ */
/* Calibration [TopTheta §3.1, Algorithm 1], one layer per call.            */
/* ------------------------------------------------------------------------ */
enum { TOPT_CALIB_RESET = 1, TOPT_CALIB_FINALIZE = 2, TOPT_CALIB_FIT = 4 };

typedef struct {
  int32_t n_seqs;       /* N >= 0 calibration sequences in this call */
  int32_t n_q_heads;    /* Hq */
  int32_t n_kv_heads;   /* Hkv */
  int32_t head_dim;     /* d: 64 or 128 */
  int32_t n_rows;       /* R query rows per sequence */
  int32_t n_keys;       /* Nk keys per sequence */
  int32_t theta_len;    /* Lmax */
  int32_t dtype;        /* topt_dtype of q and keys */
  int32_t mode;         /* topt_mode: quantile taken on a (PRE) or softmax(a) (POST) */
  int32_t k;            /* target kept elements per row, >= 1 */
  float alpha;          /* offset in standard deviations */
  int32_t flags;        /* TOPT_CALIB_RESET: zero the accumulators first;
                           TOPT_CALIB_FINALIZE: write theta after accumulating;
                           TOPT_CALIB_FIT (with FINALIZE): write the fitted
                           function of ln L described below instead of the
                           nearest-row fill */
  const void* q;        /* [N][Hq][R][d] */
  const void* keys;     /* [N][Hkv][Nk][d] */
  const int32_t* row_len; /* [R] keys seen by each query row, 1..Nk (causal prefill: r+1) */
  double* acc;          /* [2][Hq][Lmax] running sum and sum of squares of samples */
  int32_t* count;       /* [Hq][Lmax] number of samples */
  float* theta;         /* [Hq][Lmax] written on FINALIZE */
  int32_t* status;
  void* workspace;
  size_t workspace_bytes;
} topt_calib_args;

/* Minimum workspace is one row of scores per 8 rows; more lets a call process
 * more rows per launch.  *bytes is the size that processes every row of the
 * call at once, capped at 1 GiB. */
topt_status topt_calibrate_workspace(const topt_calib_args* args, size_t* bytes);

/* For every sequence, query head h and row i with L = row_len[i] > k: adds
 * the k-th largest score of the row (PRE) or its softmax value (POST) to the
 * accumulators at [h][L-1].  FINALIZE then writes, per head and L:
 *   count > 0         mean + alpha * std (std with ddof 1; 0 for one sample)
 *   L <= k            -INFINITY (the row is kept whole)
 *   otherwise         the value of the nearest calibrated L (ties: smaller L);
 *                     -INFINITY if the head has no calibrated row.
 * With TOPT_CALIB_FIT every L > k instead takes a least-squares line in
 * ln L through the n calibrated values (PRE; a constant when n = 1), or exp
 * of one through their logarithms (POST, positive values only); a head with
 * no usable value is dense.  The paper mentions fitting thresholds as a
 * function of the sequence length without giving the form. */
topt_status topt_calibrate(const topt_calib_args* args, topt_stream stream);

/* ------------------------------------------------------------------------ */
/* Offline-calibrated SDC [TopTheta §3.2.1, estimator 1], one layer per      */
/* call: a static E~ per (head, row) calibrated beside a pre-softmax theta.  */
/* ------------------------------------------------------------------------ */
typedef struct {
  int32_t n_seqs;       /* N >= 0 calibration sequences in this call */
  int32_t n_q_heads;    /* Hq */
  int32_t n_kv_heads;   /* Hkv */
  int32_t head_dim;     /* d: 64 or 128 */
  int32_t n_rows;       /* R query rows per sequence */
  int32_t n_keys;       /* Nk keys per sequence */
  int32_t theta_len;    /* Lmax */
  int32_t dtype;        /* topt_dtype of q and keys */
  int32_t flags;        /* TOPT_CALIB_RESET / TOPT_CALIB_FINALIZE, as topt_calibrate */
  const void* q;        /* [N][Hq][R][d] */
  const void* keys;     /* [N][Hkv][Nk][d] */
  const int32_t* row_len; /* [R] keys seen by each query row, 1..min(Nk, Lmax) */
  const float* theta;   /* [Hq][Lmax] pre-softmax thresholds the table is for (input) */
  double* acc;          /* [Hq][Lmax] running sum of E samples */
  int32_t* count;       /* [Hq][Lmax] number of samples */
  float* e_tilde;       /* [Hq][Lmax] written on FINALIZE */
  int32_t* status;
  void* workspace;
  size_t workspace_bytes;
} topt_sdc_calib_args;

/* Same workspace rule as topt_calibrate_workspace. */
topt_status topt_calibrate_sdc_workspace(const topt_sdc_calib_args* args, size_t* bytes);

/* For every sequence, head h and row i with L = row_len[i] and a finite
 * theta[h][L-1]: adds E = sum over keys j < L with a_j < theta of
 * exp(a_j - m) (m the row maximum) to the accumulators at [h][L-1].
 * FINALIZE then writes, per head and L:
 *   theta = -INFINITY  0 (the row is kept whole)
 *   count > 0          the mean of the samples
 *   otherwise          the mean of the nearest sampled L (ties: smaller L);
 *                      0 if the head has no sample. */
topt_status topt_calibrate_sdc(const topt_sdc_calib_args* args, topt_stream stream);

/* ------------------------------------------------------------------------ */
/* Multi-k cumulative calibration (MKC) [TopTheta App. D, Algorithm 2,      */
/* Eq. 8], one layer per call: the threshold tables of several target k     */
/* from one pass over the calibration rows, so that k can be chosen when    */
/* serving by offsetting the theta pointer by ki * Hq * Lmax.                */
/* ------------------------------------------------------------------------ */
typedef struct {
  int32_t n_seqs;       /* N >= 1 calibration sequences */
  int32_t n_q_heads;    /* Hq (<= 65535) */
  int32_t n_kv_heads;   /* Hkv */
  int32_t head_dim;     /* d: 64 or 128 */
  int32_t n_rows;       /* R query rows per sequence */
  int32_t n_keys;       /* Nk keys per sequence, < 2^20 */
  int32_t theta_len;    /* Lmax */
  int32_t dtype;        /* topt_dtype of q and keys */
  int32_t mode;         /* topt_mode: intervals of a (PRE) or of softmax(a) (POST) */
  int32_t n_k;          /* number of target k values, 1..65535 */
  const int32_t* ks;    /* [n_k] device, each >= 1 (any order, repeats allowed) */
  const void* q;        /* [N][Hq][R][d] device, 16-byte aligned */
  const void* keys;     /* [N][Hkv][Nk][d] device, 16-byte aligned */
  const int32_t* row_len; /* [R] device: keys seen by each query row, 1..min(Nk, Lmax) */
  float* theta;         /* [n_k][Hq][Lmax] device, written */
  int32_t* status;      /* device int32 or NULL; set to TOPT_EINVAL on a bad row_len
                           or k, or when more than 4096 rows (N times the rows of
                           one length) share a head and a length; theta is then
                           undefined */
  void* workspace;      /* device, 256-byte aligned, caller-owned */
  size_t workspace_bytes;
} topt_mkc_args;

/* Minimum workspace: the row index, n_k*Hq*Lmax floats and the scores of one
 * head (N*R*Nk floats); every further head's scores let one pass cover more
 * heads.  *bytes covers all heads at once, capped at 1 GiB (but not below
 * the minimum). */
topt_status topt_calibrate_multik_workspace(const topt_mkc_args* args, size_t* bytes);

/* For every head h and row length r that some row has, the calibration rows
 * of length r of all N sequences give the function k_bar_r(theta) of Eq. 8:
 * the mean, over the rows whose [min, max) holds theta, of the number of
 * their scores (PRE) or softmax values (POST) above theta.  Then, per target
 * k (index ki):
 *   theta[ki][h][r-1] = sup{theta : k_bar_r(theta) >= k}, one of the
 *                       calibration values (the paper leaves the inverse of
 *                       k_bar open; this is the largest threshold up to
 *                       which the rows keep at least k on average), or
 *                       -INFINITY when no theta reaches k;
 *   L <= k            -INFINITY (the row is kept whole);
 *   other L           the value of the nearest calibrated r > k (ties:
 *                     smaller r); -INFINITY if there is none.
 * For N = 1 and a row whose k-th largest value exceeds its minimum, the
 * result is that k-th largest value, as Algorithm 1 gives with alpha = 0. */
topt_status topt_calibrate_multik(const topt_mkc_args* args, topt_stream stream);

/* Building block of calibration, exposed for testing: out[r] = the k-th
 * largest of x[r][0 .. row_len[r]-1] (x is [rows][row_stride] fp32 on the
 * device; -0.0 counts as +0.0; -INFINITY if row_len[r] < k).  Exact: the
 * result is one of the inputs, bit for bit. */
topt_status topt_select_kth(const float* x, int32_t rows, int32_t row_stride,
                            const int32_t* row_len, int32_t k, float* out,
                            int32_t* status, topt_stream stream);

/* ------------------------------------------------------------------------ */
/* Running mean of V rows [TopTheta §3.2.2: in decode, mu is updated with    */
/* each new row instead of being recomputed]                                  */
/* ------------------------------------------------------------------------ */
typedef struct {
  int32_t batch, n_kv_heads, head_dim, cache_len;
  int32_t dtype;        /* topt_dtype of v_cache (and of k_cache, k_new, v_new) */
  int32_t n_new;        /* t >= 1 rows appended per sequence */
  void* v_cache;        /* [B][Hkv][Nmax][d]; written only when v_new is given */
  const int32_t* n_old; /* [B] rows already in mu; new rows are n_old..n_old+t-1 */
  float* mu;            /* [B][Hkv][d] fp32, updated in place */
  int32_t* status;
  /* Optional append of the step's new rows (NULL: the caches already hold
   * them).  v_new [B][Hkv][t][d] is copied to v_cache rows n_old.. and its
   * values are the ones averaged; k_new [B][Hkv][t][d] is copied to k_cache
   * [B][Hkv][Nmax][d] rows n_old.. (k_cache required with k_new).  16-byte
   * aligned, dtype as v_cache. */
  void* k_cache;
  const void* k_new;
  const void* v_new;
} topt_vmean_args;

/* mu <- (n_old * mu + sum of the t new rows) / (n_old + t).  t = 1 is the
 * per-token decode update; n_old = 0, t = S initialises mu from a prefill.
 * With k_new / v_new the same launch first appends the new K and V rows. */
topt_status topt_vmean_update(const topt_vmean_args* args, topt_stream stream);

/* Library version (major*10000 + minor*100 + patch) and status names. */
int32_t topt_version(void);
const char* topt_status_string(topt_status s);

#ifdef __cplusplus
}
#endif
#endif /* TOPT_H_ */

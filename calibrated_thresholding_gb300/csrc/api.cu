// C ABI of libtopt: host-side validation, workspace queries and launches.
// The operations are defined in topt.h; this file only checks arguments and
// dispatches to the kernels (decode.cu, prefill.cu, calibrate.cu, vmean.cu).
#include <cmath>

#include "common.cuh"
#include "internal.h"

using namespace topt;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool dim_ok(int d) { return d == 64 || d == 128; }

topt_status cuda_status(cudaError_t e) { return e == cudaSuccess ? TOPT_OK : TOPT_ECUDA; }

topt_status check_common_mode(int mode, int sdc) {
  if (mode != TOPT_PRE && mode != TOPT_POST) return TOPT_EINVAL;
  if (sdc < TOPT_SDC_NONE || sdc > TOPT_SDC_OFFLINE) return TOPT_EINVAL;
  return TOPT_OK;
}

topt_status check_decode_shape(const topt_decode_args* a) {
  if (!a) return TOPT_EINVAL;
  if (a->batch < 1 || a->n_q_heads < 1 || a->n_kv_heads < 1 || a->cache_len < 1 || a->theta_len < 1)
    return TOPT_ESHAPE;
  if (!dim_ok(a->head_dim)) return TOPT_ESHAPE;
  if (a->n_q_heads % a->n_kv_heads != 0) return TOPT_ESHAPE;
  if (a->n_q_heads / a->n_kv_heads > 8) return TOPT_ESHAPE;
  if ((long)a->batch * a->n_kv_heads > decode_max_pairs()) return TOPT_ESHAPE;
  if (a->cache_len > decode_max_cache()) return TOPT_ESHAPE;
  if (a->gqa_policy < TOPT_GQA_OWN || a->gqa_policy > TOPT_GQA_VOTE) return TOPT_EINVAL;
  if (a->gqa_policy == TOPT_GQA_VOTE && a->gqa_min_heads < 1) return TOPT_EINVAL;
  return check_common_mode(a->mode, a->sdc);
}

topt_status check_prefill_shape(const topt_prefill_args* a) {
  if (!a) return TOPT_EINVAL;
  if (a->batch < 1 || a->n_q_heads < 1 || a->n_kv_heads < 1 || a->seq < 1 || a->theta_len < 1)
    return TOPT_ESHAPE;
  if (!dim_ok(a->head_dim)) return TOPT_ESHAPE;
  if (a->n_q_heads % a->n_kv_heads != 0) return TOPT_ESHAPE;
  if (a->dtype != TOPT_BF16 && a->dtype != TOPT_F32) return TOPT_EDTYPE;
  if ((size_t)a->batch * a->n_q_heads > 65535u * 1024u || a->n_q_heads > 65535 || a->batch > 65535)
    return TOPT_ESHAPE;
  // tensor-core grid: one CTA per 128 query rows of every (batch, head)
  if ((size_t)a->batch * a->n_q_heads * ((size_t)(a->seq + 127) / 128) > 0x7fffffffu) return TOPT_ESHAPE;
  return check_common_mode(a->mode, a->sdc);
}

topt_status check_calib_shape(const topt_calib_args* a) {
  if (!a) return TOPT_EINVAL;
  if (a->n_seqs < 0 || a->n_q_heads < 1 || a->n_kv_heads < 1 || a->theta_len < 1) return TOPT_ESHAPE;
  if (a->n_seqs > 0 && (a->n_rows < 1 || a->n_keys < 1)) return TOPT_ESHAPE;
  if (!dim_ok(a->head_dim)) return TOPT_ESHAPE;
  if (a->n_q_heads % a->n_kv_heads != 0) return TOPT_ESHAPE;
  if (a->dtype != TOPT_BF16 && a->dtype != TOPT_F32) return TOPT_EDTYPE;
  if (a->mode != TOPT_PRE && a->mode != TOPT_POST) return TOPT_EINVAL;
  if (a->k < 1) return TOPT_EINVAL;
  if (!std::isfinite(a->alpha)) return TOPT_EINVAL;
  if (a->flags & ~(TOPT_CALIB_RESET | TOPT_CALIB_FINALIZE | TOPT_CALIB_FIT)) return TOPT_EINVAL;
  return TOPT_OK;
}

topt_status check_mkc_shape(const topt_mkc_args* a) {
  if (!a) return TOPT_EINVAL;
  if (a->n_seqs < 1 || a->n_q_heads < 1 || a->n_kv_heads < 1 || a->n_rows < 1 || a->n_keys < 1 ||
      a->theta_len < 1)
    return TOPT_ESHAPE;
  if (!dim_ok(a->head_dim)) return TOPT_ESHAPE;
  if (a->n_q_heads % a->n_kv_heads != 0 || a->n_q_heads > 65535) return TOPT_ESHAPE;
  if (a->dtype != TOPT_BF16 && a->dtype != TOPT_F32) return TOPT_EDTYPE;
  if (a->mode != TOPT_PRE && a->mode != TOPT_POST) return TOPT_EINVAL;
  if (a->n_k < 1 || a->n_k > 65535) return TOPT_EINVAL;
  // pooled counts of one (head, length) group stay below 2^32
  if (a->n_keys >= (1 << 20)) return TOPT_ESHAPE;
  if ((size_t)a->n_seqs * a->n_q_heads * a->n_rows > 0x7fffffffu) return TOPT_ESHAPE;
  return TOPT_OK;
}

}  // namespace

extern "C" {

int32_t topt_version(void) { return 100; }

const char* topt_status_string(topt_status s) {
  switch (s) {
    case TOPT_OK: return "ok";
    case TOPT_EINVAL: return "invalid argument";
    case TOPT_EDTYPE: return "unsupported dtype";
    case TOPT_ESHAPE: return "unsupported shape";
    case TOPT_ECUDA: return "CUDA error";
    case TOPT_ETIMEOUT: return "device wait timed out";
    case TOPT_EWORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

// ------------------------------------------------------------------ decode
topt_status topt_decode_workspace(const topt_decode_args* a, size_t* bytes) {
  topt_status st = check_decode_shape(a);
  if (st != TOPT_OK) return st;
  if (!bytes) return TOPT_EINVAL;
  *bytes = decode_workspace_bytes(*a);
  return TOPT_OK;
}

topt_status topt_decode(const topt_decode_args* a, topt_stream stream) {
  topt_status st = check_decode_shape(a);
  if (st != TOPT_OK) return st;
  if (!a->q || !a->k_cache || !a->v_cache || !a->seq_len || !a->theta || !a->out) return TOPT_EINVAL;
  if (a->vmc && !a->mu) return TOPT_EINVAL;
  if (!aligned16(a->q) || !aligned16(a->k_cache) || !aligned16(a->v_cache)) return TOPT_EINVAL;
  if (a->sdc == TOPT_SDC_EXPTH && !(a->gamma >= 0.f && std::isfinite(a->gamma))) return TOPT_EINVAL;
  if (a->mode == TOPT_PRE && a->sdc == TOPT_SDC_OFFLINE && !a->e_tilde) return TOPT_EINVAL;
  const size_t need = decode_workspace_bytes(*a);
  if (!a->workspace || a->workspace_bytes < need || (reinterpret_cast<uintptr_t>(a->workspace) & 255u))
    return TOPT_EWORKSPACE;
  return cuda_status(decode_launch(*a, (cudaStream_t)stream));
}

topt_status topt_decode_noalloc(const topt_decode_args* a, topt_stream stream) {
  topt_status st = check_decode_shape(a);
  if (st != TOPT_OK) return st;
  if (!a->q || !a->k_cache || !a->v_cache || !a->seq_len || !a->theta || !a->out) return TOPT_EINVAL;
  if (a->vmc && !a->mu) return TOPT_EINVAL;
  if (!aligned16(a->q) || !aligned16(a->k_cache) || !aligned16(a->v_cache)) return TOPT_EINVAL;
  if (a->sdc == TOPT_SDC_EXPTH && !(a->gamma >= 0.f && std::isfinite(a->gamma))) return TOPT_EINVAL;
  if (a->mode == TOPT_PRE && a->sdc == TOPT_SDC_OFFLINE && !a->e_tilde) return TOPT_EINVAL;
  if (decode_workspace_bytes(*a) > decode_noalloc_capacity()) return TOPT_EWORKSPACE;
  return cuda_status(decode_noalloc_launch(*a, (cudaStream_t)stream));
}

// ----------------------------------------------------------------- prefill
topt_status topt_prefill_workspace(const topt_prefill_args* a, size_t* bytes) {
  topt_status st = check_prefill_shape(a);
  if (st != TOPT_OK) return st;
  if (!bytes) return TOPT_EINVAL;
  *bytes = prefill_workspace_bytes(*a);
  return TOPT_OK;
}

topt_status topt_prefill_tile_shape(const topt_prefill_args* a, int32_t* rows, int32_t* keys) {
  topt_status st = check_prefill_shape(a);
  if (st != TOPT_OK) return st;
  if (!rows || !keys) return TOPT_EINVAL;
  prefill_tile_shape(*a, rows, keys);
  return TOPT_OK;
}

topt_status topt_prefill(const topt_prefill_args* a, topt_stream stream) {
  topt_status st = check_prefill_shape(a);
  if (st != TOPT_OK) return st;
  if (!a->q || !a->k || !a->v || !a->theta || !a->out) return TOPT_EINVAL;
  if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v) || !aligned16(a->out))
    return TOPT_EINVAL;
  if (a->sdc == TOPT_SDC_EXPTH && !(a->gamma >= 0.f && std::isfinite(a->gamma))) return TOPT_EINVAL;
  if (a->mode == TOPT_PRE && a->sdc == TOPT_SDC_OFFLINE && !a->e_tilde) return TOPT_EINVAL;
  const size_t need = prefill_workspace_bytes(*a);
  if (need > 0 && (!a->workspace || a->workspace_bytes < need ||
                   (reinterpret_cast<uintptr_t>(a->workspace) & 255u)))
    return TOPT_EWORKSPACE;
  return cuda_status(prefill_launch(*a, (cudaStream_t)stream));
}

topt_status topt_prefill_test_timeout(const topt_prefill_args* a, topt_stream stream) {
  topt_status st = check_prefill_shape(a);
  if (st != TOPT_OK) return st;
  if (a->dtype != TOPT_BF16 || !a->status) return TOPT_EINVAL;
  if (!a->q || !a->k || !a->v || !a->theta || !a->out) return TOPT_EINVAL;
  if (a->mode == TOPT_PRE && a->sdc == TOPT_SDC_OFFLINE && !a->e_tilde) return TOPT_EINVAL;
  if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v) || !aligned16(a->out))
    return TOPT_EINVAL;
  const size_t need = prefill_workspace_bytes(*a);
  if (need > 0 && (!a->workspace || a->workspace_bytes < need ||
                   (reinterpret_cast<uintptr_t>(a->workspace) & 255u)))
    return TOPT_EWORKSPACE;
  return cuda_status(prefill_launch(*a, (cudaStream_t)stream, 1));
}

// --------------------------------------------------------------- calibrate
topt_status topt_calibrate_workspace(const topt_calib_args* a, size_t* bytes) {
  topt_status st = check_calib_shape(a);
  if (st != TOPT_OK) return st;
  if (!bytes) return TOPT_EINVAL;
  const size_t rows = (size_t)a->n_seqs * a->n_q_heads * a->n_rows;
  size_t want = calibrate_workspace_bytes(*a, rows > 0 ? rows : 1);
  const size_t cap = (size_t)1 << 30;
  const size_t minimum = calibrate_workspace_bytes(*a, calibrate_min_rows_per_pass());
  if (want > cap) want = cap > minimum ? cap : minimum;
  *bytes = want;
  return TOPT_OK;
}

topt_status topt_calibrate(const topt_calib_args* a, topt_stream stream) {
  topt_status st = check_calib_shape(a);
  if (st != TOPT_OK) return st;
  if (!a->acc || !a->count) return TOPT_EINVAL;
  if ((a->flags & TOPT_CALIB_FINALIZE) && !a->theta) return TOPT_EINVAL;
  if (a->n_seqs > 0) {
    if (!a->q || !a->keys || !a->row_len) return TOPT_EINVAL;
    if (!aligned16(a->q) || !aligned16(a->keys)) return TOPT_EINVAL;
    const size_t minimum = calibrate_workspace_bytes(*a, calibrate_min_rows_per_pass());
    if (!a->workspace || a->workspace_bytes < minimum) return TOPT_EWORKSPACE;
  }
  return cuda_status(calibrate_launch(*a, (cudaStream_t)stream));
}

static topt_status check_sdc_calib_shape(const topt_sdc_calib_args* a) {
  if (!a) return TOPT_EINVAL;
  if (a->n_seqs < 0 || a->n_q_heads < 1 || a->n_kv_heads < 1 || a->theta_len < 1) return TOPT_ESHAPE;
  if (a->n_seqs > 0 && (a->n_rows < 1 || a->n_keys < 1)) return TOPT_ESHAPE;
  if (!dim_ok(a->head_dim)) return TOPT_ESHAPE;
  if (a->n_q_heads % a->n_kv_heads != 0) return TOPT_ESHAPE;
  if (a->dtype != TOPT_BF16 && a->dtype != TOPT_F32) return TOPT_EDTYPE;
  if (a->flags & ~(TOPT_CALIB_RESET | TOPT_CALIB_FINALIZE)) return TOPT_EINVAL;
  return TOPT_OK;
}

topt_status topt_calibrate_sdc_workspace(const topt_sdc_calib_args* a, size_t* bytes) {
  topt_status st = check_sdc_calib_shape(a);
  if (st != TOPT_OK) return st;
  if (!bytes) return TOPT_EINVAL;
  const size_t rows = (size_t)a->n_seqs * a->n_q_heads * a->n_rows;
  size_t want = calibrate_sdc_workspace_bytes(*a, rows > 0 ? rows : 1);
  const size_t cap = (size_t)1 << 30;
  const size_t minimum = calibrate_sdc_workspace_bytes(*a, calibrate_min_rows_per_pass());
  if (want > cap) want = cap > minimum ? cap : minimum;
  *bytes = want;
  return TOPT_OK;
}

topt_status topt_calibrate_sdc(const topt_sdc_calib_args* a, topt_stream stream) {
  topt_status st = check_sdc_calib_shape(a);
  if (st != TOPT_OK) return st;
  if (!a->acc || !a->count || !a->theta) return TOPT_EINVAL;
  if ((a->flags & TOPT_CALIB_FINALIZE) && !a->e_tilde) return TOPT_EINVAL;
  if (a->n_seqs > 0) {
    if (!a->q || !a->keys || !a->row_len) return TOPT_EINVAL;
    if (!aligned16(a->q) || !aligned16(a->keys)) return TOPT_EINVAL;
    const size_t minimum = calibrate_sdc_workspace_bytes(*a, calibrate_min_rows_per_pass());
    if (!a->workspace || a->workspace_bytes < minimum) return TOPT_EWORKSPACE;
  }
  return cuda_status(calibrate_sdc_launch(*a, (cudaStream_t)stream));
}

topt_status topt_calibrate_multik_workspace(const topt_mkc_args* a, size_t* bytes) {
  topt_status st = check_mkc_shape(a);
  if (st != TOPT_OK) return st;
  if (!bytes) return TOPT_EINVAL;
  const size_t fixed = calibrate_multik_fixed_bytes(*a), head = calibrate_multik_head_bytes(*a);
  const size_t minimum = fixed + head;
  size_t want = fixed + head * (size_t)a->n_q_heads;
  const size_t cap = (size_t)1 << 30;
  if (want > cap) want = cap > minimum ? cap : minimum;
  *bytes = want;
  return TOPT_OK;
}

topt_status topt_calibrate_multik(const topt_mkc_args* a, topt_stream stream) {
  topt_status st = check_mkc_shape(a);
  if (st != TOPT_OK) return st;
  if (!a->q || !a->keys || !a->row_len || !a->ks || !a->theta) return TOPT_EINVAL;
  if (!aligned16(a->q) || !aligned16(a->keys)) return TOPT_EINVAL;
  const size_t minimum = calibrate_multik_fixed_bytes(*a) + calibrate_multik_head_bytes(*a);
  if (!a->workspace || a->workspace_bytes < minimum || (reinterpret_cast<uintptr_t>(a->workspace) & 255u))
    return TOPT_EWORKSPACE;
  return cuda_status(calibrate_multik_launch(*a, (cudaStream_t)stream));
}

topt_status topt_select_kth(const float* x, int32_t rows, int32_t row_stride, const int32_t* row_len,
                            int32_t k, float* out, int32_t* status, topt_stream stream) {
  if (rows < 0 || row_stride < 1 || k < 1) return TOPT_EINVAL;
  if (rows > 0 && (!x || !row_len || !out)) return TOPT_EINVAL;
  return cuda_status(select_kth_launch(x, rows, row_stride, row_len, k, out, status, (cudaStream_t)stream));
}

// ------------------------------------------------------------------- vmean
topt_status topt_vmean_update(const topt_vmean_args* a, topt_stream stream) {
  if (!a) return TOPT_EINVAL;
  if (a->batch < 1 || a->n_kv_heads < 1 || a->cache_len < 1 || a->n_new < 1) return TOPT_ESHAPE;
  if (!dim_ok(a->head_dim)) return TOPT_ESHAPE;
  if (a->dtype != TOPT_BF16 && a->dtype != TOPT_F32) return TOPT_EDTYPE;
  if (a->n_new > a->cache_len) return TOPT_ESHAPE;
  if (!a->v_cache || !a->n_old || !a->mu) return TOPT_EINVAL;
  if (!aligned16(a->v_cache)) return TOPT_EINVAL;
  if (a->k_new && (!a->k_cache || !aligned16(a->k_cache) || !aligned16(a->k_new))) return TOPT_EINVAL;
  if (a->v_new && !aligned16(a->v_new)) return TOPT_EINVAL;
  return cuda_status(vmean_launch(*a, (cudaStream_t)stream));
}

}  // extern "C"

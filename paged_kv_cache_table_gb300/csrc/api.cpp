// Status strings and cache-description checks shared by every entry point.
#include <climits>

#include "pa_internal.h"

namespace pa {

pa_status validate_desc(const pa_cache_desc* d) {
  if (!d) return PA_ERR_INVALID_ARG;
  if (d->num_seqs < 0 || d->num_q_heads <= 0 || d->num_kv_heads <= 0 || d->head_dim <= 0 ||
      d->block_size <= 0 || d->num_blocks <= 0 || d->max_blocks_per_seq <= 0 || d->num_sink < 0 ||
      d->sliding_window < 0)
    return PA_ERR_INVALID_ARG;
  if (d->num_q_heads % d->num_kv_heads != 0) return PA_ERR_INVALID_ARG;
  if (d->block_size != PA_BLOCK_SIZE) return PA_ERR_UNSUPPORTED;
  if (d->head_dim != 64 && d->head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (d->num_q_heads / d->num_kv_heads > 8) return PA_ERR_UNSUPPORTED;
  // slot indices are 32-bit
  if ((long long)d->num_blocks * PA_BLOCK_SIZE > (long long)INT_MAX) return PA_ERR_INVALID_ARG;
  const bool bf16 = d->k_dtype == PA_BF16 && d->v_dtype == PA_BF16;
  const bool q8 = d->k_dtype == PA_FP8_E4M3 && d->v_dtype == PA_INT8;
  const bool q4 = d->k_dtype == PA_INT4 && d->v_dtype == PA_INT4;
  if (!bf16 && !q8 && !q4) {
    auto known = [](pa_dtype t) { return t == PA_BF16 || t == PA_FP8_E4M3 || t == PA_INT8 || t == PA_INT4; };
    return known(d->k_dtype) && known(d->v_dtype) ? PA_ERR_UNSUPPORTED : PA_ERR_INVALID_ARG;
  }
  if (q8) {
    if (d->head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (!d->k_scales || !d->v_scales) return PA_ERR_INVALID_ARG;
  }
  if (q4 && (d->head_dim != 128 || d->num_kv_heads % 2 != 0)) return PA_ERR_UNSUPPORTED;
  if (d->num_sink > 0 && (!d->k_sink || !d->v_sink)) return PA_ERR_INVALID_ARG;
  return PA_OK;
}

}  // namespace pa

extern "C" const char* pa_status_string(pa_status s) {
  switch (s) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_WORKSPACE_TOO_SMALL: return "PA_ERR_WORKSPACE_TOO_SMALL";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_OUT_OF_BLOCKS: return "PA_ERR_OUT_OF_BLOCKS";
  }
  return "PA_ERR_UNKNOWN";
}

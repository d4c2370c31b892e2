// Status strings, cache-description checks and per-device launch state shared by every entry point.
#include <cudaTypedefs.h>

#include <climits>
#include <map>
#include <mutex>
#include <utility>

#include "pa_internal.h"

namespace pa {

namespace {

// The driver's context calls, through the runtime's entry-point lookup (no link to libcuda).
struct CtxCalls {
  PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  PFN_cuCtxGetId_v12000 get_id = nullptr;
};

const CtxCalls& ctx_calls() {
  static CtxCalls calls;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      calls.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(ptr);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      calls.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(ptr);
  });
  return calls;
}

std::mutex g_launch_mu;
std::map<int, std::pair<unsigned long long, int>> g_sms;                         // device -> (context, SMs)
std::map<std::pair<const void*, unsigned long long>, size_t> g_smem_set;          // (kernel, context) -> bytes

}  // namespace

unsigned long long current_ctx_id() {
  const CtxCalls& c = ctx_calls();
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!c.get_current || !c.get_id || c.get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (c.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

int sm_count_current() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const unsigned long long ctx = current_ctx_id();
  std::lock_guard<std::mutex> lock(g_launch_mu);
  auto it = g_sms.find(dev);
  if (ctx != 0 && it != g_sms.end() && it->second.first == ctx) return it->second.second;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (ctx != 0) g_sms[dev] = {ctx, n};
  return n;
}

bool ensure_dynamic_smem(const void* kernel, size_t bytes) {
  const unsigned long long ctx = current_ctx_id();
  std::lock_guard<std::mutex> lock(g_launch_mu);
  if (ctx != 0) {
    auto it = g_smem_set.find({kernel, ctx});
    if (it != g_smem_set.end() && it->second >= bytes) return true;
  }
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)) !=
      cudaSuccess)
    return false;
  if (ctx != 0) g_smem_set[{kernel, ctx}] = bytes;
  return true;
}

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
  const bool q8t = d->k_dtype == PA_FP8_E4M3_TOKEN && d->v_dtype == PA_INT8;
  const bool q4 = d->k_dtype == PA_INT4 && d->v_dtype == PA_INT4;
  if (!bf16 && !q8 && !q8t && !q4) {
    auto known = [](pa_dtype t) {
      return t == PA_BF16 || t == PA_FP8_E4M3 || t == PA_INT8 || t == PA_INT4 || t == PA_FP8_E4M3_TOKEN;
    };
    return known(d->k_dtype) && known(d->v_dtype) ? PA_ERR_UNSUPPORTED : PA_ERR_INVALID_ARG;
  }
  if (q8) {
    if (d->head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (!d->k_scales || !d->v_scales) return PA_ERR_INVALID_ARG;
  }
  if (q8t) {
    // the scales of a block's heads move as 16-byte TMA rows: num_kv_heads a multiple of 4
    if (d->head_dim != 128 || d->num_kv_heads % 4 != 0) return PA_ERR_UNSUPPORTED;
    if (!d->v_scales) return PA_ERR_INVALID_ARG;
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

// Copy-on-write block copy.
//
// "KV Cache 的显存账本：PagedAttention 与连续批处理" §四: requests with a common prefix point
// at the same physical blocks and copy only where they diverge.  "大模型推理KV Cache显存优化：
// 从PagedAttention到AI内存系统演进" §3.2: a sequence that must write into a shared block first
// copies it, so the other sequences never see the write.
//
// A physical block is one contiguous chunk (16 slots x kv_heads x head_dim) in the slot-major
// cache.  Grid: (pair, tensor); each CTA streams one block of K or V with 16-byte vectors.

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

// grid.y = tensor (K, V) x region: region 0 is the block's codes (block_vecs vectors per block),
// region 1 its group parameters (int4 pools) or per-token scales (K of a PA_FP8_E4M3_TOKEN pool):
// param_vecs per block at param_base, for the tensors whose bit is set in param_mask.
__global__ void __launch_bounds__(256) block_copy_kernel(const int32_t* pairs, int num_blocks,
                                                         size_t block_vecs, size_t param_base,
                                                         size_t param_vecs, int param_mask, uint4* k_cache,
                                                         uint4* v_cache, int32_t* err) {
  const int i = blockIdx.x;
  const int src = pairs[2 * i];
  const int dst = pairs[2 * i + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0) set_error(err, PA_EFLAG_BAD_BLOCK_ID);
    return;
  }
  if (src == dst) return;
  if (blockIdx.y >= 2 && !((param_mask >> (blockIdx.y & 1)) & 1)) return;
  uint4* base = (blockIdx.y & 1) == 0 ? k_cache : v_cache;
  size_t n = block_vecs;
  if (blockIdx.y >= 2) {
    base += param_base;
    n = param_vecs;
  }
  const uint4* s = base + static_cast<size_t>(src) * n;
  uint4* d = base + static_cast<size_t>(dst) * n;
  for (size_t j = threadIdx.x; j < n; j += blockDim.x) d[j] = s[j];
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_block_copy(const pa_cache_desc* desc, void* k_cache, void* v_cache,
                                   const int32_t* src_dst_pairs, int n_pairs, int32_t* err_flag,
                                   void* stream) {
  pa_status st = pa::validate_desc(desc);
  if (st != PA_OK) return st;
  if (n_pairs < 0) return PA_ERR_INVALID_ARG;
  if (n_pairs == 0) return PA_OK;
  if (!k_cache || !v_cache || !src_dst_pairs) return PA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15u)
    return PA_ERR_INVALID_ARG;
  const bool int4 = pa::is_int4(desc), tok = pa::has_token_scales(desc);
  const size_t row = int4 ? pa::int4_code_row_bytes(desc)
                          : static_cast<size_t>(desc->head_dim) * pa::dtype_bytes(desc->k_dtype);
  const size_t kbytes = static_cast<size_t>(PA_BLOCK_SIZE) * desc->num_kv_heads * row;
  // int4: both tensors' group parameters; per-token K: 16 x num_kv_heads fp32 scales (a multiple
  // of 16 bytes, num_kv_heads being a multiple of 4)
  const size_t pbytes = int4  ? static_cast<size_t>(PA_BLOCK_SIZE) * desc->num_kv_heads * pa::int4_param_row_bytes(desc)
                        : tok ? static_cast<size_t>(PA_BLOCK_SIZE) * desc->num_kv_heads * 4
                              : 0;
  const size_t pbase = int4 ? pa::int4_params_offset(desc) : (tok ? pa::token_scales_offset(desc) : 0);
  const int mask = int4 ? 3 : (tok ? 1 : 0);
  pa::block_copy_kernel<<<dim3(n_pairs, mask ? 4 : 2), 256, 0, pa::as_stream(stream)>>>(
      src_dst_pairs, desc->num_blocks, kbytes / 16, pbase / 16, pbytes / 16, mask, static_cast<uint4*>(k_cache),
      static_cast<uint4*>(v_cache), err_flag);
  return pa::launch_status();
}

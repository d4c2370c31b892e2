// Host-side helpers shared by the translation units of the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <utility>

#include "pa.h"

namespace pa {

inline int dtype_bytes(pa_dtype t) { return t == PA_BF16 ? 2 : 1; }

inline bool is_quantized(const pa_cache_desc* d) { return d->k_dtype != PA_BF16; }

inline bool is_int4(const pa_cache_desc* d) { return d->k_dtype == PA_INT4; }

// PA_FP8_E4M3_TOKEN: the K pool holds every slot's codes, then an fp32 scale per (slot, head).
inline bool has_token_scales(const pa_cache_desc* d) { return d->k_dtype == PA_FP8_E4M3_TOKEN; }
inline size_t token_scales_offset(const pa_cache_desc* d) {
  return static_cast<size_t>(d->num_blocks) * PA_BLOCK_SIZE * d->num_kv_heads * d->head_dim;
}

// INT4 pools: code bytes of every slot first, then the group parameter words.
constexpr int kInt4Group = 32;
inline size_t int4_code_row_bytes(const pa_cache_desc* d) { return static_cast<size_t>(d->head_dim) / 2; }
inline size_t int4_param_row_bytes(const pa_cache_desc* d) {
  return static_cast<size_t>(d->head_dim) / kInt4Group * 4;
}
inline size_t int4_params_offset(const pa_cache_desc* d) {
  return static_cast<size_t>(d->num_blocks) * PA_BLOCK_SIZE * d->num_kv_heads * int4_code_row_bytes(d);
}

// Checks a cache description against what the kernels implement.
pa_status validate_desc(const pa_cache_desc* d);

// TMA descriptor of a paged cache pool viewed as (128-byte chunk, kv_head x chunk, slot) with
// boxes of `box_rows` chunks x 16 slots (tensor_map.cpp).
bool encode_cache_map(CUtensorMap* map, const void* base, int elem_bytes, int rows, int box_rows,
                      long long slots);

// TMA descriptor of a bf16 or 8-bit cache pool viewed as (128-byte chunk elements, chunk, slot,
// kv_head) with boxes of nc chunks x 16 slots x box_heads heads, landing head-major (tensor_map.cpp).
bool encode_cache_map_heads(CUtensorMap* map, const void* base, int elem_bytes, int heads, int nc, int box_heads,
                            long long slots);

// The same view with boxes of one 128-byte chunk x 16 slots x one head, landing as [slot][128 B]
// swizzled (tensor_map.cpp).
bool encode_cache_map_chunk(CUtensorMap* map, const void* base, int elem_bytes, int heads, int nc, long long slots);

// TMA descriptor of the INT4 group parameters viewed as (16-byte head row, kv_head, slot) with
// boxes of `box_heads` heads x 16 slots, no swizzle (tensor_map.cpp).
bool encode_param_map(CUtensorMap* map, const void* base, int heads, int box_heads, long long slots);

// TMA descriptor of per-token K scales [slots][heads] fp32 with boxes of box_heads heads x 16 slots,
// no swizzle (tensor_map.cpp).
bool encode_scale_map(CUtensorMap* map, const void* base, int heads, int box_heads, long long slots);

// TMA descriptor of bf16 queries [T][heads][128] viewed as (64 dims, half, head, token) with boxes
// of one half x G heads x tokens_per_box tokens, 128-byte swizzle (tensor_map.cpp).
bool encode_query_map(CUtensorMap* map, const void* base, int heads, int G, int tokens_per_box, long long tokens);

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Unique id of the calling thread's current CUDA context (never reused within a process), or 0
// when there is none yet or the driver cannot tell (api.cpp).
unsigned long long current_ctx_id();

// SMs of the current device, looked up once per context (0 on failure).
int sm_count_current();

// Raise a kernel's dynamic shared-memory limit to at least `bytes` in the current context; the
// runtime call is made only when a (kernel, context) pair needs more than it was given before.
bool ensure_dynamic_smem(const void* kernel, size_t bytes);

// The tcgen05 chunked-prefill kernel (prefill_tc.cu): head_dim 128 and a power-of-two number of
// query heads per KV head; arguments as pa_prefill_attention after its checks.
// step: the previous kernel on the stream is the append of this prefill step (it writes only
// K/V slots), so only the K/V copies wait for it.
pa_status launch_prefill_tc(const pa_cache_desc* desc, void* out, const void* q, const void* k_cache,
                            const void* v_cache, const int32_t* block_tables, const int32_t* q_start,
                            const int32_t* context_lens, int max_query_len, float scale, int32_t* err_flag,
                            cudaStream_t stream, bool step);

// Shared-prefix decode (shared_prefix.cu).  Per-sequence flags, zeroed then or-ed by the prefix
// kernel: kSharedMember = listed, in range, context covering the prefix; kSharedMismatch = some
// prefix block of its table differs from the first listed sequence's.  Exactly kSharedUse means
// the decode kernel starts past the prefix and the merge folds in the prefix's partial rows.
constexpr int kSharedMember = 1;
constexpr int kSharedMismatch = 2;
constexpr int kSharedUse = kSharedMember;
constexpr int kSharedChunkBlocks = 8;  // prefix blocks per partial row (128 keys)
inline int shared_prefix_chunks(int shared_len) {
  const int nsb = shared_len / PA_BLOCK_SIZE;
  return (nsb + kSharedChunkBlocks - 1) / kSharedChunkBlocks;
}
size_t shared_prefix_smem_bytes(int head_dim);

// Zeroes flags[0..num_seqs) and launches the prefix kernel: partial rows
// extra[s][chunk][h][head_dim + 4] (o, then m and l in log2 units) for every listed sequence s.
pa_status launch_shared_prefix(const pa_cache_desc* desc, const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, const int32_t* context_lens, int max_context_len,
                               float scale, const int32_t* shared_seqs, int n_shared, int shared_len,
                               int32_t* flags, float* extra, int32_t* err_flag, cudaStream_t stream);

inline pa_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// Launch with programmatic stream serialization: the kernel may begin while the previous
// kernel of the stream is still running and must call griddepcontrol.wait before touching
// anything that kernel writes.
template <typename... KArgs, typename... Args>
inline pa_status launch_overlapped(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                   cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa

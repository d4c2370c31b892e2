// TMA tensor maps over the slot-major paged cache (host side).
#include <cudaTypedefs.h>

#include <mutex>

#include "pa_internal.h"

namespace pa {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

}  // namespace

// The cache as a 3-D tensor: (128-byte chunk of a head row, kv_head x chunk, slot).  One box is
// `box_rows` consecutive 128-byte rows (chunks of one head row) of 16 consecutive slots, i.e. of
// one physical block, and lands in shared memory as [slot][row][128 B] with the 128-byte
// swizzle.
bool encode_cache_map(CUtensorMap* map, const void* base, int elem_bytes, int rows, int box_rows,
                      long long slots) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(128 / elem_bytes), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(slots)};
  cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(rows) * 128};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / elem_bytes), static_cast<cuuint32_t>(box_rows),
                       PA_BLOCK_SIZE};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt =
      elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  return fn(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The cache as a 4-D tensor (elements of a 128-byte chunk, chunk of the head row, slot, KV head)
// with boxes of every chunk x 16 slots x `box_heads` heads.  The box runs heads outermost, so it
// lands as [head][slot][chunk][128 B] with the 128-byte swizzle: each head's rows of a block form
// the same contiguous tile that a one-head box gives, and one box carries a block of many heads.
bool encode_cache_map_heads(CUtensorMap* map, const void* base, int elem_bytes, int heads, int nc, int box_heads,
                            long long slots) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(128 / elem_bytes), static_cast<cuuint64_t>(nc),
                        static_cast<cuuint64_t>(slots), static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[3] = {128, static_cast<cuuint64_t>(heads) * nc * 128, static_cast<cuuint64_t>(nc) * 128};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / elem_bytes), static_cast<cuuint32_t>(nc), PA_BLOCK_SIZE,
                       static_cast<cuuint32_t>(box_heads)};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType dt =
      elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  return fn(map, dt, 4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same 4-D view with boxes of one 128-byte chunk x 16 slots x one head: a box lands as
// [slot][128 B] with the 128-byte swizzle, so that eight consecutive slots take eight distinct
// swizzle phases.
bool encode_cache_map_chunk(CUtensorMap* map, const void* base, int elem_bytes, int heads, int nc, long long slots) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(128 / elem_bytes), static_cast<cuuint64_t>(nc),
                        static_cast<cuuint64_t>(slots), static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[3] = {128, static_cast<cuuint64_t>(heads) * nc * 128, static_cast<cuuint64_t>(nc) * 128};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / elem_bytes), 1, PA_BLOCK_SIZE, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType dt =
      elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  return fn(map, dt, 4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_param_map(CUtensorMap* map, const void* base, int heads, int box_heads, long long slots) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[3] = {4, static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(slots)};
  cuuint64_t strides[2] = {16, static_cast<cuuint64_t>(heads) * 16};
  cuuint32_t box[3] = {4, static_cast<cuuint32_t>(box_heads), PA_BLOCK_SIZE};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Per-token K scales [slots][heads] fp32 as a 2-D tensor with boxes of box_heads heads x 16 slots
// (one block), no swizzle: a box lands as [slot][head] fp32.  box_heads * 4 and heads * 4 must be
// multiples of 16 bytes.
bool encode_scale_map(CUtensorMap* map, const void* base, int heads, int box_heads, long long slots) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(slots)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(heads) * 4};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_heads), PA_BLOCK_SIZE};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Queries [T][H_q][128] bf16 as a 4-D tensor (64 dims of a half row, half, query head, token) with
// boxes of one half x G heads x tokens_per_box tokens: a box lands as tokens_per_box * G rows of
// 128 bytes, row (token, head), with the 128-byte swizzle.  `tokens` is the extent of the token
// dimension; boxes must stay inside the rows the caller allocated.
bool encode_query_map(CUtensorMap* map, const void* base, int heads, int G, int tokens_per_box, long long tokens) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[4] = {64, 2, static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(tokens)};
  cuuint64_t strides[3] = {128, 256, static_cast<cuuint64_t>(heads) * 256};
  cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(tokens_per_box)};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace pa

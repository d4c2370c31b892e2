// Append: write each new token's K and V rows into its paged slot.
//
// untitled KV-cache article at ldpk.cn/news/58971 §2.3: every generated token's K and V are
// written at the sequence's current length.  "KV Cache 的显存账本：PagedAttention 与连续批处理"
// §四: the slot is table[pos / 16] * 16 + pos % 16 (the locate() sketch).  Same page §七:
// 8-bit caches hold K as FP8 and V as INT8 with one scale per KV head, and sink tokens keep
// their original precision.  Untitled KV-cache article at ldpk.cn/news/58971 §5.2: 4-bit caches
// keep a scale and a zero point besides the codes; here one of each per 32 dims of a token's
// head row (the PA_INT4 rule in pa.h).  Same section: K's outlier channels call for finer scales
// than one per head; PA_FP8_E4M3_TOKEN K rows carry their own scale, max|x| / 448.
//
// bf16 and 8-bit caches: one warp per appended row, 8 rows per CTA; a lane moves 16-byte bf16
// vectors.  The row's K and V are loaded before the table lookup that places them (they do
// not depend on it), so the two memory round trips overlap.  The row's kv_heads x head_dim
// elements are contiguous in the slot-major cache, so the stores are fully coalesced.  INT4
// caches: one CTA per row, one thread per 32-dim group.

#include <cuda_fp8.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

struct AppendParams {
  int num_rows, num_seqs, H_kv, D, num_blocks, max_blocks, num_sink;
  const int32_t* token_seq;  // NULL: row r belongs to sequence r
  const int32_t* positions;
  const int32_t* block_tables;
  const uint4* k_new;
  const uint4* v_new;
  void* k_cache;
  void* v_cache;
  const float* k_scales;
  const float* v_scales;
  uint4* k_sink;
  uint4* v_sink;
  size_t params_offset;  // int4: byte offset of the group parameters in each pool; per-token K: of
                         // the K scales
  int32_t* err;
};

__device__ __forceinline__ void unpack_bf16x8(const uint4& v, float (&x)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// x / scale in IEEE fp32, then FP8 E4M3 round-to-nearest-even with saturation.
__device__ __forceinline__ uint2 encode_e4m3x8(const uint4& v, float scale) {
  float x[8];
  unpack_bf16x8(v, x);
  uint32_t out[2] = {0, 0};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 e = make_float2(__fdiv_rn(x[2 * i], scale), __fdiv_rn(x[2 * i + 1], scale));
    const uint32_t two = __nv_cvt_float2_to_fp8x2(e, __NV_SATFINITE, __NV_E4M3);
    out[i / 2] |= (two & 0xFFFFu) << (16 * (i % 2));
  }
  return make_uint2(out[0], out[1]);
}

// x / scale in IEEE fp32, round half to even, clamp to [-127, 127].
__device__ __forceinline__ uint2 encode_int8x8(const uint4& v, float scale) {
  float x[8];
  unpack_bf16x8(v, x);
  uint32_t out[2] = {0, 0};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    int q = __float2int_rn(__fdiv_rn(x[i], scale));
    q = max(-127, min(127, q));
    out[i / 4] |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * (i % 4));
  }
  return make_uint2(out[0], out[1]);
}

// One thread per (tensor, kv head, 32-dim group) of the row: range, bf16 scale, zero point and
// codes in IEEE fp32, then the codes in the K or V byte order of PA_INT4 and the group's
// parameter word after the code bytes of every slot.
__device__ __forceinline__ void encode_int4_group(const uint4* src, int h, int g, int tensor, int H_kv,
                                                  size_t slot, uint8_t* cache, size_t params_offset) {
  float x[32];
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    float t[8];
    unpack_bf16x8(src[v], t);
#pragma unroll
    for (int e = 0; e < 8; ++e) x[8 * v + e] = t[e];
  }
  float lo = 0.f, hi = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    lo = fminf(lo, x[i]);
    hi = fmaxf(hi, x[i]);
  }
  const float s = __fdiv_rn(__fsub_rn(hi, lo), 15.f);
  uint32_t sb = __bfloat16_as_ushort(__float2bfloat16_rn(s));
  if ((sb & 0x7FFFu) == 0) sb = 0x3F80u;  // an all-zero group
  const float sf = __uint_as_float(sb << 16);
  const float z = fminf(fmaxf(rintf(__fdiv_rn(-lo, sf)), 0.f), 15.f);
  uint32_t q[32];
#pragma unroll
  for (int i = 0; i < 32; ++i)
    q[i] = static_cast<uint32_t>(fminf(fmaxf(rintf(__fdiv_rn(x[i], sf)) + z, 0.f), 15.f));
  uint8_t* row = cache + (slot * H_kv + h) * 64;
  if (tensor == 0) {  // K: word 4c + g holds dims 32g + 8c + i at bits 4i
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t w = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) w |= q[8 * c + i] << (4 * i);
      reinterpret_cast<uint32_t*>(row)[4 * c + g] = w;
    }
  } else {  // V: byte 8r + m holds dim 16m + r (low) and 16m + r + 8 (high); m = 2g, 2g + 1
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const uint32_t b0 = q[r] | (q[r + 8] << 4), b1 = q[16 + r] | (q[24 + r] << 4);
      reinterpret_cast<uint16_t*>(row + 8 * r + 2 * g)[0] = static_cast<uint16_t>(b0 | (b1 << 8));
    }
  }
  reinterpret_cast<uint32_t*>(cache + params_offset)[(slot * H_kv + h) * 4 + g] =
      sb | (static_cast<uint32_t>(z) << 16);
}

template <int KIND>  // 0 bf16, 1 fp8 K / int8 V, 2 fp8 K with per-token scales / int8 V
__global__ void __launch_bounds__(256) kv_append_rows_kernel(const AppendParams p) {
  // the decode kernel that usually follows may start its prologue now: it waits for this
  // kernel's completion before it reads the cache
  grid_dep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= p.num_rows) return;
  const int vecs = p.H_kv * p.D / 8;  // 16-byte bf16 vectors per row
  const uint4* kin = p.k_new + static_cast<size_t>(r) * vecs;
  const uint4* vin = p.v_new + static_cast<size_t>(r) * vecs;
  const int s = p.token_seq ? p.token_seq[r] : r;
  const int pos = p.positions[r];
  constexpr int kAhead = 4;  // vectors per lane loaded ahead of the lookup (a whole row up to 1024 dims)
  uint4 kv[kAhead], vv[kAhead];
#pragma unroll
  for (int j = 0; j < kAhead; ++j) {
    const int i = lane + 32 * j;
    if (i < vecs) {
      kv[j] = kin[i];
      vv[j] = vin[i];
    }
  }
  if (s < 0 || s >= p.num_seqs) {
    if (lane == 0) set_error(p.err, PA_EFLAG_BAD_SEQ);
    return;
  }
  if (pos < 0) return;  // padding row
  if (pos < p.num_sink) {  // sink rows keep bf16 in their own buffer
    const size_t base = (static_cast<size_t>(s) * p.num_sink + pos) * vecs;
#pragma unroll
    for (int j = 0; j < kAhead; ++j) {
      const int i = lane + 32 * j;
      if (i < vecs) {
        p.k_sink[base + i] = kv[j];
        p.v_sink[base + i] = vv[j];
      }
    }
    for (int i = lane + 32 * kAhead; i < vecs; i += 32) {
      p.k_sink[base + i] = kin[i];
      p.v_sink[base + i] = vin[i];
    }
    return;
  }
  const int lb = pos / PA_BLOCK_SIZE;
  if (lb >= p.max_blocks) {
    if (lane == 0) set_error(p.err, PA_EFLAG_CTX_OVERFLOW);
    return;
  }
  const int pb = p.block_tables[static_cast<size_t>(s) * p.max_blocks + lb];
  if (pb < 0 || pb >= p.num_blocks) {
    if (lane == 0) set_error(p.err, PA_EFLAG_BAD_BLOCK_ID);
    return;
  }
  const size_t slot = static_cast<size_t>(pb) * PA_BLOCK_SIZE + pos % PA_BLOCK_SIZE;
  // Every lane of the warp calls put for the same number of vectors (vecs is a multiple of 32 on
  // the per-token path), so the half-warp reductions below see all their lanes.
  auto put = [&](int i, const uint4& k4, const uint4& v4) {
    if constexpr (KIND == 2) {
      // head_dim 128: a head row is 16 vectors, held by one half-warp
      const int h = i >> 4;
      float x[8];
      unpack_bf16x8(k4, x);
      float a = 0.f;  // fmaxf leaves NaN out of the maximum
#pragma unroll
      for (int e = 0; e < 8; ++e) a = fmaxf(a, fabsf(x[e]));
#pragma unroll
      for (int m = 1; m < 16; m <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, m));
      float sc = __fdiv_rn(a, 448.f);
      if (sc == 0.f) sc = 1.f;  // an all-zero row: any scale encodes it exactly
      reinterpret_cast<uint2*>(p.k_cache)[slot * vecs + i] = encode_e4m3x8(k4, sc);
      reinterpret_cast<uint2*>(p.v_cache)[slot * vecs + i] = encode_int8x8(v4, p.v_scales[h]);
      if ((i & 15) == 0)
        reinterpret_cast<float*>(static_cast<uint8_t*>(p.k_cache) + p.params_offset)[slot * p.H_kv + h] = sc;
    } else if constexpr (KIND == 1) {
      const int h = (i * 8) / p.D;
      reinterpret_cast<uint2*>(p.k_cache)[slot * vecs + i] = encode_e4m3x8(k4, p.k_scales[h]);
      reinterpret_cast<uint2*>(p.v_cache)[slot * vecs + i] = encode_int8x8(v4, p.v_scales[h]);
    } else {
      reinterpret_cast<uint4*>(p.k_cache)[slot * vecs + i] = k4;
      reinterpret_cast<uint4*>(p.v_cache)[slot * vecs + i] = v4;
    }
  };
#pragma unroll
  for (int j = 0; j < kAhead; ++j) {
    const int i = lane + 32 * j;
    if (i < vecs) put(i, kv[j], vv[j]);
  }
  for (int i = lane + 32 * kAhead; i < vecs; i += 32) put(i, kin[i], vin[i]);
}

__global__ void __launch_bounds__(256) kv_append_int4_kernel(const AppendParams p) {
  grid_dep_launch_dependents();
  const int r = blockIdx.x;
  const int s = p.token_seq ? p.token_seq[r] : r;
  if (s < 0 || s >= p.num_seqs) {
    if (threadIdx.x == 0) set_error(p.err, PA_EFLAG_BAD_SEQ);
    return;
  }
  const int pos = p.positions[r];
  if (pos < 0) return;  // padding row
  const int vecs = p.H_kv * p.D / 8;  // 16-byte bf16 vectors per row
  const uint4* kin = p.k_new + static_cast<size_t>(r) * vecs;
  const uint4* vin = p.v_new + static_cast<size_t>(r) * vecs;
  if (pos < p.num_sink) {  // sink rows keep bf16 in their own buffer
    const size_t base = (static_cast<size_t>(s) * p.num_sink + pos) * vecs;
    for (int i = threadIdx.x; i < vecs; i += blockDim.x) {
      p.k_sink[base + i] = kin[i];
      p.v_sink[base + i] = vin[i];
    }
    return;
  }
  const int lb = pos / PA_BLOCK_SIZE;
  if (lb >= p.max_blocks) {
    if (threadIdx.x == 0) set_error(p.err, PA_EFLAG_CTX_OVERFLOW);
    return;
  }
  const int pb = p.block_tables[static_cast<size_t>(s) * p.max_blocks + lb];
  if (pb < 0 || pb >= p.num_blocks) {
    if (threadIdx.x == 0) set_error(p.err, PA_EFLAG_BAD_BLOCK_ID);
    return;
  }
  const size_t slot = static_cast<size_t>(pb) * PA_BLOCK_SIZE + pos % PA_BLOCK_SIZE;
  const int groups = p.H_kv * 4;  // head_dim 128
  for (int i = threadIdx.x; i < 2 * groups; i += blockDim.x) {
    const int tensor = i / groups, h = (i % groups) / 4, g = i % 4;
    encode_int4_group((tensor ? vin : kin) + h * 16 + g * 4, h, g, tensor, p.H_kv, slot,
                      static_cast<uint8_t*>(tensor ? p.v_cache : p.k_cache), p.params_offset);
  }
}

pa_status append_impl(const pa_cache_desc* d, void* k_cache, void* v_cache, const void* k_new,
                      const void* v_new, int num_rows, const int32_t* token_seq,
                      const int32_t* positions, const int32_t* block_tables, int32_t* err,
                      void* stream) {
  pa_status st = validate_desc(d);
  if (st != PA_OK) return st;
  if (num_rows < 0) return PA_ERR_INVALID_ARG;
  if (num_rows == 0) return PA_OK;
  if (!k_cache || !v_cache || !k_new || !v_new || !positions || !block_tables)
    return PA_ERR_INVALID_ARG;
  const auto aligned16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; };
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (d->num_sink > 0 && (!aligned16(d->k_sink) || !aligned16(d->v_sink))))
    return PA_ERR_INVALID_ARG;
  AppendParams p;
  p.num_rows = num_rows;
  p.num_seqs = d->num_seqs;
  p.H_kv = d->num_kv_heads;
  p.D = d->head_dim;
  p.num_blocks = d->num_blocks;
  p.max_blocks = d->max_blocks_per_seq;
  p.num_sink = d->num_sink;
  p.token_seq = token_seq;
  p.positions = positions;
  p.block_tables = block_tables;
  p.k_new = static_cast<const uint4*>(k_new);
  p.v_new = static_cast<const uint4*>(v_new);
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.k_scales = d->k_scales;
  p.v_scales = d->v_scales;
  p.k_sink = static_cast<uint4*>(d->k_sink);
  p.v_sink = static_cast<uint4*>(d->v_sink);
  p.err = err;
  p.params_offset = is_int4(d) ? int4_params_offset(d) : (has_token_scales(d) ? token_scales_offset(d) : 0);
  const int vecs = p.H_kv * p.D / 8;
  constexpr int kRowsPerCta = 8;
  const int grid = (num_rows + kRowsPerCta - 1) / kRowsPerCta;
  if (is_int4(d))
    kv_append_int4_kernel<<<num_rows, min(256, ((vecs + 31) / 32) * 32), 0, as_stream(stream)>>>(p);
  else if (has_token_scales(d))
    kv_append_rows_kernel<2><<<grid, 32 * kRowsPerCta, 0, as_stream(stream)>>>(p);
  else if (is_quantized(d))
    kv_append_rows_kernel<1><<<grid, 32 * kRowsPerCta, 0, as_stream(stream)>>>(p);
  else
    kv_append_rows_kernel<0><<<grid, 32 * kRowsPerCta, 0, as_stream(stream)>>>(p);
  return launch_status();
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_kv_append(const pa_cache_desc* desc, void* k_cache, void* v_cache,
                                  const void* k_new, const void* v_new,
                                  const int32_t* block_tables, const int32_t* positions,
                                  int32_t* err_flag, void* stream) {
  if (!desc) return PA_ERR_INVALID_ARG;
  return pa::append_impl(desc, k_cache, v_cache, k_new, v_new, desc->num_seqs, nullptr, positions,
                         block_tables, err_flag, stream);
}

extern "C" pa_status pa_kv_append_tokens(const pa_cache_desc* desc, void* k_cache, void* v_cache,
                                         const void* k_new, const void* v_new, int num_tokens,
                                         const int32_t* token_seq, const int32_t* token_pos,
                                         const int32_t* block_tables, int32_t* err_flag,
                                         void* stream) {
  if (!desc || !token_seq) return PA_ERR_INVALID_ARG;
  return pa::append_impl(desc, k_cache, v_cache, k_new, v_new, num_tokens, token_seq, token_pos,
                         block_tables, err_flag, stream);
}

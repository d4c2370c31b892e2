// Decode attention of many sequences over one shared prompt prefix, attended once for all of them.
//
// Prefix sharing (AI内存系统 §3.1: requests with the same prefix point their block tables at one
// stored copy of its blocks; §3.3: only whole blocks are shared) makes every member sequence's
// decode read the same prefix blocks.  Attention is a sum over positions, so it splits exactly at
// a block boundary: with the softmax kept as (running max m, sum l, unnormalised output o) per
// part, two parts combine as
//   M = max(m1, m2),  l = e^{m1-M} l1 + e^{m2-M} l2,  o = e^{m1-M} o1 + e^{m2-M} o2,  out = o / l
// (the same rule that merges the split-context partials of the decode kernel).  Here the prefix
// part is computed once per (KV head, 128-key chunk) for all member rows together — every member's
// G query heads stacked as the rows of one warp-level matrix product, so each prefix K/V tile
// crosses HBM once instead of once per member — and the decode kernel then visits only each
// member's own positions past the prefix, its merge folding the prefix rows in.
//
// Membership is checked, not trusted: a listed sequence uses the prefix rows only if its context
// covers the prefix and its table maps every prefix block to the first listed sequence's physical
// block.  Any other sequence (listed or not) is attended in full by the decode kernel, so results
// never depend on the list being right.
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kRowsPerCta = 64;  // (member, query head) rows: 4 warps x 16
constexpr int kThreads = 128;
constexpr int kChunkKeys = kSharedChunkBlocks * PA_BLOCK_SIZE;

struct PrefixParams {
  const __nv_bfloat16* q;  // [B][H_q][D]
  const __nv_bfloat16* k;  // pool [slots][H_kv][D]
  const __nv_bfloat16* v;
  const int32_t* block_tables;  // [B][max_blocks]
  const int32_t* context_lens;  // [B]
  const int32_t* shared_seqs;   // [n_shared]; the first is the one whose table is read
  int32_t* flags;               // [B], zeroed before this kernel: kSharedMember | kSharedMismatch
  float* extra;                 // [B][n_chunks][H_q][D + 4]
  int32_t* err;
  int B, H_q, H_kv, G, num_blocks, max_blocks, max_ctx;
  int n_shared, shared_len, n_chunks;
  float scale_log2;
};

constexpr int kGroupBlocks = 2;  // blocks per copy group (one barrier each for K and for V)
constexpr int kGroups = kSharedChunkBlocks / kGroupBlocks;

__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Byte offset of (token t of a block, dim d) in a block's tile as its TMA boxes land it: one
// [16 slots][128 bytes] box per 64 dims, under the 128-byte swizzle (the 16-byte unit index XOR
// the slot mod 8), so that the eight rows of an ldmatrix fall in eight distinct bank groups.
__device__ __forceinline__ uint32_t tile_off(int t, int d) {
  return static_cast<uint32_t>((d >> 6) * (PA_BLOCK_SIZE * 128) + t * 128 + ((((d & 63) >> 3) ^ (t & 7)) << 4));
}

// grid (n_chunks, H_kv, ceil(n_shared * G / 64)), 128 threads.  CTA (x, y, z): KV head y, prefix
// blocks [kSharedChunkBlocks x, +kSharedChunkBlocks), member rows [64 z, 64 z + 64) in
// member-major order (row r: member r / G, query head y G + r % G); warp w takes the 16 rows
// 64 z + 16 w .. +15 over all of the chunk's keys.
template <int D>
__global__ void __launch_bounds__(kThreads, 3)
    shared_prefix_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                         const PrefixParams p) {
  constexpr int TB = PA_BLOCK_SIZE * D * 2;  // bytes of one block's tile (one KV head)
  constexpr int KK = D / 16;                  // k-steps of the score product
  constexpr int NT = kChunkKeys / 8;          // 8-key tiles of a chunk
  extern __shared__ uint8_t smem_raw[];
  // tiles 1024-byte aligned (the swizzle pattern's period): K tiles, then V tiles
  uint8_t* ks = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* vs = ks + kSharedChunkBlocks * TB;
  __shared__ int blk[kSharedChunkBlocks];
  __shared__ int any_bad;
  __shared__ __align__(8) uint64_t bars[2 * kGroups];  // K groups, then V groups: one phase each

  // the decode kernel that follows may be scheduled as this grid's CTAs finish; it waits for the
  // whole grid (and its memory) before reading anything this kernel writes
  grid_dep_launch_dependents();

  const int x = blockIdx.x, y = blockIdx.y, z = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int rows_total = p.n_shared * p.G;
  const int r0 = z * kRowsPerCta;
  const int wr0 = r0 + warp * 16;
  // Every load below depends on at most two others, and the chains run side by side: the list
  // entries of this thread's two rows and the first listed sequence go out together.
  const int leader = p.shared_seqs[0];
  int srow[2] = {-1, -1}, hrow[2] = {0, 0};
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    const int r = wr0 + g + 8 * hf;
    if (r < rows_total) {
      srow[hf] = p.shared_seqs[r / p.G];
      hrow[hf] = y * p.G + r % p.G;
    }
  }
  if (leader < 0 || leader >= p.B) {
    if (x == 0 && y == 0 && z == 0 && tid == 0) set_error(p.err, PA_EFLAG_BAD_SEQ);
    return;
  }
  const int b0 = x * kSharedChunkBlocks;
  const int nblk = min(kSharedChunkBlocks, p.shared_len / PA_BLOCK_SIZE - b0);
  const int32_t* ltab = p.block_tables + static_cast<size_t>(leader) * p.max_blocks;
  // The leader's table is read before its context length is known: every id is range-checked
  // before use, and when the context does not cover the prefix no sequence takes these rows.
  if (tid == 0) {
    any_bad = 0;
#pragma unroll
    for (int i = 0; i < 2 * kGroups; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  const int nrows = nblk * PA_BLOCK_SIZE;
  // V tiles past the prefix's end (its last chunk) hold zeros: their weights are exactly 0, and
  // 0 times stale bits could be NaN.  (K rows there are masked in the softmax instead.)
  for (int i = nblk * TB / 16 + tid; i < kSharedChunkBlocks * TB / 16; i += kThreads)
    reinterpret_cast<uint4*>(vs)[i] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  if (tid < nblk) {
    const int b = ltab[b0 + tid];
    const bool ok = b >= 0 && b < p.num_blocks;
    blk[tid] = ok ? b : -1;
    if (!ok) any_bad = 1;
  }
  __syncthreads();

  // ---- K then V of this chunk into shared memory: TMA boxes of a block's 16 slots of KV head y
  // (one per 64 dims), in groups of two blocks with a barrier each, so that the products start
  // on the first keys while the rest are in flight.  A block with an invalid id is not
  // loaded (its rows' results are discarded). ----
  if (tid == 0) {
    const uint64_t pol = l2_evict_last_policy();  // each chunk is read by every row-tile CTA
#pragma unroll 1
    for (int gi = 0; gi < 2 * kGroups; ++gi) {
      const int kv = gi / kGroups;
      int n = 0;
      for (int bi = (gi % kGroups) * kGroupBlocks; bi < (gi % kGroups + 1) * kGroupBlocks; ++bi)
        n += bi < nblk && blk[bi] >= 0;
      mbar_arrive_expect_tx(&bars[gi], n * TB);
      for (int bi = (gi % kGroups) * kGroupBlocks; bi < (gi % kGroups + 1) * kGroupBlocks; ++bi)
        if (bi < nblk && blk[bi] >= 0)
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_4d((kv == 0 ? ks : vs) + bi * TB + c * (PA_BLOCK_SIZE * 128), kv == 0 ? &tmK : &tmV, &bars[gi],
                        0, c, blk[bi] * PA_BLOCK_SIZE, y, pol);
    }
  }
  const uint32_t ks_a = smem_u32(ks), vs_a = smem_u32(vs);

  // ---- this warp's 16 rows: query fragments straight from global memory ----
#pragma unroll
  for (int hf = 0; hf < 2; ++hf)
    if (srow[hf] >= p.B) srow[hf] = -1;  // out-of-range entries (negative ones are -1 or below)
  uint32_t qa[KK][4];
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    const uint32_t* qr = srow[hf] >= 0
        ? reinterpret_cast<const uint32_t*>(p.q + (static_cast<size_t>(srow[hf]) * p.H_q + hrow[hf]) * D)
        : nullptr;
#pragma unroll
    for (int kk = 0; kk < KK; ++kk) {
      qa[kk][hf] = qr ? qr[kk * 8 + t] : 0u;          // dims 16kk + 2t, +1
      qa[kk][2 + hf] = qr ? qr[kk * 8 + 4 + t] : 0u;  // dims 16kk + 8 + 2t, +1
    }
  }

  // ---- membership checks (the CTAs of KV head 0), while the tiles are in flight: the member
  // bit once per sequence, table agreement per chunk ----
  if (y == 0) {
    const int lctx = p.context_lens[leader];
    const bool leader_ok = lctx >= p.shared_len && lctx <= p.max_ctx;
    if (z == 0 && tid == 0 && any_bad && leader_ok) set_error(p.err, PA_EFLAG_BAD_BLOCK_ID);
    const int j_lo = r0 / p.G, j_hi = min(p.n_shared, (min(r0 + kRowsPerCta, rows_total) + p.G - 1) / p.G);
    const int nj = j_hi - j_lo;
    for (int i = tid; i < nj * nblk; i += kThreads) {
      const int j = j_lo + i / nblk, bi = i % nblk;
      const int s = p.shared_seqs[j];
      if (s < 0 || s >= p.B) {
        if (x == 0 && bi == 0) set_error(p.err, PA_EFLAG_BAD_SEQ);
        continue;
      }
      if (x == 0 && bi == 0 && leader_ok) {
        const int c = p.context_lens[s];
        if (c >= p.shared_len && c <= p.max_ctx) atomicOr(p.flags + s, kSharedMember);
      }
      if (p.block_tables[static_cast<size_t>(s) * p.max_blocks + b0 + bi] != ltab[b0 + bi])
        atomicOr(p.flags + s, kSharedMismatch);
    }
  }

  // ---- S = Q K^T over the chunk, one copy group at a time (every warp waits for every group,
  // so that none leaves while a copy into this CTA may be in flight) ----
  const bool active = wr0 < rows_total;
  bool late = false;
  float sacc[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
  const int li = lane >> 3, lr = lane & 7;
#pragma unroll
  for (int gi = 0; gi < kGroups; ++gi) {
    late |= !mbar_wait(&bars[gi], 0);
    if (active) {
#pragma unroll
      for (int kk = 0; kk < KK; ++kk) {
#pragma unroll
        for (int np = gi * kGroupBlocks; np < (gi + 1) * kGroupBlocks; ++np) {
          // block np; matrices: (keys 0..7, dims 16kk), (keys 0..7, dims +8), (keys 8..15, dims 16kk),
          // (keys 8..15, dims +8)
          const uint32_t a = ks_a + np * TB + tile_off(lr + 8 * (li >> 1), kk * 16 + 8 * (li & 1));
          uint32_t b00, b01, b10, b11;
          ldsm_x4(a, b00, b01, b10, b11);
          mma_bf16(sacc[2 * np], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b00, b01);
          mma_bf16(sacc[2 * np + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b10, b11);
        }
      }
    }
  }

  // ---- softmax of the chunk in log2 units: m = row max, p = 2^(s - m), l = sum p ----
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) sacc[n][e] *= p.scale_log2;
  if (nrows < kChunkKeys) {  // the prefix's last chunk: keys n*8 + 2t + (e & 1) past its end
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (n * 8 + 2 * t + (e & 1) >= nrows) sacc[n][e] = -INFINITY;
  }
  float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    mx[0] = fmaxf(mx[0], fmaxf(sacc[n][0], sacc[n][1]));
    mx[1] = fmaxf(mx[1], fmaxf(sacc[n][2], sacc[n][3]));
  }
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    mx[hf] = warp_max_xor(mx[hf], 1);
    mx[hf] = warp_max_xor(mx[hf], 2);
  }
  // (every chunk holds at least one block of the prefix, so m is finite)
  float ls[2] = {0.f, 0.f};
#pragma unroll
  for (int n = 0; n < NT; ++n) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      sacc[n][e] = ex2(sacc[n][e] - mx[e >> 1]);
      ls[e >> 1] += sacc[n][e];
    }
  }
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    ls[hf] += __shfl_xor_sync(0xffffffffu, ls[hf], 1);
    ls[hf] += __shfl_xor_sync(0xffffffffu, ls[hf], 2);
  }

  // ---- O = P V, one copy group at a time ----
  float oacc[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) oacc[n][0] = oacc[n][1] = oacc[n][2] = oacc[n][3] = 0.f;
#pragma unroll
  for (int kt = 0; kt < NT / 2; ++kt) {  // block kt
    if (kt % kGroupBlocks == 0) late |= !mbar_wait(&bars[kGroups + kt / kGroupBlocks], 0);
    if (active) {
      const uint32_t a0 = pack_bf16(sacc[2 * kt][0], sacc[2 * kt][1]);
      const uint32_t a1 = pack_bf16(sacc[2 * kt][2], sacc[2 * kt][3]);
      const uint32_t a2 = pack_bf16(sacc[2 * kt + 1][0], sacc[2 * kt + 1][1]);
      const uint32_t a3 = pack_bf16(sacc[2 * kt + 1][2], sacc[2 * kt + 1][3]);
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        // transposed matrices: (keys 0..7, dims 16dp), (keys 8..15, dims 16dp), (keys 0..7, dims +8),
        // (keys 8..15, dims +8)
        const uint32_t a = vs_a + kt * TB + tile_off(lr + 8 * (li & 1), dp * 16 + 8 * (li >> 1));
        uint32_t b00, b01, b10, b11;
        ldsm_x4_t(a, b00, b01, b10, b11);
        mma_bf16(oacc[2 * dp], a0, a1, a2, a3, b00, b01);
        mma_bf16(oacc[2 * dp + 1], a0, a1, a2, a3, b10, b11);
      }
    }
  }

  // ---- the partial rows: o (unnormalised), m, l (-1 when a prefix block id was invalid or a copy
  // did not land in time) ----
  late = __any_sync(0xffffffffu, late);
  if (late && lane == 0) set_error(p.err, PA_EFLAG_TIMEOUT);
  const bool bad = any_bad != 0 || late;
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    if (srow[hf] < 0) continue;
    float* row = p.extra + ((static_cast<size_t>(srow[hf]) * p.n_chunks + x) * p.H_q + hrow[hf]) * (D + 4);
    if (!bad) {
#pragma unroll
      for (int n = 0; n < D / 8; ++n)
        *reinterpret_cast<float2*>(row + n * 8 + 2 * t) = make_float2(oacc[n][2 * hf], oacc[n][2 * hf + 1]);
    }
    if (t == 0) {
      row[D] = mx[hf];
      row[D + 1] = bad ? -1.f : ls[hf];
    }
  }
}

}  // namespace

size_t shared_prefix_smem_bytes(int head_dim) {
  // K and V tiles of a chunk, plus the slack for their 1024-byte alignment
  return static_cast<size_t>(2) * kSharedChunkBlocks * PA_BLOCK_SIZE * head_dim * 2 + 1024;
}

pa_status launch_shared_prefix(const pa_cache_desc* desc, const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, const int32_t* context_lens, int max_context_len,
                               float scale, const int32_t* shared_seqs, int n_shared, int shared_len,
                               int32_t* flags, float* extra, int32_t* err_flag, cudaStream_t stream) {
  PrefixParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k_cache);
  p.v = static_cast<const __nv_bfloat16*>(v_cache);
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.shared_seqs = shared_seqs;
  p.flags = flags;
  p.extra = extra;
  p.err = err_flag;
  p.B = desc->num_seqs;
  p.H_q = desc->num_q_heads;
  p.H_kv = desc->num_kv_heads;
  p.G = desc->num_q_heads / desc->num_kv_heads;
  p.num_blocks = desc->num_blocks;
  p.max_blocks = desc->max_blocks_per_seq;
  p.max_ctx = max_context_len;
  p.n_shared = n_shared;
  p.shared_len = shared_len;
  p.n_chunks = shared_prefix_chunks(shared_len);
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  const long long rows = static_cast<long long>(n_shared) * p.G;
  const dim3 grid(p.n_chunks, p.H_kv, static_cast<unsigned>((rows + kRowsPerCta - 1) / kRowsPerCta));
  const size_t smem = shared_prefix_smem_bytes(desc->head_dim);
  // the pools as (64 dims, 64-dim chunk, slot, KV head), boxes of one chunk of one block's 16 slots
  const long long slots = static_cast<long long>(desc->num_blocks) * PA_BLOCK_SIZE;
  const int nc = desc->head_dim * 2 / 128;
  CUtensorMap mk, mv;
  if (!encode_cache_map_chunk(&mk, k_cache, 2, desc->num_kv_heads, nc, slots) ||
      !encode_cache_map_chunk(&mv, v_cache, 2, desc->num_kv_heads, nc, slots))
    return PA_ERR_CUDA;
  if (cudaMemsetAsync(flags, 0, static_cast<size_t>(p.B) * sizeof(int32_t), stream) != cudaSuccess)
    return PA_ERR_CUDA;
  auto kern = desc->head_dim == 128 ? shared_prefix_kernel<128> : shared_prefix_kernel<64>;
  if (!ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem)) return PA_ERR_CUDA;
  kern<<<grid, kThreads, smem, stream>>>(mk, mv, p);
  return launch_status();
}

}  // namespace pa

// Chunked-prefill (extend) attention over the paged KV cache.
//
// untitled KV-cache article at ldpk.cn/news/58971 §2.2: in prefill every position's query
// attends to the keys of the positions up to itself under the causal mask, and only K and V are
// kept for later steps; §7 splits a long prompt into chunks to cap the activation peak.  Here a
// chunk of n new tokens per sequence (their K/V already appended to the cache) attends over the
// whole cached context through the block table ("KV Cache 的显存账本：PagedAttention 与连续批处理"
// §四), with GQA grouping (same page §二).  Under a sliding window of W tokens (ldpk §5.3) the
// query at position p reads keys p-W+1 .. p only, and blocks before a tile's window are not read.
//
// Design: one CTA per (sequence, KV head, tile of query tokens).  Four consumer warps own 16
// (query token, query head) rows each, so every K/V element a warp loads serves up to 16 query
// rows; S = Q·Kᵀ and O += P·V are m16n8k16 tensor-core products with the queries as M, and P is
// reused straight from the S accumulator registers as the A operand of P·V.  A producer warp
// streams the KV head's blocks with TMA (one 16-slot x 128-byte box per chunk of the head row,
// 128-byte swizzle, conflict-free ldmatrix) into an mbarrier ring.  Keys beyond a row's own
// position are masked; whole blocks beyond a warp's last position are skipped.

#include <algorithm>
#include <cmath>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kPfWarps = 4;            // consumer warps per CTA
constexpr int kPfThreads = (kPfWarps + 1) * 32;
constexpr int kPfStages = 4;
constexpr int kChunkTile = 2048;      // one box: 16 slots x 128 bytes
constexpr float kNegInfP = -INFINITY;

struct PrefillParams {
  int B, H_q, H_kv, G, num_blocks, max_blocks, max_q;
  int window;  // sliding window in tokens, 0 = whole context
  int tpw;     // query tokens per warp (16 / G)
  int q_tile;  // query tokens per CTA
  int nc;      // 128-byte chunks per head row
  float scale_log2;
  const int32_t* q_start;
  const int32_t* context_lens;
  const int32_t* block_tables;
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  int32_t* err;
};

template <int D>
__global__ void __launch_bounds__(kPfThreads)
    prefill_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const PrefillParams p) {
  constexpr int NC = D * 2 / 128;       // chunks per head row (bf16)
  constexpr int KT = D / 16;            // k-steps of Q·Kᵀ
  constexpr int NT = D / 8;             // n-tiles of P·V
  constexpr int STAGE = 2 * NC * kChunkTile;
  __shared__ __align__(1024) uint8_t stages[kPfStages][STAGE];
  __shared__ uint64_t full[kPfStages], empty[kPfStages];
  __shared__ int bad_stage[kPfStages];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int s = blockIdx.y, h_kv = blockIdx.z, tile = blockIdx.x;
  // launched with programmatic dependent launch: the previous kernel of the stream may still be
  // writing any input (q, lengths, tables, cache), so everything below waits for it
  grid_dep_wait();
  const int qs = p.q_start[s];
  const int n = p.q_start[s + 1] - qs;
  const int ctx = p.context_lens[s];
  const bool valid = n >= 0 && n <= ctx && n <= p.max_q && ctx <= p.max_blocks * PA_BLOCK_SIZE;
  if (!valid) {
    if (tile == 0 && h_kv == 0 && tid == 0) set_error(p.err, PA_EFLAG_CTX_OVERFLOW);
    // zero the rows this CTA would have produced (those inside the query range it can see)
    const int rows = min(max(n, 0), p.max_q);
    for (int t = tile * p.q_tile + warp; t < min(rows, (tile + 1) * p.q_tile); t += kPfWarps + 1)
      for (int i = lane; i < p.G * D; i += 32)
        p.out[(static_cast<size_t>(qs + t) * p.H_q + h_kv * p.G) * D + i] = __float2bfloat16_rn(0.f);
    return;
  }
  const int t0 = tile * p.q_tile;
  if (t0 >= n) return;
  const int first_pos = ctx - n;
  const int t_end = min(n, t0 + p.q_tile);
  const int kv_end = first_pos + t_end;  // keys [kv_lo, kv_end) are visible to this tile
  const int kv_lo = p.window > 0 ? max(0, first_pos + t0 - p.window + 1) : 0;
  const int kb0 = kv_lo / PA_BLOCK_SIZE;  // first logical block read
  const int n_blocks = (kv_end + PA_BLOCK_SIZE - 1) / PA_BLOCK_SIZE - kb0;

  if (tid == 0) {
    for (int i = 0; i < kPfStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kPfWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kPfWarps) {
    // ------------------------------ producer ------------------------------
    const uint64_t policy = l2_evict_first_policy();
    const int32_t* row = p.block_tables + static_cast<size_t>(s) * p.max_blocks + kb0;
    int cur = lane < n_blocks ? row[lane] : -1;
    int nxt = 32 + lane < n_blocks ? row[32 + lane] : -1;
    int k = 0;
    for (; k < n_blocks; ++k) {
      if (k > 0 && (k & 31) == 0) {
        cur = nxt;
        nxt = k + 32 + lane < n_blocks ? row[k + 32 + lane] : -1;
      }
      const int pb = __shfl_sync(0xffffffffu, cur, k & 31);
      const bool bad = pb < 0 || pb >= p.num_blocks;
      const int st = k % kPfStages;
      const uint32_t ph = static_cast<uint32_t>(k / kPfStages) & 1u;
      if (!mbar_wait(&empty[st], ph ^ 1u)) {
        if (lane == 0) set_error(p.err, PA_EFLAG_TIMEOUT);
        break;
      }
      if (lane == 0) {
        bad_stage[st] = bad ? 1 : 0;
        if (bad) {
          set_error(p.err, PA_EFLAG_BAD_BLOCK_ID);
          mbar_arrive(&full[st]);
        } else {
          mbar_arrive_expect_tx(&full[st], STAGE);
        }
      }
      __syncwarp();
      if (!bad && lane < 2 * NC) {
        const int tensor = lane / NC, c = lane % NC;
        tma_load_3d(&stages[st][(tensor * NC + c) * kChunkTile], tensor ? &tmV : &tmK, &full[st], 0,
                    h_kv * NC + c, pb * PA_BLOCK_SIZE, policy);
      }
    }
    for (int st = 0; st < kPfStages && st < k; ++st) {
      const int last = st + kPfStages * ((k - 1 - st) / kPfStages);
      if (!mbar_wait(&full[st], static_cast<uint32_t>(last / kPfStages) & 1u) && lane == 0)
        set_error(p.err, PA_EFLAG_TIMEOUT);
    }
    return;
  }

  // ------------------------------ consumers ------------------------------
  const int t4 = lane >> 2, tq = lane & 3;
  const int wt0 = t0 + warp * p.tpw;                  // this warp's first query token (chunk index)
  const int w_tokens = max(0, min(p.tpw, t_end - wt0));
  const int w_last_pos = first_pos + wt0 + w_tokens - 1;  // last query position of this warp
  // lowest key any row of this warp reads (its first token's window start)
  const int w_lo = p.window > 0 ? max(0, first_pos + wt0 - p.window + 1) : 0;
  // rows of the 16-row tile: row r = (token r / G, head r % G); rows past the tokens are padding
  const int rows_used = w_tokens * p.G;
  int row_pos[2];
  bool row_ok[2];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = t4 + 8 * half;
    row_ok[half] = r < rows_used;
    row_pos[half] = row_ok[half] ? first_pos + wt0 + r / p.G : -1;
  }
  // Q fragments (A operand, rows x head_dim)
  uint32_t qa[KT][4];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = t4 + 8 * half;
    const __nv_bfloat16* qrow =
        p.q + (static_cast<size_t>(qs + wt0 + (row_ok[half] ? r / p.G : 0)) * p.H_q + h_kv * p.G +
               (row_ok[half] ? r % p.G : 0)) * D;
#pragma unroll
    for (int kk = 0; kk < KT; ++kk) {
      qa[kk][half] = row_ok[half] ? *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 2 * tq) : 0u;
      qa[kk][2 + half] = row_ok[half] ? *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 8 + 2 * tq) : 0u;
    }
  }
  float o[NT][4];
#pragma unroll
  for (int i = 0; i < NT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m[2] = {kNegInfP, kNegInfP}, l[2] = {0.f, 0.f};
  bool bad = false;

  for (int k = 0; k < n_blocks; ++k) {
    const int st = k % kPfStages;
    const uint32_t ph = static_cast<uint32_t>(k / kPfStages) & 1u;
    if (!mbar_wait(&full[st], ph)) {
      if (lane == 0) set_error(p.err, PA_EFLAG_TIMEOUT);
      return;
    }
    const int kbase_pos = (kb0 + k) * PA_BLOCK_SIZE;
    if (bad_stage[st]) {
      bad = true;
    } else if (w_tokens > 0 && kbase_pos <= w_last_pos && kbase_pos + PA_BLOCK_SIZE > w_lo) {
      const uint8_t* kt = stages[st];
      const uint8_t* vt = stages[st] + NC * kChunkTile;
      // S = Q Kᵀ for the 16 keys (two n-tiles of 8)
      float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      {
        const int key = (lane & 7) + ((lane >> 4) & 1) * 8;  // matrices: [k0-7,d0],[k0-7,d8],[k8-15,d0],[k8-15,d8]
        const int dhalf = (lane >> 3) & 1;
#pragma unroll
        for (int kk = 0; kk < KT; ++kk) {
          const int ch16 = (kk & 3) * 2 + dhalf;
          const uint32_t addr =
              smem_u32(kt + (kk >> 2) * kChunkTile + key * 128 + ((ch16 ^ (key & 7)) << 4));
          uint32_t b0, b1, b2, b3;
          ldsm_x4(addr, b0, b1, b2, b3);
          mma_bf16(sacc[0], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
          mma_bf16(sacc[1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
        }
      }
      // causal mask and online softmax (rows t4 and t4 + 8; keys nt*8 + 2tq + {0,1})
      float sv[2][2][2];  // [half][nt][j]
      float bm[2] = {kNegInfP, kNegInfP};
#pragma unroll
      for (int half = 0; half < 2; ++half)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const int kp = kbase_pos + nt * 8 + 2 * tq + jj;
            const bool ok = row_ok[half] && kp <= row_pos[half] && (p.window <= 0 || kp > row_pos[half] - p.window);
            const float v = ok ? sacc[nt][2 * half + jj] * p.scale_log2 : kNegInfP;
            sv[half][nt][jj] = v;
            bm[half] = fmaxf(bm[half], v);
          }
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        bm[half] = warp_max_xor(bm[half], 1);
        bm[half] = warp_max_xor(bm[half], 2);
      }
      float mn[2], ms[2];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        mn[half] = (m[half] == kNegInfP || bm[half] > m[half] + 8.f) ? fmaxf(m[half], bm[half]) : m[half];
        ms[half] = mn[half] == kNegInfP ? 0.f : mn[half];
      }
      if (__any_sync(0xffffffffu, mn[0] != m[0] || mn[1] != m[1])) {
        const float a0 = ex2(m[0] - ms[0]), a1 = ex2(m[1] - ms[1]);
        l[0] *= a0;
        l[1] *= a1;
#pragma unroll
        for (int i = 0; i < NT; ++i) {
          o[i][0] *= a0;
          o[i][1] *= a0;
          o[i][2] *= a1;
          o[i][3] *= a1;
        }
      }
      m[0] = mn[0];
      m[1] = mn[1];
      float pv[2][2][2];
#pragma unroll
      for (int half = 0; half < 2; ++half)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            pv[half][nt][jj] = ex2(sv[half][nt][jj] - ms[half]);
            l[half] += pv[half][nt][jj];
          }
      // P as the A operand of P·V: keys 0-7 from n-tile 0, keys 8-15 from n-tile 1
      const uint32_t pa0 = pack_bf16(pv[0][0][0], pv[0][0][1]);
      const uint32_t pa1 = pack_bf16(pv[1][0][0], pv[1][0][1]);
      const uint32_t pa2 = pack_bf16(pv[0][1][0], pv[0][1][1]);
      const uint32_t pa3 = pack_bf16(pv[1][1][0], pv[1][1][1]);
      // Slots at or beyond kv_end in the last block may never have been written, and slots
      // before the warp's window may hold anything (NaN included); 0 * NaN would poison the
      // sum, so zero those keys' V elements.  This lane's B fragments hold keys 2tq, 2tq+1
      // (b0, b2) and 8+2tq, 9+2tq (b1, b3).
      uint32_t vlo = 0xFFFFFFFFu, vhi = 0xFFFFFFFFu;
      if (kbase_pos + PA_BLOCK_SIZE > kv_end || kbase_pos < w_lo) {
        const int hi = kv_end - kbase_pos, lo = w_lo - kbase_pos;
        auto keep = [&](int r) { return r < hi && r >= lo; };
        vlo = (keep(2 * tq) ? 0x0000FFFFu : 0u) | (keep(2 * tq + 1) ? 0xFFFF0000u : 0u);
        vhi = (keep(2 * tq + 8) ? 0x0000FFFFu : 0u) | (keep(2 * tq + 9) ? 0xFFFF0000u : 0u);
      }
      {
        const int key = (lane & 7) + ((lane >> 3) & 1) * 8;  // matrices: [k0-7,d0],[k8-15,d0],[k0-7,d8],[k8-15,d8]
        const int dhalf = lane >> 4;
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {  // pairs of 8-wide d tiles = 16 d values
          const int ch16 = (np & 3) * 2 + dhalf;
          const uint32_t addr =
              smem_u32(vt + (np >> 2) * kChunkTile + key * 128 + ((ch16 ^ (key & 7)) << 4));
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(addr, b0, b1, b2, b3);
          mma_bf16(o[2 * np], pa0, pa1, pa2, pa3, b0 & vlo, b1 & vhi);
          mma_bf16(o[2 * np + 1], pa0, pa1, pa2, pa3, b2 & vlo, b3 & vhi);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }

  // finalize: reduce l over the quad, divide, write bf16 rows
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    l[half] += __shfl_xor_sync(0xffffffffu, l[half], 1);
    l[half] += __shfl_xor_sync(0xffffffffu, l[half], 2);
  }
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    if (!row_ok[half]) continue;
    const int r = t4 + 8 * half;
    const float inv = (bad || !(l[half] > 0.f)) ? 0.f : 1.f / l[half];
    __nv_bfloat16* orow =
        p.out + (static_cast<size_t>(qs + wt0 + r / p.G) * p.H_q + h_kv * p.G + r % p.G) * D;
#pragma unroll
    for (int i = 0; i < NT; ++i)
      *reinterpret_cast<uint32_t*>(orow + i * 8 + 2 * tq) = pack_bf16(o[i][2 * half] * inv, o[i][2 * half + 1] * inv);
  }
}

}  // namespace
}  // namespace pa

namespace pa {
namespace {
// Host checks of pa_prefill_attention; *work = false when there is nothing to enqueue.
pa_status prefill_check(const pa_cache_desc* desc, const void* out, const void* q, const void* k_cache,
                        const void* v_cache, const int32_t* block_tables, const int32_t* q_start,
                        const int32_t* context_lens, int max_query_len, float scale, bool* work) {
  *work = false;
  pa_status st = validate_desc(desc);
  if (st != PA_OK) return st;
  if (is_quantized(desc) || desc->num_sink > 0) return PA_ERR_UNSUPPORTED;
  if (max_query_len < 0 || !std::isfinite(scale)) return PA_ERR_INVALID_ARG;
  if (desc->num_seqs == 0 || max_query_len == 0) return PA_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !q_start || !context_lens)
    return PA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache) |
       reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 15u)
    return PA_ERR_INVALID_ARG;
  if (desc->num_seqs > 65535 || desc->num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
  *work = true;
  return PA_OK;
}

// pa_prefill_attention after its checks; step: the previous kernel is this step's append.
pa_status prefill_launch(const pa_cache_desc* desc, void* out, const void* q, const void* k_cache,
                         const void* v_cache, const int32_t* block_tables, const int32_t* q_start,
                         const int32_t* context_lens, int max_query_len, float scale, int32_t* err_flag,
                         void* stream, bool step) {
  const int D = desc->head_dim;
  const int G = desc->num_q_heads / desc->num_kv_heads;
#ifndef PA_PREFILL_WARP_MMA_ONLY
  if (D == 128 && (G & (G - 1)) == 0)  // the tensor-core (tcgen05) kernel
    return launch_prefill_tc(desc, out, q, k_cache, v_cache, block_tables, q_start, context_lens, max_query_len,
                             scale, err_flag, as_stream(stream), step);
#endif
  (void)step;  // the warp-MMA kernel waits for its predecessor before it starts
  const int nc = D * 2 / 128;
  const long long slots = static_cast<long long>(desc->num_blocks) * PA_BLOCK_SIZE;
  CUtensorMap mk, mv;
  if (!encode_cache_map(&mk, k_cache, 2, desc->num_kv_heads * nc, 1, slots) ||
      !encode_cache_map(&mv, v_cache, 2, desc->num_kv_heads * nc, 1, slots))
    return PA_ERR_CUDA;
  PrefillParams p;
  p.B = desc->num_seqs;
  p.H_q = desc->num_q_heads;
  p.H_kv = desc->num_kv_heads;
  p.G = desc->num_q_heads / desc->num_kv_heads;
  p.num_blocks = desc->num_blocks;
  p.max_blocks = desc->max_blocks_per_seq;
  p.max_q = max_query_len;
  p.window = desc->sliding_window;
  p.tpw = 16 / p.G;
  p.q_tile = kPfWarps * p.tpw;
  p.nc = nc;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.q_start = q_start;
  p.context_lens = context_lens;
  p.block_tables = block_tables;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.err = err_flag;
  const dim3 grid((max_query_len + p.q_tile - 1) / p.q_tile, p.B, p.H_kv);
  cudaStream_t s = as_stream(stream);
  if (D == 128)
    return launch_overlapped(prefill_kernel<128>, grid, dim3(kPfThreads), 0, s, mk, mv, p);
  return launch_overlapped(prefill_kernel<64>, grid, dim3(kPfThreads), 0, s, mk, mv, p);
}
}  // namespace
}  // namespace pa

extern "C" pa_status pa_prefill_attention(const pa_cache_desc* desc, void* out, const void* q,
                                          const void* k_cache, const void* v_cache,
                                          const int32_t* block_tables, const int32_t* q_start,
                                          const int32_t* context_lens, int max_query_len, float scale,
                                          int32_t* err_flag, void* stream) {
  bool work = false;
  const pa_status st = pa::prefill_check(desc, out, q, k_cache, v_cache, block_tables, q_start, context_lens,
                                         max_query_len, scale, &work);
  if (st != PA_OK || !work) return st;
  return pa::prefill_launch(desc, out, q, k_cache, v_cache, block_tables, q_start, context_lens, max_query_len,
                            scale, err_flag, stream, false);
}

extern "C" pa_status pa_prefill_step(const pa_cache_desc* desc, void* out, const void* q, void* k_cache,
                                     void* v_cache, const void* k_new, const void* v_new, int num_tokens,
                                     const int32_t* token_seq, const int32_t* token_pos,
                                     const int32_t* block_tables, const int32_t* q_start,
                                     const int32_t* context_lens, int max_query_len, float scale,
                                     int32_t* err_flag, void* stream) {
  // every argument of the attention half is checked before the append is enqueued
  bool work = false;
  const pa_status st = pa::prefill_check(desc, out, q, k_cache, v_cache, block_tables, q_start, context_lens,
                                         max_query_len, scale, &work);
  if (st != PA_OK) return st;
  const pa_status sa = pa_kv_append_tokens(desc, k_cache, v_cache, k_new, v_new, num_tokens, token_seq,
                                           token_pos, block_tables, err_flag, stream);
  if (sa != PA_OK || !work) return sa;
  return pa::prefill_launch(desc, out, q, k_cache, v_cache, block_tables, q_start, context_lens, max_query_len,
                            scale, err_flag, stream, num_tokens > 0);
}

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
//
// Caches that are not plain bf16 (8-bit K/V with per-head or per-token K scales, INT4 codes with
// a scale and zero point per 32 dims: "KV Cache 的显存账本" §七 and ldpk §5.2; or bf16 with sink
// tokens kept in their own buffer, same §七) go through prefill_dq_kernel: the same warps and tile
// math, but the four warps first load each 16-token block's codes (and the sink rows of sink
// positions) and write it as bf16 values, code times scale, into a double-buffered shared-memory
// tile in the layout the bf16 path reads, so each block is decoded once for all query rows.

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
  // prefill_dq_kernel only: the pools as bytes, the scales, the sink buffers and the byte offset
  // of the INT4 group parameters or per-token K scales inside each pool
  int num_sink;
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const float* k_scales;
  const float* v_scales;
  const __nv_bfloat16* k_sink;
  const __nv_bfloat16* v_sink;
  size_t extra_offset;
};

// One consumer warp's 16 query rows of a prefill tile: row r = (token r / G, query head r % G) of
// the warp's tpw = 16 / G query tokens.  S = Q·Kᵀ and O += P·V are m16n8k16 tensor-core products
// with the queries as M; P is reused straight from the S accumulator registers as the A operand
// of P·V.  block() takes one 16-key block whose K and V sit in shared memory as bf16 tiles of
// [16 slots][128 bytes] per 128-byte chunk of the head row, with the 128-byte swizzle.
template <int D>
struct PrefillRows {
  static constexpr int KT = D / 16;  // k-steps of Q·Kᵀ
  static constexpr int NT = D / 8;   // n-tiles of P·V
  int lane, t4, tq, wt0, w_tokens, w_last_pos, w_lo;
  int row_pos[2];
  bool row_ok[2];
  uint32_t qa[KT][4];  // Q fragments (A operand, rows x head_dim)
  float o[NT][4];
  float m[2], l[2];
  bool bad;

  __device__ __forceinline__ void init(const PrefillParams& p, int warp, int lane_, int qs, int h_kv, int t0,
                                       int t_end, int first_pos) {
    lane = lane_;
    t4 = lane >> 2;
    tq = lane & 3;
    wt0 = t0 + warp * p.tpw;  // this warp's first query token (chunk index)
    w_tokens = max(0, min(p.tpw, t_end - wt0));
    w_last_pos = first_pos + wt0 + w_tokens - 1;  // last query position of this warp
    // lowest key any row of this warp reads (its first token's window start)
    w_lo = p.window > 0 ? max(0, first_pos + wt0 - p.window + 1) : 0;
    // rows past the tokens are padding
    const int rows_used = w_tokens * p.G;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int r = t4 + 8 * half;
      row_ok[half] = r < rows_used;
      row_pos[half] = row_ok[half] ? first_pos + wt0 + r / p.G : -1;
    }
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
#pragma unroll
    for (int i = 0; i < NT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    m[0] = m[1] = kNegInfP;
    l[0] = l[1] = 0.f;
    bad = false;
  }

  // One block of 16 keys at positions kbase_pos.. (kv_end: first key past the tile's queries).
  __device__ __forceinline__ void block(const PrefillParams& p, const uint8_t* kt, const uint8_t* vt, int kbase_pos,
                                        int kv_end) {
    if (!(w_tokens > 0 && kbase_pos <= w_last_pos && kbase_pos + PA_BLOCK_SIZE > w_lo)) return;
    // S = Q Kᵀ for the 16 keys (two n-tiles of 8)
    float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      const int key = (lane & 7) + ((lane >> 4) & 1) * 8;  // matrices: [k0-7,d0],[k0-7,d8],[k8-15,d0],[k8-15,d8]
      const int dhalf = (lane >> 3) & 1;
#pragma unroll
      for (int kk = 0; kk < KT; ++kk) {
        const int ch16 = (kk & 3) * 2 + dhalf;
        const uint32_t addr = smem_u32(kt + (kk >> 2) * kChunkTile + key * 128 + ((ch16 ^ (key & 7)) << 4));
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
        const uint32_t addr = smem_u32(vt + (np >> 2) * kChunkTile + key * 128 + ((ch16 ^ (key & 7)) << 4));
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(addr, b0, b1, b2, b3);
        mma_bf16(o[2 * np], pa0, pa1, pa2, pa3, b0 & vlo, b1 & vhi);
        mma_bf16(o[2 * np + 1], pa0, pa1, pa2, pa3, b2 & vlo, b3 & vhi);
      }
    }
  }

  // reduce l over the quad, divide, write bf16 rows (zeros after a bad block id)
  __device__ __forceinline__ void finish(const PrefillParams& p, int qs, int h_kv) {
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
      __nv_bfloat16* orow = p.out + (static_cast<size_t>(qs + wt0 + r / p.G) * p.H_q + h_kv * p.G + r % p.G) * D;
#pragma unroll
      for (int i = 0; i < NT; ++i)
        *reinterpret_cast<uint32_t*>(orow + i * 8 + 2 * tq) =
            pack_bf16(o[i][2 * half] * inv, o[i][2 * half + 1] * inv);
    }
  }
};

template <int D>
__global__ void __launch_bounds__(kPfThreads)
    prefill_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const PrefillParams p) {
  constexpr int NC = D * 2 / 128;       // chunks per head row (bf16)
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
  PrefillRows<D> w;
  w.init(p, warp, lane, qs, h_kv, t0, t_end, first_pos);
  for (int k = 0; k < n_blocks; ++k) {
    const int st = k % kPfStages;
    const uint32_t ph = static_cast<uint32_t>(k / kPfStages) & 1u;
    if (!mbar_wait(&full[st], ph)) {
      if (lane == 0) set_error(p.err, PA_EFLAG_TIMEOUT);
      return;
    }
    if (bad_stage[st]) w.bad = true;
    else w.block(p, stages[st], stages[st] + NC * kChunkTile, (kb0 + k) * PA_BLOCK_SIZE, kv_end);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }
  w.finish(p, qs, h_kv);
}

// ------------------------------------------------------------------------------------
// Prefill over 8-bit, INT4 or sink-holding caches.  KIND 0: bf16 with sinks; 1: E4M3 K / INT8 V
// with per-head scales; 2: INT4 K and V (PA_INT4); 3: E4M3 K with per-token scales / INT8 V.
// A block's 2 x 16 x D/32 (tensor, token, 32-dim group) pieces are decoded by one thread each.
// ------------------------------------------------------------------------------------
template <int D, int KIND>
struct DqPiece {
  static constexpr int GROUPS = D / 32;
  uint32_t w[16];  // the piece's raw bytes (up to 64) as loaded
  float sc;        // its scale (8-bit), or the INT4 group's parameter word
  bool sink;       // a sink position: w holds bf16 values from the sink buffer

  // Load the piece of tensor t (0 K, 1 V), slot `slot` (the paged position pos), group g.
  __device__ __forceinline__ void load(const PrefillParams& p, int t, int s, int h, int pos, size_t slot, int g) {
    sink = pos < p.num_sink;
    if (sink || KIND == 0) {  // bf16 rows: 32 values = 64 bytes
      const __nv_bfloat16* src =
          sink ? (t ? p.v_sink : p.k_sink) + ((static_cast<size_t>(s) * p.num_sink + pos) * p.H_kv + h) * D + 32 * g
               : reinterpret_cast<const __nv_bfloat16*>(t ? p.v_cache : p.k_cache) + (slot * p.H_kv + h) * D + 32 * g;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 v = reinterpret_cast<const uint4*>(src)[i];
        w[4 * i] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
      }
      return;
    }
    if constexpr (KIND == 1 || KIND == 3) {  // 32 one-byte codes
      const uint8_t* src = (t ? p.v_cache : p.k_cache) + (slot * p.H_kv + h) * D + 32 * g;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint4 v = reinterpret_cast<const uint4*>(src)[i];
        w[4 * i] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
      }
      if (t) sc = p.v_scales[h];
      else if (KIND == 1) sc = p.k_scales[h];
      else sc = reinterpret_cast<const float*>(p.k_cache + p.extra_offset)[slot * p.H_kv + h];
    } else if constexpr (KIND == 2) {
      const uint8_t* row = (t ? p.v_cache : p.k_cache) + (slot * p.H_kv + h) * (D / 2);
      if (t == 0) {  // K: word 4c + g holds dims 32g + 8c + i at bits 4i
#pragma unroll
        for (int c = 0; c < 4; ++c) w[c] = reinterpret_cast<const uint32_t*>(row)[4 * c + g];
      } else {  // V: byte 8r + m holds dims 16m + r (bits 0-3) and 16m + r + 8 (bits 4-7); m = 2g, 2g + 1
#pragma unroll
        for (int r = 0; r < 8; ++r) w[r] = reinterpret_cast<const uint16_t*>(row + 8 * r + 2 * g)[0];
      }
      sc = __uint_as_float(reinterpret_cast<const uint32_t*>((t ? p.v_cache : p.k_cache) + p.extra_offset)
                               [(slot * p.H_kv + h) * GROUPS + g]);
    }
  }

  // The piece's 32 values as bf16 pairs, dims in order: code times scale in fp32, rounded.
  __device__ __forceinline__ void decode(int t, uint32_t (&out)[16]) const {
    if (sink || KIND == 0) {
#pragma unroll
      for (int i = 0; i < 16; ++i) out[i] = w[i];
    } else if constexpr (KIND == 1 || KIND == 3) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {  // word i: bytes = dims 4i .. 4i + 3
        float x[4];
        if (t == 0) {  // E4M3, decoded exactly through fp16
          const uint32_t lo = e4m3x2_to_f16x2(w[i]), hi = e4m3x2_to_f16x2(w[i] >> 16);
          const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
          const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
          x[0] = a.x, x[1] = a.y, x[2] = b.x, x[3] = b.y;
        } else {  // INT8
#pragma unroll
          for (int e = 0; e < 4; ++e) x[e] = static_cast<float>(static_cast<int8_t>((w[i] >> (8 * e)) & 0xFFu));
        }
        out[2 * i] = pack_bf16(x[0] * sc, x[1] * sc);
        out[2 * i + 1] = pack_bf16(x[2] * sc, x[3] * sc);
      }
    } else if constexpr (KIND == 2) {
      const uint32_t prm = __float_as_uint(sc);
      const float s = __uint_as_float(prm << 16), z = static_cast<float>((prm >> 16) & 0xFFu);
      float x[32];  // the group's dims in order
      if (t == 0) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 8; ++i) x[8 * c + i] = static_cast<float>((w[c] >> (4 * i)) & 0xFu);
      } else {
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          x[r] = static_cast<float>(w[r] & 0xFu);               // dim 32g + r       (m = 2g)
          x[8 + r] = static_cast<float>((w[r] >> 4) & 0xFu);    // dim 32g + 8 + r
          x[16 + r] = static_cast<float>((w[r] >> 8) & 0xFu);   // dim 32g + 16 + r  (m = 2g + 1)
          x[24 + r] = static_cast<float>((w[r] >> 12) & 0xFu);  // dim 32g + 24 + r
        }
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) out[i] = pack_bf16(s * (x[2 * i] - z), s * (x[2 * i + 1] - z));
    }
  }

  // Write the piece's 32 values as bf16 into row `row` of a [16 rows][128 B]-per-chunk tile with
  // the 128-byte swizzle: dims 32g + 8u .. + 7 form 16-byte unit 4g + u of the row.
  __device__ __forceinline__ void store(int t, uint8_t* tile, int row, int g) const {
    uint32_t out[16];
    decode(t, out);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int du = 4 * g + u, c = du >> 3, uu = du & 7;
      *reinterpret_cast<uint4*>(tile + c * kChunkTile + row * 128 + ((uu ^ (row & 7)) << 4)) =
          make_uint4(out[4 * u], out[4 * u + 1], out[4 * u + 2], out[4 * u + 3]);
    }
  }
};

template <int D, int KIND>
__global__ void __launch_bounds__(kPfWarps * 32)
    prefill_dq_kernel(const PrefillParams p) {
  constexpr int NC = D * 2 / 128;          // 128-byte chunks per bf16 head row
  constexpr int TILE = NC * kChunkTile;    // one tensor's bf16 tile of a block
  constexpr int GROUPS = D / 32;
  constexpr int PIECES = 2 * 16 * GROUPS;  // (tensor, token, group) pieces of a block: <= 128 threads
  __shared__ __align__(1024) uint8_t work[2][2 * TILE];
  __shared__ int bad_blk[2];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int s = blockIdx.y, h_kv = blockIdx.z, tile = blockIdx.x;
  grid_dep_wait();  // the previous kernel of the stream may still be writing any input
  const int qs = p.q_start[s];
  const int n = p.q_start[s + 1] - qs;
  const int ctx = p.context_lens[s];
  const bool valid = n >= 0 && n <= ctx && n <= p.max_q && ctx <= p.max_blocks * PA_BLOCK_SIZE;
  if (!valid) {
    if (tile == 0 && h_kv == 0 && tid == 0) set_error(p.err, PA_EFLAG_CTX_OVERFLOW);
    const int rows = min(max(n, 0), p.max_q);
    for (int t = tile * p.q_tile + warp; t < min(rows, (tile + 1) * p.q_tile); t += kPfWarps)
      for (int i = lane; i < p.G * D; i += 32)
        p.out[(static_cast<size_t>(qs + t) * p.H_q + h_kv * p.G) * D + i] = __float2bfloat16_rn(0.f);
    return;
  }
  const int t0 = tile * p.q_tile;
  if (t0 >= n) return;
  const int first_pos = ctx - n;
  const int t_end = min(n, t0 + p.q_tile);
  const int kv_end = first_pos + t_end;
  const int kv_lo = p.window > 0 ? max(0, first_pos + t0 - p.window + 1) : 0;
  const int kb0 = kv_lo / PA_BLOCK_SIZE;
  const int n_blocks = (kv_end + PA_BLOCK_SIZE - 1) / PA_BLOCK_SIZE - kb0;
  const int32_t* trow = p.block_tables + static_cast<size_t>(s) * p.max_blocks + kb0;

  PrefillRows<D> w;
  w.init(p, warp, lane, qs, h_kv, t0, t_end, first_pos);

  // this thread's piece: tensor pt, token row pr, 32-dim group pg
  const bool piece = tid < PIECES;
  const int pt = tid / (16 * GROUPS), pr = (tid / GROUPS) % 16, pg = tid % GROUPS;
  DqPiece<D, KIND> cur;
  // Block k's table entry, or -1 when the block holds only sink positions (its slots are never
  // read) and -2 when the entry is outside the pool.
  auto entry = [&](int k) -> int {
    const int kpos = (kb0 + k) * PA_BLOCK_SIZE;
    if (kpos + PA_BLOCK_SIZE <= p.num_sink) return -1;
    const int e = trow[k];
    return (e < 0 || e >= p.num_blocks) ? -2 : e;
  };
  auto load = [&](int k, int e) {
    const int pos = (kb0 + k) * PA_BLOCK_SIZE + pr;
    if (piece && e != -2 && (e >= 0 || pos < p.num_sink))
      cur.load(p, pt, s, h_kv, pos, static_cast<size_t>(max(e, 0)) * PA_BLOCK_SIZE + pr, pg);
  };
  int e = n_blocks > 0 ? entry(0) : 0;
  if (n_blocks > 0) load(0, e);
  for (int k = 0; k < n_blocks; ++k) {
    uint8_t* wk = work[k & 1];
    if (piece && e != -2) cur.store(pt, wk + pt * TILE, pr, pg);
    if (tid == 0) {
      bad_blk[k & 1] = e == -2 ? 1 : 0;
      if (e == -2) set_error(p.err, PA_EFLAG_BAD_BLOCK_ID);
    }
    // the next block's codes are read while this one is computed
    if (k + 1 < n_blocks) {
      e = entry(k + 1);
      load(k + 1, e);
    }
    __syncthreads();
    if (bad_blk[k & 1]) w.bad = true;
    else w.block(p, wk, wk + TILE, (kb0 + k) * PA_BLOCK_SIZE, kv_end);
  }
  w.finish(p, qs, h_kv);
}

// ------------------------------------------------------------------------------------
// Decoded copy for the tensor-core prefill (pa_prefill_attention_ws).  CTA (b, s) decodes
// logical block b of sequence s, if the chunk's queries can attend it, into block s * mb + b of
// a bf16 pool with the cache's slot-major layout (the same DqPiece arithmetic as
// prefill_dq_kernel: code times scale in fp32 rounded to bf16, sink positions from the sink
// buffers), and writes the dense table entry dense[s][b]: that block, or -1 for a block no query
// attends or whose table entry lies outside the pool (the attention kernel then reports it).
// ------------------------------------------------------------------------------------
template <int D, int KIND>
__global__ void __launch_bounds__(256)
    prefill_expand_kernel(const PrefillParams p, int mb, __nv_bfloat16* kx, __nv_bfloat16* vx, int32_t* dense) {
  constexpr int GROUPS = D / 32;
  const int b = blockIdx.x, s = blockIdx.y;
  grid_dep_wait();  // the previous kernel of the stream may still be writing any input
  const int n = p.q_start[s + 1] - p.q_start[s];
  const int ctx = p.context_lens[s];
  const bool valid = n >= 0 && n <= ctx && n <= p.max_q && ctx <= p.max_blocks * PA_BLOCK_SIZE &&
                     ctx <= mb * PA_BLOCK_SIZE;
  // the positions the chunk's queries attend: from the first query's window start to ctx - 1
  const int lo = p.window > 0 ? max(0, ctx - n - p.window + 1) : 0;
  int e = -1;  // the block's pool entry (0 for a block of sink positions only: none is read)
  if (valid && b >= lo / PA_BLOCK_SIZE && b * PA_BLOCK_SIZE < ctx) {
    if ((b + 1) * PA_BLOCK_SIZE <= p.num_sink) {
      e = 0;
    } else {
      const int t = p.block_tables[static_cast<size_t>(s) * p.max_blocks + b];
      e = (t < 0 || t >= p.num_blocks) ? -1 : t;
    }
  }
  const size_t xb = static_cast<size_t>(s) * mb + b;  // the block of the bf16 pool
  if (threadIdx.x == 0) dense[xb] = e >= 0 ? static_cast<int32_t>(xb) : -1;
  if (e < 0) return;
  const int pieces = 2 * PA_BLOCK_SIZE * p.H_kv * GROUPS;  // (tensor, slot, head, 32-dim group)
  for (int i = threadIdx.x; i < pieces; i += blockDim.x) {
    const int g = i % GROUPS, h = (i / GROUPS) % p.H_kv;
    const int r = (i / (GROUPS * p.H_kv)) % PA_BLOCK_SIZE, t = i / (GROUPS * p.H_kv * PA_BLOCK_SIZE);
    DqPiece<D, KIND> pc;
    pc.load(p, t, s, h, b * PA_BLOCK_SIZE + r, static_cast<size_t>(e) * PA_BLOCK_SIZE + r, g);
    uint32_t out[16];
    pc.decode(t, out);
    uint4* dst = reinterpret_cast<uint4*>((t ? vx : kx) + ((xb * PA_BLOCK_SIZE + r) * p.H_kv + h) * D + 32 * g);
#pragma unroll
    for (int u = 0; u < 4; ++u) dst[u] = make_uint4(out[4 * u], out[4 * u + 1], out[4 * u + 2], out[4 * u + 3]);
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

PrefillParams prefill_params(const pa_cache_desc* desc, void* out, const void* q, const void* k_cache,
                             const void* v_cache, const int32_t* block_tables, const int32_t* q_start,
                             const int32_t* context_lens, int max_query_len, float scale, int32_t* err_flag) {
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
  p.nc = desc->head_dim * 2 / 128;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.q_start = q_start;
  p.context_lens = context_lens;
  p.block_tables = block_tables;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.err = err_flag;
  p.num_sink = desc->num_sink;
  p.k_cache = static_cast<const uint8_t*>(k_cache);
  p.v_cache = static_cast<const uint8_t*>(v_cache);
  p.k_scales = desc->k_scales;
  p.v_scales = desc->v_scales;
  p.k_sink = static_cast<const __nv_bfloat16*>(desc->k_sink);
  p.v_sink = static_cast<const __nv_bfloat16*>(desc->v_sink);
  p.extra_offset = is_int4(desc) ? int4_params_offset(desc) : (has_token_scales(desc) ? token_scales_offset(desc) : 0);
  return p;
}

// pa_prefill_attention after its checks; step: the previous kernel is this step's append.
pa_status prefill_launch(const pa_cache_desc* desc, void* out, const void* q, const void* k_cache,
                         const void* v_cache, const int32_t* block_tables, const int32_t* q_start,
                         const int32_t* context_lens, int max_query_len, float scale, int32_t* err_flag,
                         void* stream, bool step) {
  const int D = desc->head_dim;
  const int G = desc->num_q_heads / desc->num_kv_heads;
  const bool dq = is_quantized(desc) || desc->num_sink > 0;  // decoded per block (prefill_dq_kernel)
#ifndef PA_PREFILL_WARP_MMA_ONLY
  if (!dq && D == 128 && (G & (G - 1)) == 0)  // the tensor-core (tcgen05) kernel
    return launch_prefill_tc(desc, out, q, k_cache, v_cache, block_tables, q_start, context_lens, max_query_len,
                             scale, err_flag, as_stream(stream), step);
#endif
  (void)step;  // the warp-MMA kernel waits for its predecessor before it starts
  const int nc = D * 2 / 128;
  const long long slots = static_cast<long long>(desc->num_blocks) * PA_BLOCK_SIZE;
  CUtensorMap mk, mv;
  if (!dq && (!encode_cache_map(&mk, k_cache, 2, desc->num_kv_heads * nc, 1, slots) ||
              !encode_cache_map(&mv, v_cache, 2, desc->num_kv_heads * nc, 1, slots)))
    return PA_ERR_CUDA;
  const PrefillParams p = prefill_params(desc, out, q, k_cache, v_cache, block_tables, q_start, context_lens,
                                         max_query_len, scale, err_flag);
  const dim3 grid((max_query_len + p.q_tile - 1) / p.q_tile, p.B, p.H_kv);
  cudaStream_t s = as_stream(stream);
  if (dq) {  // 8-bit and INT4 caches have head_dim 128 (validate_desc)
    const dim3 block(kPfWarps * 32);
    if (is_int4(desc)) return launch_overlapped(prefill_dq_kernel<128, 2>, grid, block, 0, s, p);
    if (has_token_scales(desc)) return launch_overlapped(prefill_dq_kernel<128, 3>, grid, block, 0, s, p);
    if (is_quantized(desc)) return launch_overlapped(prefill_dq_kernel<128, 1>, grid, block, 0, s, p);
    if (D == 128) return launch_overlapped(prefill_dq_kernel<128, 0>, grid, block, 0, s, p);
    return launch_overlapped(prefill_dq_kernel<64, 0>, grid, block, 0, s, p);
  }
  if (D == 128)
    return launch_overlapped(prefill_kernel<128>, grid, dim3(kPfThreads), 0, s, mk, mv, p);
  return launch_overlapped(prefill_kernel<64>, grid, dim3(kPfThreads), 0, s, mk, mv, p);
}

// Bytes of pa_prefill_attention_ws's workspace (and the bf16 pool's blocks per sequence in *mb):
// 0 when the call needs none (a bf16 cache without sinks, or a shape the tensor-core kernel does
// not take) or the arguments are invalid.
size_t prefill_ws_bytes(const pa_cache_desc* d, int max_ctx, int* mb_out) {
  if (validate_desc(d) != PA_OK || max_ctx < 0 ||
      static_cast<long long>(max_ctx) > static_cast<long long>(d->max_blocks_per_seq) * PA_BLOCK_SIZE)
    return 0;
#ifdef PA_PREFILL_WARP_MMA_ONLY
  return 0;
#else
  const int G = d->num_q_heads / d->num_kv_heads;
  const bool dq = is_quantized(d) || d->num_sink > 0;
  if (!dq || d->head_dim != 128 || (G & (G - 1)) != 0) return 0;
  const int mb = std::max(1, (max_ctx + PA_BLOCK_SIZE - 1) / PA_BLOCK_SIZE);
  // slot indices of the bf16 pool stay within int32 (the tensor maps' coordinates)
  if (static_cast<long long>(d->num_seqs) * mb * PA_BLOCK_SIZE > 0x7FFFFFFFLL) return 0;
  if (mb_out) *mb_out = mb;
  const size_t table = (static_cast<size_t>(d->num_seqs) * mb * 4 + 255) / 256 * 256;
  const size_t pool = static_cast<size_t>(d->num_seqs) * mb * PA_BLOCK_SIZE * d->num_kv_heads * 128 * 2;
  return table + 2 * pool;
#endif
}

// The expanded path: decode every attended block once into the workspace's bf16 pool, then the
// tensor-core kernel over that pool and its dense table (as a bf16 cache without sinks).
pa_status prefill_expanded(const pa_cache_desc* desc, void* out, const void* q, const void* k_cache,
                           const void* v_cache, const int32_t* block_tables, const int32_t* q_start,
                           const int32_t* context_lens, int max_query_len, float scale, int mb, void* workspace,
                           int32_t* err_flag, void* stream) {
  const PrefillParams p = prefill_params(desc, out, q, k_cache, v_cache, block_tables, q_start, context_lens,
                                         max_query_len, scale, err_flag);
  const size_t table = (static_cast<size_t>(desc->num_seqs) * mb * 4 + 255) / 256 * 256;
  const size_t pool = static_cast<size_t>(desc->num_seqs) * mb * PA_BLOCK_SIZE * desc->num_kv_heads * 128 * 2;
  int32_t* dense = static_cast<int32_t*>(workspace);
  auto* kx = reinterpret_cast<__nv_bfloat16*>(static_cast<uint8_t*>(workspace) + table);
  auto* vx = reinterpret_cast<__nv_bfloat16*>(static_cast<uint8_t*>(workspace) + table + pool);
  cudaStream_t s = as_stream(stream);
  const dim3 grid(mb, desc->num_seqs), block(256);
  pa_status st;
  if (is_int4(desc)) st = launch_overlapped(prefill_expand_kernel<128, 2>, grid, block, 0, s, p, mb, kx, vx, dense);
  else if (has_token_scales(desc))
    st = launch_overlapped(prefill_expand_kernel<128, 3>, grid, block, 0, s, p, mb, kx, vx, dense);
  else if (is_quantized(desc))
    st = launch_overlapped(prefill_expand_kernel<128, 1>, grid, block, 0, s, p, mb, kx, vx, dense);
  else st = launch_overlapped(prefill_expand_kernel<128, 0>, grid, block, 0, s, p, mb, kx, vx, dense);
  if (st != PA_OK) return st;
  pa_cache_desc x = *desc;  // the bf16 pool: every attended block, sinks included, in place
  x.k_dtype = x.v_dtype = PA_BF16;
  x.k_scales = x.v_scales = nullptr;
  x.k_sink = x.v_sink = nullptr;
  x.num_sink = 0;
  x.num_blocks = desc->num_seqs * mb;
  x.max_blocks_per_seq = mb;
  return launch_prefill_tc(&x, out, q, kx, vx, dense, q_start, context_lens, max_query_len, scale, err_flag, s,
                           false);
}
}  // namespace
}  // namespace pa

extern "C" size_t pa_prefill_workspace_size(const pa_cache_desc* desc, int max_context_len) {
  return pa::prefill_ws_bytes(desc, max_context_len, nullptr);
}

extern "C" pa_status pa_prefill_attention_ws(const pa_cache_desc* desc, void* out, const void* q,
                                             const void* k_cache, const void* v_cache,
                                             const int32_t* block_tables, const int32_t* q_start,
                                             const int32_t* context_lens, int max_query_len, int max_context_len,
                                             float scale, void* workspace, size_t workspace_bytes,
                                             int32_t* err_flag, void* stream) {
  bool work = false;
  const pa_status st = pa::prefill_check(desc, out, q, k_cache, v_cache, block_tables, q_start, context_lens,
                                         max_query_len, scale, &work);
  if (st != PA_OK) return st;
  if (max_context_len < 0 ||
      static_cast<long long>(max_context_len) > static_cast<long long>(desc->max_blocks_per_seq) * PA_BLOCK_SIZE)
    return PA_ERR_INVALID_ARG;
  int mb = 0;
  const size_t need = pa::prefill_ws_bytes(desc, max_context_len, &mb);
  if (need > 0) {
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return PA_ERR_INVALID_ARG;
    if (workspace_bytes < need) return PA_ERR_WORKSPACE_TOO_SMALL;
  }
  if (!work) return PA_OK;
  if (need == 0)
    return pa::prefill_launch(desc, out, q, k_cache, v_cache, block_tables, q_start, context_lens, max_query_len,
                              scale, err_flag, stream, false);
  return pa::prefill_expanded(desc, out, q, k_cache, v_cache, block_tables, q_start, context_lens, max_query_len,
                              scale, mb, workspace, err_flag, stream);
}

extern "C" pa_status pa_prefill_step_ws(const pa_cache_desc* desc, void* out, const void* q, void* k_cache,
                                        void* v_cache, const void* k_new, const void* v_new, int num_tokens,
                                        const int32_t* token_seq, const int32_t* token_pos,
                                        const int32_t* block_tables, const int32_t* q_start,
                                        const int32_t* context_lens, int max_query_len, int max_context_len,
                                        float scale, void* workspace, size_t workspace_bytes, int32_t* err_flag,
                                        void* stream) {
  // every argument of the attention half is checked before the append is enqueued
  bool work = false;
  const pa_status st = pa::prefill_check(desc, out, q, k_cache, v_cache, block_tables, q_start, context_lens,
                                         max_query_len, scale, &work);
  if (st != PA_OK) return st;
  if (max_context_len < 0 ||
      static_cast<long long>(max_context_len) > static_cast<long long>(desc->max_blocks_per_seq) * PA_BLOCK_SIZE)
    return PA_ERR_INVALID_ARG;
  int mb = 0;
  const size_t need = pa::prefill_ws_bytes(desc, max_context_len, &mb);
  if (need > 0) {
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return PA_ERR_INVALID_ARG;
    if (workspace_bytes < need) return PA_ERR_WORKSPACE_TOO_SMALL;
  }
  const pa_status sa = pa_kv_append_tokens(desc, k_cache, v_cache, k_new, v_new, num_tokens, token_seq,
                                           token_pos, block_tables, err_flag, stream);
  if (sa != PA_OK || !work) return sa;
  if (need == 0)
    return pa::prefill_launch(desc, out, q, k_cache, v_cache, block_tables, q_start, context_lens, max_query_len,
                              scale, err_flag, stream, num_tokens > 0);
  // the expand kernel waits for the append before it reads anything
  return pa::prefill_expanded(desc, out, q, k_cache, v_cache, block_tables, q_start, context_lens, max_query_len,
                              scale, mb, workspace, err_flag, stream);
}

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

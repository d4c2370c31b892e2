// Chunked-prefill attention on the fifth-generation tensor cores (tcgen05, TMEM).
//
// What is computed is the same as the warp-MMA kernel in prefill_attention.cu: untitled KV-cache
// article at ldpk.cn/news/58971 §2.2 (causal attention of every new position over the positions up
// to itself) and §7 (chunked prefill), over the paged cache through the block table ("KV Cache 的显存
// 账本：PagedAttention 与连续批处理" §四), GQA grouping (same page §二), and an optional sliding
// window (ldpk §5.3).
//
// Design (head_dim 128, G = 1, 2, 4 or 8 query heads per KV head):
//  * One CTA per (256 query rows, sequence, KV head): two query tiles of 128 rows, a row being
//    (token, query head), share every K/V tile.  A 128-key tile is 8 scattered physical blocks and
//    the canonical operand layout needs one TMA box per block and 64-dim half (32 boxes per K+V
//    tile); sharing it between two query tiles halves the boxes per flop, which is what bounds the
//    copy engine here.
//  * S = Q·Kᵀ and O += P·V are tcgen05.mma (kind::f16, bf16 operands, M = N = 128, fp32
//    accumulators in TMEM: S0, S1, O0, O1 in 4 x 128 columns), issued by one thread; the next
//    tile's S is issued as soon as the softmax has read this one, ahead of this tile's P·V.
//    Q, K, P are K-major and V is MN-major shared-memory operands with the 128-byte swizzle.
//  * A producer warp streams K through a two-stage ring and V through one stage.
//  * Two softmax warpgroups (one per query tile) own one query row per thread through TMEM
//    lanes: they read S, mask (causal, window), keep the running maximum (moved only when a score
//    exceeds it by 2^8), write P as bf16 into their swizzled P tile, rescale O in TMEM when the
//    maximum moved, and finally normalise O into the output.  V rows of keys that are not loaded
//    or lie beyond the context are zeroed before P·V reads them, so bits left in unused slots (NaN
//    included) cannot leak.
//  * Every wait is bounded; TMEM is released on every path.

#include <algorithm>
#include <cmath>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kTcThreads = 320;                 // 10 warps: producer, MMA, 2 x 4 softmax
constexpr int kHalf = 128 * 128;                // 128 rows x 128 bytes (64 bf16): one K-half
constexpr int kTile = 2 * kHalf;                // a 128 x 128 bf16 operand tile
constexpr int kQOff = 0;                        // Q0, Q1
constexpr int kKOff = kQOff + 2 * kTile;        // K stages 0, 1
constexpr int kVOff = kKOff + 2 * kTile;        // V (one stage)
constexpr int kPOff = kVOff + kTile;            // P0, P1
constexpr int kBarOff = kPOff + 2 * kTile;
constexpr int kTcSmem = kBarOff + 256 + 1024;   // barriers, and slack for 1024-byte alignment
constexpr uint32_t kTmemCols = 512;             // S0 0..127, S1 128..255, O0 256..383, O1 384..511
constexpr float kNegInfTc = -INFINITY;

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator (bits 4-5 = 1), bf16 A and B
// (bits 7-9, 10-12 = 1), K-major A (bit 15 = 0), N / 8 in bits 17-22, M / 16 in bits 24-28.
// Bit 16 selects an MN-major B (V in P·V).
constexpr uint32_t kIdescS = (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kIdescPV = kIdescS | (1u << 16);

struct TcParams {
  int B, H_q, H_kv, G, num_blocks, max_blocks, max_q, window;
  int tpq;  // tokens per query tile: 128 / G (a CTA holds two tiles)
  float scale_log2;
  const int32_t* q_start;
  const int32_t* context_lens;
  const int32_t* block_tables;
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  int32_t* err;
};

// Shared-memory operand descriptor, 128-byte swizzle: start address (bits 0-13), leading and
// stride byte offsets (bits 16-29, 32-45; all encoded >> 4), the fixed 0b001 of bits 46-48, and
// swizzle mode 2 in bits 61-63.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// This warp's 32 TMEM lanes x 32 consecutive fp32 columns: thread i gets lane base + i.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31]) : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// A wait that every lane of the warp leaves with the same answer.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const TcParams p) {
  constexpr int D = 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBarOff);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;   // [2]
  uint64_t* k_empty = bars + 3;  // [2]
  uint64_t* v_full = bars + 5;
  uint64_t* v_empty = bars + 6;
  uint64_t* s_full = bars + 7;   // [2] per query tile
  uint64_t* s_free = bars + 9;   // [2]
  uint64_t* p_full = bars + 11;  // [2]
  uint64_t* o_done = bars + 13;  // [2]
  uint64_t* drain = bars + 15;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  int* flags = reinterpret_cast<int*>(bars + 17);  // [0] a bad block id, [1] a wait gave up

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int s = blockIdx.y, h_kv = blockIdx.z, tile = blockIdx.x;
  const int tpc = 2 * p.tpq;  // tokens per CTA
  // launched with programmatic dependent launch: the previous kernel may still write any input
  grid_dep_wait();
  const int qs = p.q_start[s];
  const int n = p.q_start[s + 1] - qs;
  const int ctx = p.context_lens[s];
  const bool valid = n >= 0 && n <= ctx && n <= p.max_q && ctx <= p.max_blocks * PA_BLOCK_SIZE;
  if (!valid) {
    if (tile == 0 && h_kv == 0 && tid == 0) set_error(p.err, PA_EFLAG_CTX_OVERFLOW);
    const int rows = min(max(n, 0), p.max_q);
    for (int t = tile * tpc + warp; t < min(rows, (tile + 1) * tpc); t += kTcThreads / 32)
      for (int i = lane; i < p.G * D; i += 32)
        p.out[(static_cast<size_t>(qs + t) * p.H_q + h_kv * p.G) * D + i] = __float2bfloat16_rn(0.f);
    return;
  }
  const int t0 = tile * tpc;
  if (t0 >= n) return;
  const bool has1 = t0 + p.tpq < n;  // the second query tile holds tokens
  const int first_pos = ctx - n;
  const int t_end = min(n, t0 + tpc);
  const int kv_end = first_pos + t_end;  // keys [kv_lo, kv_end) are visible to this CTA
  const int kv_lo = p.window > 0 ? max(0, first_pos + t0 - p.window + 1) : 0;
  const int kb0 = kv_lo / PA_BLOCK_SIZE;
  const int kb_end = (kv_end + PA_BLOCK_SIZE - 1) / PA_BLOCK_SIZE;
  const int n_tiles = (kb_end - kb0 + 7) / 8;
  const int loaded_end = min(ctx, kb_end * PA_BLOCK_SIZE);  // keys past this hold no loaded data

  if (tid == 0) {
    mbar_init(q_full, 256);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 128);
      mbar_init(&p_full[i], 128);
      mbar_init(&o_done[i], 1);
    }
    mbar_init(v_full, 1);
    mbar_init(v_empty, 1);
    mbar_init(drain, 1);
    flags[0] = flags[1] = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------ producer ------------------------------
    const int32_t* row = p.block_tables + static_cast<size_t>(s) * p.max_blocks;
    const int i = lane >> 1, half = lane & 1;  // lanes 0..15: block i of the tile, 64-dim half
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(policy));
    // one K or V tile: 16 boxes of 16 slots x 128 bytes; returns false when a wait gave up
    auto load = [&](int k, const CUtensorMap* map, uint64_t* full, uint64_t* empty, uint32_t parity,
                    uint8_t* dst) -> bool {
      if (!warp_wait(empty, parity)) return false;
      const int kb = kb0 + 8 * k + i;
      int pb = -1;
      if (lane < 16 && kb < kb_end) {
        pb = row[kb];
        if (pb < 0 || pb >= p.num_blocks) {
          if (half == 0) {
            flags[0] = 1;
            set_error(p.err, PA_EFLAG_BAD_BLOCK_ID);
          }
          pb = -1;
        }
      }
      const unsigned loads = __ballot_sync(0xffffffffu, pb >= 0);
      if (lane == 0) {
        const uint32_t bytes = __popc(loads) * 2048u;
        if (bytes) mbar_arrive_expect_tx(full, bytes);
        else mbar_arrive(full);
      }
      __syncwarp();
      if (pb >= 0)
        tma_load_3d(dst + half * kHalf + i * 2048, map, full, 0, h_kv * 2 + half, pb * PA_BLOCK_SIZE, policy);
      return true;
    };
    auto load_k = [&](int k) {
      return load(k, &tmK, &k_full[k & 1], &k_empty[k & 1], (static_cast<uint32_t>(k >> 1) & 1u) ^ 1u,
                  sm + kKOff + (k & 1) * kTile);
    };
    auto load_v = [&](int k) {
      return load(k, &tmV, v_full, v_empty, (static_cast<uint32_t>(k) & 1u) ^ 1u, sm + kVOff);
    };
    // K runs one tile ahead of V (V has a single stage and is freed last)
    int nk = 0, nv = 0;
    bool ok = load_k(0);
    nk += ok;
    if (ok && n_tiles > 1) nk += (ok = load_k(1));
    if (ok) nv += (ok = load_v(0));
    for (int k = 1; ok && k < n_tiles; ++k) {
      if (k + 1 < n_tiles) {
        if (!(ok = load_k(k + 1))) break;
        ++nk;
      }
      if (!(ok = load_v(k))) break;
      ++nv;
    }
    if (!ok && lane == 0) flags[1] = 1;
    // do not leave while a copy into shared memory may still be in flight
    for (int st = 0; st < 2 && st < nk; ++st) {
      const int last = st + 2 * ((nk - 1 - st) / 2);
      if (!warp_wait(&k_full[st], static_cast<uint32_t>(last >> 1) & 1u) && lane == 0) flags[1] = 1;
    }
    if (nv > 0 && !warp_wait(v_full, static_cast<uint32_t>(nv - 1) & 1u) && lane == 0) flags[1] = 1;
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      auto issue_s = [&](int w, int k) {  // S_w = Q_w K^T of tile k
        const uint32_t qb = smem_u32(sm + kQOff + w * kTile);
        const uint32_t kbuf = smem_u32(sm + kKOff + (k & 1) * kTile);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          tc_mma(tmem + w * 128, sw128_desc(qb + off, 16, 1024), sw128_desc(kbuf + off, 16, 1024), kIdescS, kk > 0);
        }
        tc_commit(&s_full[w]);
      };
      auto issue_pv = [&](int w, int k) {  // O_w += P_w V of tile k
        const uint32_t pbuf = smem_u32(sm + kPOff + w * kTile);
        const uint32_t vbuf = smem_u32(sm + kVOff);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t aoff = (kk >> 2) * kHalf + (kk & 3) * 32;  // P: keys 16kk .. 16kk+15
          const uint32_t boff = kk * 16 * 128;                      // V: key rows 16kk .. of both halves
          tc_mma(tmem + 256 + w * 128, sw128_desc(pbuf + aoff, 16, 1024), sw128_desc(vbuf + boff, kHalf, 1024),
                 kIdescPV, (k > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&o_done[w]);
      };
      bool ok = mbar_wait(q_full, 0) && mbar_wait(&k_full[0], 0);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        if (has1) issue_s(1, 0);
        tc_commit(&k_empty[0]);
      }
      for (int k = 0; ok && k < n_tiles; ++k) {
        const uint32_t ph = static_cast<uint32_t>(k) & 1u;
        // S of the next tile as soon as each softmax group has read this one
        if (k + 1 < n_tiles) {
          ok = mbar_wait(&s_free[0], ph) && mbar_wait(&k_full[(k + 1) & 1], static_cast<uint32_t>((k + 1) >> 1) & 1u);
          if (!ok) break;
          tc_fence_after();
          issue_s(0, k + 1);
          if (has1) {
            if (!(ok = mbar_wait(&s_free[1], ph))) break;
            tc_fence_after();
            issue_s(1, k + 1);
          }
          tc_commit(&k_empty[(k + 1) & 1]);
        }
        if (!(ok = mbar_wait(v_full, ph) && mbar_wait(&p_full[0], ph))) break;
        tc_fence_after();
        issue_pv(0, k);
        if (has1) {
          if (!(ok = mbar_wait(&p_full[1], ph))) break;
          tc_fence_after();
          issue_pv(1, k);
        }
        tc_commit(v_empty);
      }
      if (!ok) {
        flags[1] = 1;
        // let every product already issued finish before the columns are released
        tc_commit(drain);
        mbar_wait(drain, 0);
      }
    }
  } else {
    // ------------------------------ softmax warpgroups ------------------------------
    const int wg = (warp - 2) >> 2;  // query tile of this group
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // this thread's row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + wg * 128 + lane_off, tO = tmem + 256 + wg * 128 + lane_off;
    const int tq0 = t0 + wg * p.tpq;  // first token of this query tile
    const int tok = r / p.G, hh = r - tok * p.G;
    const bool row_ok = tq0 + tok < t_end;
    const int row_pos = first_pos + tq0 + tok;
    const int row_lo = p.window > 0 ? max(0, row_pos - p.window + 1) : 0;
    uint8_t* qtile = sm + kQOff + wg * kTile;
    uint8_t* ptile = sm + kPOff + wg * kTile;
    {  // Q row -> swizzled Q tile
      const uint4* qrow = reinterpret_cast<const uint4*>(
          p.q + (static_cast<size_t>(qs + (row_ok ? tq0 + tok : t0)) * p.H_q + h_kv * p.G + hh) * D);
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const uint4 v = row_ok ? qrow[c] : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(qtile + (c >> 3) * kHalf + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = v;
      }
      fence_proxy_async();
      mbar_arrive(q_full);
    }
    const bool active = wg == 0 || has1;
    float m_run = kNegInfTc, l_run = 0.f;
    bool ok = true;
    for (int k = 0; active && k < n_tiles; ++k) {
      const uint32_t ph = static_cast<uint32_t>(k) & 1u;
      if (!warp_wait(&s_full[wg], ph)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sv[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(sv + 32 * c));
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&s_free[wg]);
      const int kbase = (kb0 + 8 * k) * PA_BLOCK_SIZE;
      // scores stay raw (the scale is positive, so the maximum commutes with it); only tiles
      // that cross a row's causal or window edge take the per-key mask
      if (!__all_sync(0xffffffffu, row_ok && kbase + 127 <= row_pos && kbase >= row_lo)) {
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          const int kp = kbase + c;
          if (!(row_ok && kp <= row_pos && kp >= row_lo)) sv[c] = __float_as_uint(kNegInfTc);
        }
      }
      float mx4[4] = {kNegInfTc, kNegInfTc, kNegInfTc, kNegInfTc};
#pragma unroll
      for (int c = 0; c < 128; ++c) mx4[c & 3] = fmaxf(mx4[c & 3], __uint_as_float(sv[c]));
      const float mraw = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      const float mx = mraw == kNegInfTc ? kNegInfTc : mraw * p.scale_log2;
      const float m_new = (m_run == kNegInfTc || mx > m_run + 8.f) ? fmaxf(m_run, mx) : m_run;
      const float ms = m_new == kNegInfTc ? 0.f : m_new;
      const float alpha = ex2(m_run - ms);
      // P·V of the previous tile must be done: P is rewritten and O may be rescaled
      if (k > 0) {
        if (!warp_wait(&o_done[wg], ph ^ 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      float ls4[4] = {0.f, 0.f, 0.f, 0.f};
      const float sl = p.scale_log2;
#pragma unroll
      for (int c = 0; c < 128; c += 8) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a = ex2(fmaf(__uint_as_float(sv[c + 2 * e]), sl, -ms));
          const float b = ex2(fmaf(__uint_as_float(sv[c + 2 * e + 1]), sl, -ms));
          ls4[e] += a + b;
          w[e] = pack_bf16(a, b);
        }
        *reinterpret_cast<uint4*>(ptile + (c >> 6) * kHalf + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4)) =
            make_uint4(w[0], w[1], w[2], w[3]);
      }
      l_run = l_run * alpha + ((ls4[0] + ls4[1]) + (ls4[2] + ls4[3]));
      if (k > 0 && __any_sync(0xffffffffu, m_new != m_run)) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t ov[32];
          tmem_ld32(tO + 32 * c, ov);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
          tmem_st32(tO + 32 * c, ov);
        }
        tmem_wait_st();
      }
      m_run = m_new;
      // key row r of V: zero it when it holds no loaded in-context data (both groups write the
      // same zeros; each must see them before its own P·V)
      const int kp_r = kbase + r;
      const bool zero_row = kp_r < kv_lo || kp_r >= loaded_end;
      if (__any_sync(0xffffffffu, zero_row)) {
        if (!warp_wait(v_full, ph)) {  // the tile's copies must have landed first
          ok = false;
          break;
        }
      }
      if (zero_row) {
        uint8_t* vrow = sm + kVOff + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          *reinterpret_cast<uint4*>(vrow + c * 16) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(vrow + kHalf + c * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(&p_full[wg]);
    }
    // epilogue: O / l -> bf16 output row, 32 columns at a time
    if (active && ok && n_tiles > 0) ok = warp_wait(&o_done[wg], static_cast<uint32_t>(n_tiles - 1) & 1u);
    if (!ok && lane == 0) flags[1] = 1;
    tc_fence_after();
    const float inv = (!ok || !(l_run > 0.f)) ? 0.f : 1.f / l_run;
    uint4* orow = reinterpret_cast<uint4*>(
        p.out + (static_cast<size_t>(qs + (row_ok ? tq0 + tok : t0)) * p.H_q + h_kv * p.G + hh) * D);
    if (active) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t ov[32];
        tmem_ld32(tO + 32 * c, ov);
        tmem_wait_ld();
        if (row_ok) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16(__uint_as_float(ov[8 * q4 + 2 * e]) * inv, __uint_as_float(ov[8 * q4 + 2 * e + 1]) * inv);
            orow[4 * c + q4] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
    tc_fence_before();
    __syncthreads();  // (1) every role is done: the flags are final
    if ((flags[0] != 0 || flags[1] != 0) && row_ok) {
#pragma unroll
      for (int c = 0; c < 16; ++c) orow[c] = make_uint4(0, 0, 0, 0);
    }
    if (tid == 64 && flags[1] != 0) set_error(p.err, PA_EFLAG_TIMEOUT);
  }
  if (warp < 2) {
    tc_fence_before();
    __syncthreads();  // (1)
  }
  __syncthreads();  // (2) no TMEM access is pending
  // ------------------------------ teardown ------------------------------
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

// Host launch (declared in pa_internal.h): the tcgen05 path of pa_prefill_attention.
pa_status launch_prefill_tc(const pa_cache_desc* desc, void* out, const void* q, const void* k_cache,
                            const void* v_cache, const int32_t* block_tables, const int32_t* q_start,
                            const int32_t* context_lens, int max_query_len, float scale, int32_t* err_flag,
                            cudaStream_t stream) {
  const long long slots = static_cast<long long>(desc->num_blocks) * PA_BLOCK_SIZE;
  CUtensorMap mk, mv;
  if (!encode_cache_map(&mk, k_cache, 2, desc->num_kv_heads * 2, 1, slots) ||
      !encode_cache_map(&mv, v_cache, 2, desc->num_kv_heads * 2, 1, slots))
    return PA_ERR_CUDA;
  TcParams p;
  p.B = desc->num_seqs;
  p.H_q = desc->num_q_heads;
  p.H_kv = desc->num_kv_heads;
  p.G = desc->num_q_heads / desc->num_kv_heads;
  p.num_blocks = desc->num_blocks;
  p.max_blocks = desc->max_blocks_per_seq;
  p.max_q = max_query_len;
  p.window = desc->sliding_window;
  p.tpq = 128 / p.G;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.q_start = q_start;
  p.context_lens = context_lens;
  p.block_tables = block_tables;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.err = err_flag;
  if (cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem) != cudaSuccess)
    return PA_ERR_CUDA;
  const dim3 grid((max_query_len + 2 * p.tpq - 1) / (2 * p.tpq), p.B, p.H_kv);
  return launch_overlapped(prefill_tc_kernel, grid, dim3(kTcThreads), kTcSmem, stream, mk, mv, p);
}

}  // namespace pa

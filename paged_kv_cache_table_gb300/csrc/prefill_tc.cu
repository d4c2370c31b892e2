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
//    (token, query head), share every K/V tile.  Two such CTAs of the same sequence and KV head
//    form a cluster and load each K/V tile once: every CTA copies half of the tile's boxes with
//    TMA multicast into both CTAs' shared memory.  Measured, one SM ingests only about 15-30
//    bytes per cycle of scattered 2 KB blocks (copy engine or cp.async alike), so halving what
//    each SM fetches per flop is what feeds the tensor core.
//  * S = Q·Kᵀ and O += P·V are tcgen05.mma (kind::f16, bf16 operands, M = N = 128, fp32
//    accumulators in TMEM: S0, S1, O0, O1 in 4 x 128 columns), issued by one thread.  Q and K are
//    K-major and V MN-major shared-memory operands with the 128-byte swizzle; P goes back into
//    TMEM over the S columns it came from (bf16 pairs) and is the A operand of P·V from there, so
//    the tensor core reads only Q, K and V from shared memory, whose bandwidth bounds it here.  A
//    group's next S is issued after its P·V (the tensor pipe runs one thread's products in order,
//    so P is read before it is overwritten); the two groups interleave on the tensor core.
//  * One copy warp streams K through a two-stage ring of 128-key tiles and another V through a
//    three-stage ring: a V tile is needed only at P·V, after the softmax, so V is fetched two tiles
//    ahead, and on its own warp its waits never hold back the next K tile.  A stage is released to the copy warps
//    by a multicast tcgen05.commit from each CTA's MMA thread, so it is refilled only when both
//    CTAs are done with it.
//  * Clusters start longest first.  A cluster's work grows with the last key it reads, which for
//    the c-th cluster of a sequence is first_pos + min(n, (c + 1) W) (W query tokens per cluster):
//    an arithmetic progression per sequence.  So the number of clusters whose last key is at
//    least X has a closed form per sequence, and each cluster finds its own item, the one at its
//    launch position in that order, by a 32-way search over X in one warp; no sort, no scratch.
//  * Two softmax warpgroups (one per query tile) own one query row per thread through TMEM
//    lanes: they read S, mask (causal, window), keep the running maximum (moved only when a score
//    exceeds it by 2^8), write P as bf16 into TMEM, rescale O in TMEM when the maximum moved (O is
//    complete by then: its P·V was issued before this S), and finally normalise O into the output.  V rows of keys that are not loaded
//    or lie beyond the context are zeroed before P·V reads them, so bits left in unused slots (NaN
//    included) cannot leak.
//  * Every wait is bounded; TMEM is released on every path.

#include <algorithm>
#include <cmath>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kTcThreads = 352;                 // 11 warps: K copies, MMA, 2 x 4 softmax, V copies
constexpr int kHalf = 128 * 128;                // 128 rows x 128 bytes (64 bf16): one K-half
constexpr int kTile = 2 * kHalf;                // a 128 x 128 bf16 operand tile
constexpr int kQOff = 0;                        // Q0, Q1
constexpr int kKOff = kQOff + 2 * kTile;        // K stages 0, 1
constexpr int kVOff = kKOff + 2 * kTile;        // V stages 0, 1, 2
constexpr int kVStages = 3;
constexpr int kBarOff = kVOff + kVStages * kTile;
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
// As tc_mma with the A operand in TMEM (M lanes x K/2 columns of bf16 pairs) instead of shared memory.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
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

// 16 bytes global -> shared without registers; `valid` false fills the 16 bytes with zeros.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Query rows of sequence s in clusters of W = 2^lw tokens: fp = first new position, n rows (those
// of an invalid sequence are only zeroed), nc clusters.
struct alignas(16) SeqGeo {
  int fp, n, nc, valid;
};
constexpr int kMaxOrderSeqs = 2 * kTile / static_cast<int>(sizeof(SeqGeo));  // staged in the K ring
__device__ __forceinline__ SeqGeo seq_geo(const TcParams& p, int s, int lw) {
  const int n = p.q_start[s + 1] - p.q_start[s], ctx = p.context_lens[s];
  SeqGeo g;
  g.valid = n >= 0 && n <= ctx && n <= p.max_q && ctx <= p.max_blocks * PA_BLOCK_SIZE;
  g.n = g.valid ? n : min(max(n, 0), p.max_q);
  g.fp = ctx - n;
  g.nc = (g.n + (1 << lw) - 1) >> lw;
  return g;
}
// Clusters of one sequence whose key is >= X (X >= 1).  The key of cluster c, strictly increasing
// in c, is the last key it reads, fp + min(n, (c + 1) W), or c + 1 for an invalid sequence.
__device__ __forceinline__ int count_ge(const SeqGeo& g, int X, int lw) {
  if (!g.valid) return min(g.nc, max(g.nc - (X - 1), 0));
  if (g.nc == 0 || X > g.fp + g.n) return 0;
  const int d = X - g.fp;  // clusters c < nc - 1 with fp + (c + 1) W < X lie below X
  const int below = d <= 0 ? 0 : min(((d + (1 << lw) - 1) >> lw) - 1, g.nc - 1);
  return g.nc - below;
}
// The work item at launch position i when the clusters of all sequences are sorted by key, largest
// first, equal keys by sequence; false past the last one.  geo: every sequence's SeqGeo in shared
// memory.  Called by all lanes of a warp.
__device__ bool cluster_item(const SeqGeo* geo, int B, int key_max, int lw, int i, int lane, int& s_out,
                             int& c_out) {
  int total = 0;
  for (int s = lane; s < B; s += 32) total += count_ge(geo[s], 1, lw);
  total = __reduce_add_sync(0xffffffffu, total);
  if (i >= total) return false;
  // largest key K with count_ge(K) > i: keep count_ge(lo) > i >= count_ge(hi), keys in [1, key_max]
  int lo = 1, hi = key_max + 1;
  while (hi - lo > 1) {
    const int step = (hi - lo + 32) >> 5;  // >= 1; candidates lo + step, lo + 2 step, ... below hi
    const int X = min(lo + step * (lane + 1), hi - 1);
    int cnt = 0;
    for (int s = 0; s < B; ++s) cnt += count_ge(geo[s], X, lw);
    const unsigned pm = __ballot_sync(0xffffffffu, cnt > i);  // X non-decreasing in lane: a prefix
    const int nt = __popc(pm);
    const int x_true = __shfl_sync(0xffffffffu, X, max(nt - 1, 0));
    const int x_false = __shfl_sync(0xffffffffu, X, min(nt, 31));
    if (nt > 0) lo = max(lo, x_true);
    if (nt < 32) hi = min(hi, x_false);
  }
  // the r-th sequence (in order) that has a cluster with key lo
  int above = 0;
  for (int s = lane; s < B; s += 32) above += count_ge(geo[s], lo + 1, lw);
  int r = i - __reduce_add_sync(0xffffffffu, above);
  for (int base = 0; base < B; base += 32) {
    const int s = base + lane;
    int has = 0, c = 0;
    if (s < B) {
      const SeqGeo g = geo[s];
      const int ge = count_ge(g, lo, lw);
      has = ge - count_ge(g, lo + 1, lw);
      c = g.nc - ge;
    }
    const unsigned hm = __ballot_sync(0xffffffffu, has != 0);
    if (r < __popc(hm)) {
      unsigned m = hm;
      for (int k = 0; k < r; ++k) m &= m - 1;  // drop the r lowest set lanes
      const int src = __ffs(m) - 1;
      s_out = base + src;
      c_out = __shfl_sync(0xffffffffu, c, src);
      return true;
    }
    r -= __popc(hm);
  }
  return false;
}

// Both CTAs of the cluster: every thread arrives, then waits for every thread of the cluster.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// TMA box copied into the same shared-memory offset of every CTA in `mask`, each of whose
// mbarrier at `bar`'s offset receives the bytes.
__device__ __forceinline__ void tma_load_3d_mc(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                               int c2, uint16_t mask, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6, %7;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "h"(mask), "l"(policy)
      : "memory");
}
// tcgen05.commit arriving on the mbarrier at `bar`'s offset in every CTA of `mask`.
__device__ __forceinline__ void tc_commit_mc(uint64_t* bar, uint16_t mask) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "h"(mask)
               : "memory");
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
  uint64_t* v_full = bars + 5;   // [3] per V stage
  uint64_t* v_empty = bars + 8;  // [3]
  uint64_t* s_full = bars + 11;  // [2] per query tile
  uint64_t* p_full = bars + 13;  // [2]
  uint64_t* o_done = bars + 15;  // [2]
  uint64_t* drain = bars + 17;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 18);
  int* flags = reinterpret_cast<int*>(bars + 19);  // [0] a bad block id, [1] a wait gave up

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Clusters of two CTAs along x; clusters start in linear order, and the linear cluster index
  // is the launch position: KV heads innermost, work items longest first.
  const int rank = blockIdx.x & 1;
  const int lc = (blockIdx.x >> 1) + (gridDim.x >> 1) * (blockIdx.y + gridDim.y * blockIdx.z);
  const int h_kv = lc % p.H_kv;
  const int tpc = 2 * p.tpq;  // tokens per CTA
  constexpr uint16_t kBoth = 0x3;
  // launched with programmatic dependent launch: the previous kernel may still write any input
  grid_dep_wait();
  int s = 0, ctile = 0;
  {
    const int lw = 31 - __clz(2 * tpc);  // W = 2 tpc = 512 / G query tokens per cluster
    bool have;
    if (p.B <= kMaxOrderSeqs) {
      // the K ring is idle until the cluster barrier below, which no copy into it precedes
      SeqGeo* geo = reinterpret_cast<SeqGeo*>(sm + kKOff);
      int* pick = reinterpret_cast<int*>(sm + kVOff);
      for (int q = tid; q < p.B; q += kTcThreads) geo[q] = seq_geo(p, q, lw);
      __syncthreads();
      if (warp == 0) {  // one warp searches, the others wait
        const int key_max = max(p.max_blocks * PA_BLOCK_SIZE, (p.max_q + (1 << lw) - 1) >> lw);
        const bool h = cluster_item(geo, p.B, key_max, lw, lc / p.H_kv, lane, s, ctile);
        if (lane == 0) {
          pick[0] = h;
          pick[1] = s;
          pick[2] = ctile;
        }
      }
      __syncthreads();
      have = pick[0] != 0;
      s = pick[1];
      ctile = pick[2];
    } else {  // many sequences: last query tiles first, sequences in order
      const int nclx = gridDim.x >> 1, per = lc / p.H_kv;
      ctile = nclx - 1 - per / p.B;
      s = per % p.B;
      have = true;
    }
    if (!have) return;  // past the last item: both CTAs leave
  }
  const int tile = 2 * ctile + rank;
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
  // the whole cluster works or leaves together: both CTAs take part in every tile's copies
  const int tc0 = 2 * ctile * tpc;  // first token of the cluster
  if (tc0 >= n) return;
  const int t0 = tile * tpc;
  const bool has0 = t0 < n, has1 = t0 + p.tpq < n;  // this CTA's query tiles that hold tokens
  const int first_pos = ctx - n;
  const int t_end = min(n, t0 + tpc);
  // keys [kv_lo, kv_end) are visible to some row of the cluster
  const int kv_end = first_pos + min(n, tc0 + 2 * tpc);
  const int kv_lo = p.window > 0 ? max(0, first_pos + tc0 - p.window + 1) : 0;
  const int kb0 = kv_lo / PA_BLOCK_SIZE;
  const int kb_end = (kv_end + PA_BLOCK_SIZE - 1) / PA_BLOCK_SIZE;
  const int n_tiles = (kb_end - kb0 + 7) / 8;
  const int loaded_end = min(ctx, kb_end * PA_BLOCK_SIZE);  // keys past this hold no loaded data

  if (tid == 0) {
    mbar_init(q_full, 256);
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 2);  // released by the MMA threads of both CTAs
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 2);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&o_done[i], 1);
    }
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
  cluster_sync();  // the peer's barriers exist before any multicast reaches them
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 || warp == 10) {
    // ---------------------- copy warps: K (warp 0), V (warp 10) ----------------------
    const int32_t* row = p.block_tables + static_cast<size_t>(s) * p.max_blocks;
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(policy));
    // Table entries live in registers, 32 consecutive blocks per chunk and one per lane, for
    // chunks c0, c0 + 1 and c0 + 2: the accesses only move forward, so a chunk is loaded two
    // chunks before it is first needed and its latency is hidden.
    auto entry = [&](int c) { const int kb = kb0 + 32 * c + lane; return kb < kb_end ? row[kb] : -1; };
    int c0 = 0, e0 = entry(0), e1 = entry(1), e2 = entry(2);
    auto table = [&](int b) -> int {  // entry of block kb0 + b; b is in the same chunk on every lane
      const int cb = __shfl_sync(0xffffffffu, b, 0) >> 5;
      while (cb > c0 + 1) {
        e0 = e1;
        e1 = e2;
        e2 = entry(c0 + 3);
        ++c0;
      }
      const int v0 = __shfl_sync(0xffffffffu, e0, b & 31), v1 = __shfl_sync(0xffffffffu, e1, b & 31);
      return cb == c0 ? v0 : v1;
    };
    // nblk blocks from tile-relative block blk0, boxes of 16 slots x 128 bytes, one per lane:
    // block lane / 2, 64-dim half lane % 2.  Both CTAs count every box of the tile; each copies
    // the half of the blocks that its rank owns, to both.  Returns false when a wait gave up.
    auto load = [&](int nblk, int blk0, const CUtensorMap* map, uint64_t* full, uint64_t* empty, uint32_t parity,
                    uint8_t* dst, int half_bytes) -> bool {
      if (!warp_wait(empty, parity)) return false;
      const int bi = lane >> 1, half = lane & 1;
      const int kb = kb0 + blk0 + bi;
      const int ent = table(blk0 + min(bi, nblk - 1));
      int pb = -1;
      if (bi < nblk && kb < kb_end) {
        pb = ent;
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
      if (pb >= 0 && bi * 2 / nblk == rank)
        tma_load_3d_mc(dst + half * half_bytes + bi * 2048, map, full, 0, h_kv * 2 + half, pb * PA_BLOCK_SIZE, kBoth,
                       policy);
      return true;
    };
    bool ok = true;
    for (int k = 0; ok && k < n_tiles; ++k) {
      if (warp == 0) {
        ok = load(8, 8 * k, &tmK, &k_full[k & 1], &k_empty[k & 1], (static_cast<uint32_t>(k >> 1) & 1u) ^ 1u,
                  sm + kKOff + (k & 1) * kTile, kHalf);
      } else {
        const int st = k % kVStages;
        ok = load(8, 8 * k, &tmV, &v_full[st], &v_empty[st], (static_cast<uint32_t>(k / kVStages) & 1u) ^ 1u,
                  sm + kVOff + st * kTile, kHalf);
      }
    }
    if (!ok && lane == 0) flags[1] = 1;
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
        const uint32_t vbuf = smem_u32(sm + kVOff + (k % kVStages) * kTile);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          // P: keys 16kk .. 16kk+15 = TMEM columns 8kk .. 8kk+7 of S_w; V: key rows 16kk .. of both halves
          tc_mma_ts(tmem + 256 + w * 128, tmem + w * 128 + 8 * kk, sw128_desc(vbuf + kk * 16 * 128, kHalf, 1024),
                    kIdescPV, (k > 0 || kk > 0) ? 1u : 0u);
        }
      };
      // groups of this CTA with rows (a CTA without any still joins every copy and release)
      const int groups = has1 ? 2 : (has0 ? 1 : 0);
      // A stage is released (in both CTAs) only when a later copy waits for it: every such
      // arrival is consumed before either CTA can finish, so none lands in a CTA that has left.
      // The K stage of tile m is refilled with tile m + 2; the V stage of tile k with tile k + 3.
      bool ok = mbar_wait(q_full, 0) && mbar_wait(&k_full[0], 0);
      if (ok) {
        tc_fence_after();
        for (int w = 0; w < groups; ++w) issue_s(w, 0);
        if (n_tiles > 2) tc_commit_mc(&k_empty[0], kBoth);
      }
      for (int k = 0; ok && k < n_tiles; ++k) {
        const uint32_t ph = static_cast<uint32_t>(k) & 1u;
        const bool next = k + 1 < n_tiles;
        if (next && !(ok = mbar_wait(&k_full[(k + 1) & 1], static_cast<uint32_t>((k + 1) >> 1) & 1u))) break;
        const int vs = k % kVStages;
        if (!(ok = mbar_wait(&v_full[vs], static_cast<uint32_t>(k / kVStages) & 1u))) break;
        // per group: P·V of this tile, then the group's S of the next tile
        for (int w = 0; ok && w < groups; ++w) {
          if (!(ok = mbar_wait(&p_full[w], ph))) break;
          tc_fence_after();
          issue_pv(w, k);
          tc_commit(&o_done[w]);
          if (next) issue_s(w, k + 1);
        }
        if (!ok) break;
        if (k + kVStages < n_tiles) tc_commit_mc(&v_empty[vs], kBoth);
        if (k + 3 < n_tiles) tc_commit_mc(&k_empty[(k + 1) & 1], kBoth);
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
    {  // this warp's 32 Q rows -> swizzled Q tile; two 256-byte rows per instruction, so that
       // the lanes of a row read it whole (16 bytes each) and the loads coalesce
      const int c = lane & 15;
#pragma unroll 4
      for (int i = 0; i < 16; ++i) {
        const int rr = quad * 32 + 2 * i + (lane >> 4);
        const int tk = rr / p.G;
        const bool ok_r = tq0 + tk < t_end;
        const __nv_bfloat16* src =
            ok_r ? p.q + (static_cast<size_t>(qs + tq0 + tk) * p.H_q + h_kv * p.G + (rr - tk * p.G)) * D + c * 8 : p.q;
        cp_async16(qtile + (c >> 3) * kHalf + rr * 128 + (((c & 7) ^ (rr & 7)) << 4), src, ok_r);
      }
      cp_async_wait_all();
      fence_proxy_async();
      mbar_arrive(q_full);
    }
    const bool active = wg == 0 ? has0 : has1;
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
      float mx8[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) mx8[j] = kNegInfTc;
#pragma unroll
      for (int c = 0; c < 128; c += 2)
        mx8[(c >> 1) & 7] = max3f(mx8[(c >> 1) & 7], __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]));
      const float mraw = fmaxf(max3f(mx8[0], mx8[1], mx8[2]), max3f(max3f(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
      const float mx = mraw == kNegInfTc ? kNegInfTc : mraw * p.scale_log2;
      const float m_new = (m_run == kNegInfTc || mx > m_run + 8.f) ? fmaxf(m_run, mx) : m_run;
      const float ms = m_new == kNegInfTc ? 0.f : m_new;
      const float alpha = ex2(m_run - ms);
      // P (bf16 pairs) over the S columns just read: column c holds keys 2c and 2c + 1
      float ls4[4] = {0.f, 0.f, 0.f, 0.f};
      const float sl = p.scale_log2;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pw[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float a = ex2(fmaf(__uint_as_float(sv[64 * h + 2 * e]), sl, -ms));
          const float b = ex2(fmaf(__uint_as_float(sv[64 * h + 2 * e + 1]), sl, -ms));
          ls4[e & 3] += a + b;
          pw[e] = pack_bf16(a, b);
        }
        tmem_st32(tS + 32 * h, pw);
      }
      tmem_wait_st();
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
      const int vs = k % kVStages;
      if (__any_sync(0xffffffffu, zero_row)) {
        // the stage's copies must have landed first
        if (!warp_wait(&v_full[vs], static_cast<uint32_t>(k / kVStages) & 1u)) {
          ok = false;
          break;
        }
        if (zero_row) {
          uint8_t* vrow = sm + kVOff + vs * kTile + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            *reinterpret_cast<uint4*>(vrow + c * 16) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(vrow + kHalf + c * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async();  // the zeros, before the tensor core reads the stage
      }
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
    if (active && ok) {
      // Every product has completed (o_done of the last tile follows them all), so the Q tile is
      // idle: the warp stages its 32 rows there as bf16 (16-byte chunk j of row i at j ^ (i & 15),
      // conflict-free both ways) and stores them two rows per instruction, coalesced.
      uint8_t* stage = qtile + quad * 32 * 256;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t ov[32];
        tmem_ld32(tO + 32 * c, ov);
        tmem_wait_ld();
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = pack_bf16(__uint_as_float(ov[8 * q4 + 2 * e]) * inv, __uint_as_float(ov[8 * q4 + 2 * e + 1]) * inv);
          *reinterpret_cast<uint4*>(stage + lane * 256 + (((4 * c + q4) ^ (lane & 15)) << 4)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      __syncwarp();
      const int c = lane & 15;
#pragma unroll 4
      for (int i = 0; i < 16; ++i) {
        const int ri = 2 * i + (lane >> 4);
        const int rr = quad * 32 + ri;
        const int tk = rr / p.G;
        if (tq0 + tk < t_end)
          reinterpret_cast<uint4*>(p.out + (static_cast<size_t>(qs + tq0 + tk) * p.H_q + h_kv * p.G + (rr - tk * p.G)) *
                                               D)[c] = *reinterpret_cast<const uint4*>(stage + ri * 256 + ((c ^ (ri & 15)) << 4));
      }
    } else if (active && row_ok) {
#pragma unroll
      for (int c = 0; c < 16; ++c) orow[c] = make_uint4(0, 0, 0, 0);
    }
    tc_fence_before();
    __syncthreads();  // (1) every role is done: the flags are final
    if ((flags[0] != 0 || flags[1] != 0) && row_ok) {
#pragma unroll
      for (int c = 0; c < 16; ++c) orow[c] = make_uint4(0, 0, 0, 0);
    }
    if (tid == 64 && flags[1] != 0) set_error(p.err, PA_EFLAG_TIMEOUT);
  }
  if (warp < 2 || warp == 10) {
    tc_fence_before();
    __syncthreads();  // (1)
  }
  __syncthreads();  // (2) no TMEM access is pending
  // neither CTA leaves while the other may still copy into its shared memory or release a stage
  cluster_sync();
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
  const int ctas_x = (max_query_len + 2 * p.tpq - 1) / (2 * p.tpq);
  const dim3 grid(2 * ((ctas_x + 1) / 2), p.B, p.H_kv);  // whole clusters of two along x
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = kTcSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, prefill_tc_kernel, mk, mv, p) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa

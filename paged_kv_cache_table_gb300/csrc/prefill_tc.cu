// Chunked-prefill attention on the fifth-generation tensor cores (tcgen05, TMEM).
//
// What is computed is the same as the warp-MMA kernel in prefill_attention.cu: untitled KV-cache
// article at ldpk.cn/news/58971 §2.2 (causal attention of every new position over the positions up
// to itself) and §7 (chunked prefill), over the paged cache through the block table ("KV Cache 的显存
// 账本：PagedAttention 与连续批处理" §四), GQA grouping (same page §二), and an optional sliding
// window (ldpk §5.3).
//
// Design (head_dim 128, G = 1, 2, 4 or 8 query heads per KV head):
//  * Work items.  An item is (sequence, tile c, KV head): the query rows of two query tiles of
//    128 rows, a row being (token, query head), i.e. 256 / G query tokens, held by one CTA.  Both
//    query tiles share every K/V tile the CTA loads, so each 32 KiB K or V tile feeds four
//    128 x 128 x 128 products.  Each CTA loads its own tiles from its own GPU's pool with plain
//    TMA boxes; the CTAs that read the same keys (the tiles of one sequence) meet in L2.
//  * Persistent CTAs, longest first.  The grid is as many CTAs as can be resident, each walking
//    its own list of items.  An item's work grows with the last key it reads, which for the c-th
//    tile of a sequence is first_pos + min(n, (c + 1) W) (W query tokens per tile): an
//    arithmetic progression per sequence.  So the number of items whose last key is at least X
//    has a closed form per sequence, every item's rank in the longest-first order is a sum over
//    sequences, and the CTAs rank all items in parallel at start-up (no sort, no scratch
//    memory), dealing the ranks to CTAs round by round, alternately in order and in reverse.
//    Barriers, TMEM and the ring phases carry across items.
//  * S = Q·Kᵀ and O += P·V are tcgen05.mma (kind::f16, bf16 operands, M = N = 128, fp32
//    accumulators in TMEM: S0, S1, O0, O1 in 4 x 128 columns), issued by one thread.  Q and K are
//    K-major and V MN-major shared-memory operands with the 128-byte swizzle; P goes back into
//    TMEM over the S columns it came from (bf16 pairs) and is the A operand of P·V from there, so
//    the tensor core reads only Q, K and V from shared memory.  P·V is issued once the softmax
//    has written all of P (p_full): the issuing thread's waits, not the products, set the pace of
//    the tile loop (~100-150 cycles per barrier wait; measured, handing over the first 64 keys'
//    P early cost more in waits than its overlap gained).  A query tile's next S is issued after
//    its P·V (the tensor pipe runs one thread's products in order, so P is read before it is
//    overwritten); the two query tiles interleave on the tensor core.
//  * Copies: two warps, one per 64-dim half, stream K through a three-stage ring of 128-key tiles
//    and V through a two-stage ring, 8 boxes of 16 slots per warp and tile (a warp issues its
//    boxes one by one, ~80 cycles each).  A tile's copy takes ~3,500-4,000 cycles from the
//    release of its stage to its landing, about one tile's time, so K runs one tile ahead of V
//    (K of tile g + 1 and V of tile g are needed together, when the MMA thread starts tile g) and
//    K's ring is the deeper one.  A third warp loads the next item's query tiles by TMA (a 4-D
//    map over q) as soon as the current item's last S products have completed.  A ring stage is
//    released to the copy warps by a tcgen05.commit of the MMA thread once every product reading
//    it has completed.
//  * Two softmax warpgroups (one per query tile) own one query row per thread through TMEM
//    lanes: they read S, mask (causal, window) only on tiles that cross a row's edge, keep the
//    running maximum (moved only when a score exceeds it by 2^8), write P as bf16 into TMEM, and
//    when the maximum moved rescale O in TMEM before handing any of P over (O is complete by
//    then: its P·V was issued before this S).  V rows of keys that are not loaded or lie beyond
//    the context are zeroed before P·V reads them, so bits left in unused slots (NaN included)
//    cannot leak.
//  * Output: O / l as bf16 is staged in the idle ring stage of the item's last tile (K for query
//    tile 0, V for query tile 1) and stored by TMA; the stage is then released to its copy warp.
//    Only a tile holding rows past its sequence is stored row by row.
//  * Launched with programmatic dependent launch.  In a prefill step (pa_prefill_step) the
//    previous kernel is the chunk's append, which writes only K/V slots, so only the K/V copy
//    warps wait for it; the work ranking and the query copies run alongside it.
//  * Every wait is bounded; TMEM is released on every path, and no warp leaves while a copy it
//    issued into this CTA's shared memory may still be in flight.

#include <algorithm>
#include <cmath>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kTcThreads = 384;                 // 12 warps: K/V copies, MMA, K/V copies, Q copies; 2 x 4 softmax
constexpr int kHalf = 128 * 128;                // 128 rows x 128 bytes (64 bf16): one K-half
constexpr int kTile = 2 * kHalf;                // a 128 x 128 bf16 operand tile
constexpr int kQOff = 0;                        // Q0, Q1
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kKOff = kQOff + 2 * kTile;               // K stages
constexpr int kVOff = kKOff + kKStages * kTile;        // V stages
constexpr int kBarOff = kVOff + kVStages * kTile;
constexpr int kMaxItems = 64;                   // work items of one CTA (the launch makes enough CTAs)
constexpr int kListOff = kBarOff + 256;         // barriers, then the CTA's item list
constexpr int kTcSmem = kListOff + kMaxItems * 24 + 1024;  // and slack for 1024-byte alignment
constexpr int kQMapTokens = 1 << 24;            // token extent of the Q tensor map (rows past it: plain copies)
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
  int step;  // the previous kernel is this step's append: only the K/V copies wait for it
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
// 16 consecutive fp32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]) : "memory");
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

// A 4-D TMA box into this CTA's shared memory, completion counted on `bar`.
__device__ __forceinline__ void tma_load_4d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2,
                                            int c3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// A 4-D TMA box from this CTA's shared memory to global memory (bulk async group of this thread).
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, const void* smem_src, int c0, int c1, int c2, int c3) {
  asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(smem_src))
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// This thread's bulk stores have read their shared memory (reads) or completed (all).
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void group_sync(int id) { asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory"); }

// Query rows of sequence s in tiles of W = 2^lw tokens: fp = first new position, n rows (those
// of an invalid sequence are only zeroed), nc tiles.
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
// Tiles of one sequence whose key is >= X (X >= 1).  The key of tile c, strictly increasing in c,
// is the last key it reads, fp + min(n, (c + 1) W), or c + 1 for an invalid sequence.
__device__ __forceinline__ int count_ge(const SeqGeo& g, int X, int lw) {
  if (!g.valid) return min(g.nc, max(g.nc - (X - 1), 0));
  if (g.nc == 0 || X > g.fp + g.n) return 0;
  const int d = X - g.fp;  // tiles c < nc - 1 with fp + (c + 1) W < X lie below X
  const int below = d <= 0 ? 0 : min(((d + (1 << lw) - 1) >> lw) - 1, g.nc - 1);
  return g.nc - below;
}
// One work item of a CTA: the query rows of tile c of sequence s (tokens [t0, t_end) with
// t0 = c tpc, tpc = 2 tpq tokens per tile) against KV head h_kv, in two query tiles of tpq tokens;
// the CTA reads the keys [kv_lo, kv_end), blocks [kb0, kb_end), in n_tiles tiles of 8 blocks.
struct Item {
  int s, h_kv, tile, qs, n, t0, t_end, first_pos, kv_lo, kb0, kb_end, n_tiles, loaded_end;
  bool valid, has0, has1;
};
// An entry of a CTA's item list (shared memory): the sequence, the tile and KV head
// (c << 16 | h), and the sequence's first query row, query rows and context length.
struct ItemRec {
  int s, ch, qs, n, ctx, pad;
};
__device__ __forceinline__ ItemRec item_rec(const TcParams& p, int s, int c, int h) {
  ItemRec e;
  e.s = s;
  e.ch = (c << 16) | h;
  e.qs = p.q_start[s];
  e.n = p.q_start[s + 1] - e.qs;
  e.ctx = p.context_lens[s];
  e.pad = 0;
  return e;
}
__device__ __forceinline__ Item make_item(const TcParams& p, const ItemRec& e) {
  Item it;
  it.s = e.s;
  it.tile = e.ch >> 16;
  it.h_kv = e.ch & 0xFFFF;
  const int tpc = 2 * p.tpq;
  it.qs = e.qs;
  it.n = e.n;
  const int ctx = e.ctx;
  it.valid = it.n >= 0 && it.n <= ctx && it.n <= p.max_q && ctx <= p.max_blocks * PA_BLOCK_SIZE;
  it.t0 = it.tile * tpc;
  it.has0 = it.valid && it.t0 < it.n;
  it.has1 = it.valid && it.t0 + p.tpq < it.n;
  it.first_pos = ctx - it.n;
  it.t_end = min(it.n, it.t0 + tpc);
  it.kv_lo = it.kb0 = it.kb_end = it.n_tiles = it.loaded_end = 0;
  if (it.has0) {
    const int kv_end = it.first_pos + it.t_end;
    it.kv_lo = p.window > 0 ? max(0, it.first_pos + it.t0 - p.window + 1) : 0;
    it.kb0 = it.kv_lo / PA_BLOCK_SIZE;
    it.kb_end = (kv_end + PA_BLOCK_SIZE - 1) / PA_BLOCK_SIZE;
    it.n_tiles = (it.kb_end - it.kb0 + 7) / 8;
    it.loaded_end = min(ctx, it.kb_end * PA_BLOCK_SIZE);  // keys past this hold no loaded data
  }
  return it;
}

// Launch position pos of round r of a CTA: rounds deal NC positions each, alternately in CTA
// order and in reverse, so that the longest items of one round and the shortest of the next land
// on the same CTA.
__device__ __forceinline__ int round_pos(int r, int NC, int cid) { return r * NC + ((r & 1) ? NC - 1 - cid : cid); }

__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmO,
                      const TcParams p) {
  constexpr int D = 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBarOff);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 2;
  uint64_t* k_full = bars + 4;   // [kKStages] per K stage
  uint64_t* k_empty = bars + 4 + kKStages;
  uint64_t* v_full = bars + 4 + 2 * kKStages;  // [kVStages] per V stage
  uint64_t* v_empty = bars + 4 + 2 * kKStages + kVStages;
  uint64_t* s_full = bars + 14;  // [2] per query tile
  uint64_t* p_full = bars + 16;  // [2]
  uint64_t* o_done = bars + 18;  // [2]
  uint64_t* drain = bars + 20;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 21);
  int* flags = reinterpret_cast<int*>(bars + 22);  // [0] tiles of all sequences, [1] a wait gave up
  ItemRec* list = reinterpret_cast<ItemRec*>(sm + kListOff);  // this CTA's items, in order

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cid = blockIdx.x, NC = gridDim.x;
  const int tpc = 2 * p.tpq;                 // W = tpc = 256 / G query tokens per tile (a power of two)
  const int lw = 31 - __clz(tpc);
  const int nclx = (p.max_q + (1 << lw) - 1) >> lw;
  const bool lpt = p.B <= kMaxOrderSeqs;
  SeqGeo* geo = reinterpret_cast<SeqGeo*>(sm + kKOff);  // scratch: the K ring is idle until the items are listed

  if (tid == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&v_full[i], 2);  // one arrival per copy warp
      mbar_init(&v_empty[i], 1);  // released by the MMA thread (or the output's store)
    }
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&k_full[i], 2);  // one arrival per copy warp
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
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
  // Launched with programmatic dependent launch: the previous kernel may still write any input,
  // so everything waits for it here.  In a prefill step the previous kernel is the append of the
  // chunk, which writes only K/V slots; then only the K/V copy warps wait (before their first
  // copy, in every CTA, so that this grid never completes before the append), and the set-up
  // and the query copies overlap the append.
  if (!p.step) grid_dep_wait();
  if (lpt)
    for (int q = tid; q < p.B; q += kTcThreads) geo[q] = seq_geo(p, q, lw);
  tc_fence_before();
  __syncthreads();
  if (lpt) {
    int part = 0;
    for (int q = tid; q < p.B; q += kTcThreads) part += geo[q].nc;
    part = __reduce_add_sync(0xffffffffu, part);
    if (lane == 0 && part) atomicAdd(&flags[0], part);
  }
  __syncthreads();
  // Work items longest first: item (s, c) of key k sits at rank = #items of larger key + #items of
  // key k in earlier sequences; with KV heads innermost, launch position = rank * H_kv + h.
  // Many sequences: last tiles first, sequences in order (slots past a sequence are empty).
  const int p_tot = lpt ? flags[0] * p.H_kv : p.B * nclx * p.H_kv;
  const int rounds = (p_tot + NC - 1) / NC;
  const int n_items = min(kMaxItems, rounds == 0 ? 0 : rounds - 1 + (round_pos(rounds - 1, NC, cid) < p_tot ? 1 : 0));
  if (lpt) {
    for (int j = tid; j < p.B * nclx; j += kTcThreads) {
      const int s = j / nclx, c = j - s * nclx;
      const SeqGeo g = geo[s];
      if (c >= g.nc) continue;
      const int key = g.valid ? g.fp + min(g.n, (c + 1) << lw) : c + 1;
      int rk = 0;
      for (int q = 0; q < p.B; ++q) {
        const SeqGeo gq = geo[q];
        const int above = count_ge(gq, key + 1, lw);
        rk += above + (q < s ? count_ge(gq, key, lw) - above : 0);
      }
      for (int h = 0; h < p.H_kv; ++h) {
        const int pos = rk * p.H_kv + h, r = pos / NC, w = pos - r * NC;
        if (((r & 1) ? NC - 1 - w : w) == cid && r < kMaxItems) list[r] = item_rec(p, s, c, h);
      }
    }
  } else {
    for (int r = tid; r < n_items; r += kTcThreads) {
      const int pos = round_pos(r, NC, cid), slot = pos / p.H_kv, h = pos - slot * p.H_kv;
      list[r] = item_rec(p, slot % p.B, nclx - 1 - slot / p.B, h);
    }
  }
  __syncthreads();  // the list is complete and the K ring is free again
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 || warp == 2) {
    // ------------------- K/V copies: warp 0 dims 0-63, warp 2 dims 64-127 -------------------
    if (p.step) grid_dep_wait();
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(policy));
    bool ok = true;
    const int half = warp >> 1;
    // tiles of this CTA whose K (gk) and V (gv) copies have been issued: ring stages and phases.
    // K runs one tile ahead of V: K of tile g + 1 and V of tile g are needed together (at the
    // start of the MMA thread's tile g), and K's ring is the deeper one.
    int gk = 0, gv = 0;
    int v_pb = -1, v_h = 0;  // the tile whose V copy is still to be issued: its block, KV head
    unsigned v_loads = 0;
    // The 8 blocks of this warp's 64-dim half of a tile, boxes of 16 slots x 128 bytes, one per
    // lane (lanes 0-7).
    auto issue = [&](const CUtensorMap* map, uint64_t* full, uint64_t* empty, uint32_t parity, uint8_t* dst,
                     int pb, unsigned loads, int h_kv) -> bool {
      if (!warp_wait(empty, parity)) return false;
      if (lane == 0) {
        const uint32_t bytes = __popc(loads) * 2048u;
        if (bytes) mbar_arrive_expect_tx(full, bytes);
        else mbar_arrive(full);
      }
      __syncwarp();
      if (pb >= 0)
        tma_load_3d(dst + half * kHalf + lane * 2048, map, full, 0, h_kv * 2 + half, pb * PA_BLOCK_SIZE, policy);
      return true;
    };
    auto issue_v = [&]() -> bool {  // V of tile gv (its blocks in v_pb)
      const int vst = gv % kVStages;
      const bool r = issue(&tmV, &v_full[vst], &v_empty[vst], (static_cast<uint32_t>(gv / kVStages) & 1u) ^ 1u,
                           sm + kVOff + vst * kTile, v_pb, v_loads, v_h);
      if (r) ++gv;
      return r;
    };
    for (int ii = 0; ok && ii < n_items; ++ii) {
      const Item it = make_item(p, list[ii]);
      if (it.n_tiles == 0) continue;
      const int32_t* row = p.block_tables + static_cast<size_t>(it.s) * p.max_blocks;
      const int kb0 = it.kb0, kb_end = it.kb_end;
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
      for (int k = 0; ok && k < it.n_tiles; ++k) {
        const int kb = kb0 + 8 * k + lane;
        const int ent = table(8 * k + min(lane, 7));
        int pb = -1;
        if (lane < 8 && kb < kb_end) {
          pb = ent;
          if (pb < 0 || pb >= p.num_blocks) {
            if (half == 0) set_error(p.err, PA_EFLAG_BAD_BLOCK_ID);
            pb = -1;
          }
        }
        const unsigned loads = __ballot_sync(0xffffffffu, pb >= 0);
        const int kst = gk % kKStages;
        ok = issue(&tmK, &k_full[kst], &k_empty[kst], (static_cast<uint32_t>(gk / kKStages) & 1u) ^ 1u,
                   sm + kKOff + kst * kTile, pb, loads, it.h_kv);
        if (!ok) break;
        ++gk;
        if (gv < gk - 1) ok = issue_v();
        v_pb = pb;
        v_loads = loads;
        v_h = it.h_kv;
      }
    }
    if (ok && gv < gk) ok = issue_v();
    // do not leave while a copy into this CTA's shared memory may still be in flight (the MMA
    // thread waits for every tile, unless one of its own waits gave up)
    for (int st = 0; st < kKStages && st < gk; ++st) {
      const int last = st + kKStages * ((gk - 1 - st) / kKStages);
      if (!warp_wait(&k_full[st], static_cast<uint32_t>(last / kKStages) & 1u)) ok = false;
    }
    for (int st = 0; st < kVStages && st < gv; ++st) {
      const int last = st + kVStages * ((gv - 1 - st) / kVStages);
      if (!warp_wait(&v_full[st], static_cast<uint32_t>(last / kVStages) & 1u)) ok = false;
    }
    if (!ok && lane == 0) flags[1] = 1;
  } else if (warp == 3) {
    // ------------------- Q copies: each item's two query tiles -------------------
    // The tiles of the next item are copied as soon as every product of the current one that
    // reads them has completed (q_empty), while its last tiles and output are still under way.
    // A tile is one TMA box per 64-dim half (tpq tokens x G heads x 128 bytes, landing as the
    // swizzled K-major operand); rows past the sequence are other sequences' queries, masked
    // later.  Only a box that would reach past the last query row q_start[B] (which the caller
    // need not have allocated) is copied row by row instead, zero-filled.
    const uint64_t policy = l2_evict_first_policy();
    const int q_rows = min(p.q_start[p.B], kQMapTokens);
    bool ok = true;
    int qi = 0;
    const int c = lane & 15;
    for (int ii = 0; ok && ii < n_items; ++ii) {
      const Item it = make_item(p, list[ii]);
      if (it.n_tiles == 0) continue;
      if (!(ok = warp_wait(q_empty, (static_cast<uint32_t>(qi) & 1u) ^ 1u))) break;
      ++qi;
      uint32_t boxes = 0;  // tiles copied by TMA
      for (int w = 0; w < 2; ++w) {
        const int tq0 = it.t0 + w * p.tpq;
        if (tq0 >= it.t_end) continue;  // no rows: its products are not issued
        if (it.qs + tq0 + p.tpq <= q_rows) {
          boxes |= 1u << w;
          continue;
        }
        uint8_t* qtile = sm + kQOff + w * kTile;
#pragma unroll 4
        for (int i = 0; i < 64; ++i) {  // two 256-byte rows per instruction, 16 bytes per lane
          const int rr = 2 * i + (lane >> 4);
          const int tk = rr / p.G;
          const bool ok_r = tq0 + tk < it.t_end;
          const __nv_bfloat16* src =
              ok_r ? p.q + (static_cast<size_t>(it.qs + tq0 + tk) * p.H_q + it.h_kv * p.G + (rr - tk * p.G)) * D + c * 8
                   : p.q;
          cp_async16(qtile + (c >> 3) * kHalf + rr * 128 + (((c & 7) ^ (rr & 7)) << 4), src, ok_r);
        }
      }
      cp_async_wait_all();
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        if (boxes) {
          mbar_arrive_expect_tx(q_full, __popc(boxes) * static_cast<uint32_t>(kTile));
          for (int w = 0; w < 2; ++w)
            if (boxes >> w & 1u)
              for (int half = 0; half < 2; ++half)
                tma_load_4d(sm + kQOff + w * kTile + half * kHalf, &tmQ, q_full, 0, half, it.h_kv * p.G,
                            it.qs + it.t0 + w * p.tpq, policy);
        } else {
          mbar_arrive(q_full);
        }
      }
    }
    // the last query copies have landed before the warp leaves
    if (qi > 0 && !warp_wait(q_full, static_cast<uint32_t>(qi - 1) & 1u)) ok = false;
    if (!ok && lane == 0) flags[1] = 1;
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      auto issue_s = [&](int w, int kst) {  // S_w = Q_w K^T of the tile in K stage kst
        const uint32_t qb = smem_u32(sm + kQOff + w * kTile);
        const uint32_t kbuf = smem_u32(sm + kKOff + kst * kTile);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          tc_mma(tmem + w * 128, sw128_desc(qb + off, 16, 1024), sw128_desc(kbuf + off, 16, 1024), kIdescS, kk > 0);
        }
        tc_commit(&s_full[w]);
      };
      // O_w (+)= P_w V of the tile in V stage vst
      auto issue_pv = [&](int w, int vst, bool first) {
        const uint32_t vbuf = smem_u32(sm + kVOff + vst * kTile);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          // P: keys 16kk .. 16kk+15 = TMEM columns 8kk .. 8kk+7 of S_w; V: key rows 16kk .. of both halves
          tc_mma_ts(tmem + 256 + w * 128, tmem + w * 128 + 8 * kk, sw128_desc(vbuf + kk * 16 * 128, kHalf, 1024),
                    kIdescPV, (!first || kk > 0) ? 1u : 0u);
        }
      };
      // A ring stage is released only when a later copy waits for it.  The K stage of tile m is
      // refilled with tile m + kKStages, the V stage of tile m with tile m + kVStages, counting
      // the tiles of all the CTA's items in order.  The K and V stages of an item's last tile
      // stage the output of query tiles 0 and 1 when those hold rows, and their groups release
      // them after it has left; otherwise they are released here.
      int g_tot = 0;
      for (int ii = 0; ii < n_items; ++ii) g_tot += make_item(p, list[ii]).n_tiles;
      bool ok = true;
      int g = 0, qi = 0;
      uint32_t sp[2] = {0u, 0u};  // tiles of each query tile so far: s_full / p_full / o_done phase
      for (int ii = 0; ok && ii < n_items; ++ii) {
        const Item it = make_item(p, list[ii]);
        const int nt = it.n_tiles;
        if (nt == 0) continue;
        const int groups = it.has1 ? 2 : 1;  // query tiles with rows (an item with tiles has rows)
        ok = mbar_wait(q_full, static_cast<uint32_t>(qi) & 1u) &&
             mbar_wait(&k_full[g % kKStages], static_cast<uint32_t>(g / kKStages) & 1u);
        ++qi;
        if (!ok) break;
        tc_fence_after();
        for (int w = 0; w < groups; ++w) issue_s(w, g % kKStages);
        if (nt == 1) tc_commit(q_empty);  // the item's last products that read Q are issued
        if (g + kKStages < g_tot && nt > 1) tc_commit(&k_empty[g % kKStages]);
        for (int k = 0; k < nt; ++k) {
          const int gk = g + k;
          const bool next = k + 1 < nt;
          if (next && !(ok = mbar_wait(&k_full[(gk + 1) % kKStages], static_cast<uint32_t>((gk + 1) / kKStages) & 1u)))
            break;
          const int vs = gk % kVStages;
          if (!(ok = mbar_wait(&v_full[vs], static_cast<uint32_t>(gk / kVStages) & 1u))) break;
          // per query tile: P·V of this tile once its P is written, then its S of the next tile
          for (int w = 0; ok && w < groups; ++w) {
            if (!(ok = mbar_wait(&p_full[w], sp[w] & 1u))) break;
            ++sp[w];
            tc_fence_after();
            issue_pv(w, vs, k == 0);
            tc_commit(&o_done[w]);
            if (next) issue_s(w, (gk + 1) % kKStages);
          }
          if (!ok) break;
          if (k == nt - 2) tc_commit(q_empty);
          if (gk + kVStages < g_tot && (next || groups < 2)) tc_commit(&v_empty[vs]);
          if (next && gk + 1 + kKStages < g_tot && k + 2 < nt) tc_commit(&k_empty[(gk + 1) % kKStages]);
        }
        g += nt;
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
    const int wg = (warp - 4) >> 2;  // query tile of this group
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // this thread's row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + wg * 128 + lane_off, tO = tmem + 256 + wg * 128 + lane_off;
    const int tok = r / p.G, hh = r - tok * p.G;
    bool ok = true;
    int g = 0;        // tiles of this CTA so far (V stage and phase)
    uint32_t sp = 0;  // tiles of this query tile so far
    int g_tot = 0;    // tiles of all the CTA's items (whether a later copy waits for a stage)
    for (int ii = 0; ii < n_items; ++ii) g_tot += make_item(p, list[ii]).n_tiles;
    for (int ii = 0; ii < n_items; ++ii) {
      const Item it = make_item(p, list[ii]);
      const int tq0 = it.t0 + wg * p.tpq;  // first token of this query tile
      uint4* orow = reinterpret_cast<uint4*>(
          p.out + (static_cast<size_t>(it.qs + tq0 + tok) * p.H_q + it.h_kv * p.G + hh) * D);
      if (!it.valid) {  // zero rows, within the rows the caller declared
        if (it.tile == 0 && it.h_kv == 0 && wg == 0 && r == 0) set_error(p.err, PA_EFLAG_CTX_OVERFLOW);
        if (tq0 + tok < min(min(max(it.n, 0), p.max_q), tq0 + p.tpq))
#pragma unroll
          for (int c = 0; c < 16; ++c) orow[c] = make_uint4(0, 0, 0, 0);
        continue;
      }
      const int nt = it.n_tiles;
      if (nt == 0 || !(wg == 0 ? it.has0 : it.has1)) {
        g += nt;
        continue;
      }
      const bool row_ok = tq0 + tok < it.t_end;
      const int row_pos = it.first_pos + tq0 + tok;
      const int row_lo = p.window > 0 ? max(0, row_pos - p.window + 1) : 0;
      float m_run = kNegInfTc, l_run = 0.f;
      for (int k = 0; ok && k < nt; ++k) {
        if (!warp_wait(&s_full[wg], sp & 1u)) {
          ok = false;
          break;
        }
        ++sp;
        tc_fence_after();
        uint32_t sv[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(sv + 32 * c));
        tmem_wait_ld();
        const int kbase = (it.kb0 + 8 * k) * PA_BLOCK_SIZE;
        // scores stay raw (the scale is positive, so the maximum commutes with it); only tiles
        // that cross a row's causal or window edge take the per-key mask, and within them only
        // the 32-key chunks that some row of the warp attends in part (a row attends the tile's
        // columns lo .. hi; on a diagonal tile a warp's rows, 32 / G tokens, put one or two of
        // the four chunks across their edges).  A chunk that no row of the warp attends (`dead`,
        // the keys past the item's last query on its diagonal tile) takes no maximum and no
        // exponentials: its P is zero.
        unsigned dead = 0;
        if (!__all_sync(0xffffffffu, row_ok && kbase + 127 <= row_pos && kbase >= row_lo)) {
          const int lo = row_lo - kbase, hi = row_ok ? row_pos - kbase : -1;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (__all_sync(0xffffffffu, lo <= 32 * q && hi >= 32 * q + 31)) continue;
            if (__all_sync(0xffffffffu, hi < 32 * q || lo > 32 * q + 31)) {
              dead |= 1u << q;
              continue;
            }
#pragma unroll
            for (int c = 32 * q; c < 32 * q + 32; ++c)
              if (c < lo || c > hi) sv[c] = __float_as_uint(kNegInfTc);
          }
        }
        float mx4[4] = {kNegInfTc, kNegInfTc, kNegInfTc, kNegInfTc};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if ((dead >> q) & 1u) continue;
#pragma unroll
          for (int c = 32 * q; c < 32 * q + 32; c += 2)
            mx4[(c >> 1) & 3] = max3f(mx4[(c >> 1) & 3], __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]));
        }
        const float mraw = fmaxf(max3f(mx4[0], mx4[1], mx4[2]), mx4[3]);
        const float mx = mraw == kNegInfTc ? kNegInfTc : mraw * p.scale_log2;
        const float m_new = (m_run == kNegInfTc || mx > m_run + 8.f) ? fmaxf(m_run, mx) : m_run;
        const float ms = m_new == kNegInfTc ? 0.f : m_new;
        const float alpha = ex2(m_run - ms);
        const bool moved = k > 0 && __any_sync(0xffffffffu, m_new != m_run);
        m_run = m_new;
        // key row r of V: zero it when it holds no loaded in-context data (both groups write the
        // same zeros; each must see them before its own P·V)
        const int kp_r = kbase + r;
        const bool zero_row = kp_r < it.kv_lo || kp_r >= it.loaded_end;
        const int gk = g + k, vs = gk % kVStages;
        if (__any_sync(0xffffffffu, zero_row)) {
          // the stage's copies must have landed first
          if (!warp_wait(&v_full[vs], static_cast<uint32_t>(gk / kVStages) & 1u)) {
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
        // P (bf16 pairs) over the S columns just read: column c holds keys 2c and 2c + 1; when the
        // maximum moved, O is rescaled before P is handed over.
        float ls4[4] = {0.f, 0.f, 0.f, 0.f};
        const float sl = p.scale_log2;
#pragma unroll
        for (int h = 0; h < 4; ++h) {  // a quarter (32 keys, 16 columns) at a time
          uint32_t pw[16];
          if ((dead >> h) & 1u) {
#pragma unroll
            for (int e = 0; e < 16; ++e) pw[e] = 0u;
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float a = ex2(fmaf(__uint_as_float(sv[32 * h + 2 * e]), sl, -ms));
              const float b = ex2(fmaf(__uint_as_float(sv[32 * h + 2 * e + 1]), sl, -ms));
              ls4[e & 3] += a + b;
              pw[e] = pack_bf16(a, b);
            }
          }
          tmem_st16(tS + 16 * h, pw);
        }
        tmem_wait_st();
        l_run = l_run * alpha + ((ls4[0] + ls4[1]) + (ls4[2] + ls4[3]));
        if (moved) {
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
        tc_fence_before();
        mbar_arrive(&p_full[wg]);
      }
      g += nt;
      // a table entry of the item's keys outside the pool: its rows become zero (read while the
      // last P·V runs)
      bool bad = false;
      {
        const int32_t* trow = p.block_tables + static_cast<size_t>(it.s) * p.max_blocks;
        for (int kb = it.kb0 + lane; kb < it.kb_end; kb += 32) {
          const int e = trow[kb];
          bad |= e < 0 || e >= p.num_blocks;
        }
        bad = __any_sync(0xffffffffu, bad);
      }
      // output: O / l as bf16 (zeros when a wait gave up or a block id was bad), staged in the
      // ring stage of the item's last tile that this group owns: K for query tile 0, V for 1.
      // o_done of the last tile follows every product of the CTA that reads either, so both are
      // idle.  One thread stores the tile with two TMA boxes (the copy engine, not the load/store
      // unit, moves the bytes), waits until they have been read and releases the stage to its
      // copy warp.  A tile that holds rows past its sequence is stored row by row instead
      // (coalesced).
      if (ok) ok = warp_wait(&o_done[wg], (sp - 1u) & 1u);
      tc_fence_after();
      // zero rows are selected, not multiplied: O may hold NaN when a block was not loaded (its
      // stage keeps earlier bytes) or no key was attended
      const bool zero_out = !ok || bad || !(l_run > 0.f);
      const float inv = zero_out ? 0.f : 1.f / l_run;
      const int g_last = g - 1;
      uint8_t* stile =
          wg == 0 ? sm + kKOff + (g_last % kKStages) * kTile : sm + kVOff + (g_last % kVStages) * kTile;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t ov[32];
        if (ok) {
          tmem_ld32(tO + 32 * c, ov);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = 0u;
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {  // 16-byte chunk j = 4c + q4 of row r (dims 8j .. 8j + 7)
          const int j = 4 * c + q4;
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = zero_out ? 0u
                            : pack_bf16(__uint_as_float(ov[8 * q4 + 2 * e]) * inv,
                                        __uint_as_float(ov[8 * q4 + 2 * e + 1]) * inv);
          *reinterpret_cast<uint4*>(stile + (j >> 3) * kHalf + r * 128 + (((j & 7) ^ (r & 7)) << 4)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      tc_fence_before();
      fence_proxy_async();  // the staged rows, before the copy engine reads them
      group_sync(1 + wg);
      const bool release = wg == 0 ? g_last + kKStages < g_tot : g_last + kVStages < g_tot;
      uint64_t* rel = wg == 0 ? &k_empty[g_last % kKStages] : &v_empty[g_last % kVStages];
      if (tq0 + p.tpq <= it.t_end) {
        if (quad == 0 && lane == 0) {
          for (int half = 0; half < 2; ++half)
            tma_store_4d(&tmO, stile + half * kHalf, 0, half, it.h_kv * p.G, it.qs + tq0);
          bulk_commit();
          bulk_wait_read();
          if (release) mbar_arrive(rel);
        }
      } else {
        const int c = lane & 15;
#pragma unroll 4
        for (int i = 0; i < 16; ++i) {  // this warp's rows, two per instruction
          const int rr = quad * 32 + 2 * i + (lane >> 4);
          const int tk = rr / p.G;
          if (tq0 + tk < it.t_end)
            reinterpret_cast<uint4*>(p.out + (static_cast<size_t>(it.qs + tq0 + tk) * p.H_q + it.h_kv * p.G +
                                              (rr - tk * p.G)) * D)[c] =
                *reinterpret_cast<const uint4*>(stile + (c >> 3) * kHalf + rr * 128 + (((c & 7) ^ (rr & 7)) << 4));
        }
        group_sync(1 + wg);  // every row has been read back before the stage is released
        if (quad == 0 && lane == 0 && release) mbar_arrive(rel);
      }
    }
    bulk_wait_all();  // this thread's output stores are complete
    if (!ok && lane == 0) flags[1] = 1;
  }
  // ------------------------------ teardown ------------------------------
  tc_fence_before();
  __syncthreads();  // no TMEM access is pending
  if (tid == 64 && flags[1] != 0) set_error(p.err, PA_EFLAG_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// CTAs that can run at once on the current device (persistent grid size).
int resident_ctas() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < 64 && cached[dev] > 0) return cached[dev];
  int sms = 0, per_sm = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, prefill_tc_kernel, kTcThreads, kTcSmem) != cudaSuccess ||
      per_sm <= 0) {
    cudaGetLastError();
    per_sm = 1;
  }
  const int n = sms * per_sm;
  if (dev < 64) cached[dev] = n;
  return n;
}

}  // namespace

// Host launch (declared in pa_internal.h): the tcgen05 path of pa_prefill_attention.
pa_status launch_prefill_tc(const pa_cache_desc* desc, void* out, const void* q, const void* k_cache,
                            const void* v_cache, const int32_t* block_tables, const int32_t* q_start,
                            const int32_t* context_lens, int max_query_len, float scale, int32_t* err_flag,
                            cudaStream_t stream, bool step) {
  const long long slots = static_cast<long long>(desc->num_blocks) * PA_BLOCK_SIZE;
  CUtensorMap mk, mv, mq, mo;
  const int G = desc->num_q_heads / desc->num_kv_heads;
  if (!encode_cache_map(&mk, k_cache, 2, desc->num_kv_heads * 2, 1, slots) ||
      !encode_cache_map(&mv, v_cache, 2, desc->num_kv_heads * 2, 1, slots) ||
      !encode_query_map(&mq, q, desc->num_q_heads, G, 128 / G, kQMapTokens) ||
      !encode_query_map(&mo, out, desc->num_q_heads, G, 128 / G, kQMapTokens))
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
  p.step = step ? 1 : 0;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.q_start = q_start;
  p.context_lens = context_lens;
  p.block_tables = block_tables;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.err = err_flag;
  if (!ensure_dynamic_smem(reinterpret_cast<const void*>(prefill_tc_kernel), kTcSmem)) return PA_ERR_CUDA;
  // Persistent CTAs: as many as run at once, but no more than there are work items, and enough
  // that none holds more than kMaxItems of them.
  const long long w_tokens = 2LL * p.tpq;  // query tokens of one tile
  const long long items = static_cast<long long>(p.B) * ((max_query_len + w_tokens - 1) / w_tokens) * p.H_kv;
  if (items > (1LL << 30)) return PA_ERR_UNSUPPORTED;
  long long nc = std::min<long long>(items, std::max(1, resident_ctas()));
  nc = std::max(nc, (items + kMaxItems - 1) / kMaxItems);
  nc = std::max(nc, 1LL);
  if (nc > 0x7FFFFFFFLL) return PA_ERR_UNSUPPORTED;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(nc));
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = kTcSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_tc_kernel, mk, mv, mq, mo, p) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa

// Decode attention over the paged KV cache: the hot path.
//
// What is computed (untitled KV-cache article at ldpk.cn/news/58971, §2.1 and §2.2): one query
// row per head against every cached key, softmax(q·Kᵀ·scale)·V.  GQA ("KV Cache 的显存账本：
// PagedAttention 与连续批处理" §二): every G consecutive query heads read one KV head.  The keys
// and values are fetched from non-contiguous physical blocks through the block table
// (ldpk §4.3; 显存账本 §四 locate()).  8-bit caches (显存账本 §七) are decoded in registers; with
// per-token K scales (ldpk §5.2) each token's score takes its own K scale.
// Under a sliding window (ldpk §5.3) only the blocks holding the last W positions are listed,
// so the work, the bytes and the table entries read scale with W, not with the context.
//
// Design (GB300, sm_103a):
//  * Work unit = one 16-token physical block of one head group.  A CTA owns a contiguous range
//    of the (sequence, logical block) list: in balanced mode the list of all sequences is cut
//    into equal ranges, one per SM, so that any mix of context lengths keeps every SM busy; in
//    fixed mode each CTA owns one partition of partition_size tokens of one sequence.
//  * A producer warp resolves block-table entries and streams every block with TMA
//    (cp.async.bulk.tensor, 128-byte swizzle) into a ring of shared-memory stages guarded by
//    mbarriers.  The slot-major cache keeps each block's rows of all heads contiguous; one box per
//    tensor carries the block for all heads of the group, head-major (each head's 16 slots form a
//    tile), so a stage holds whole blocks and no byte is fetched twice.
//  * One consumer warp per (KV head, block of the stage).  q·Kᵀ for the G query heads of the KV
//    head and the 16 tokens of the block is an m16n8k16 tensor-core product (tokens = M, query
//    heads = N); the probabilities are transposed in registers (movmatrix) into the B operand
//    of P·V (head_dim = M).  The softmax is the online (running max) form in fp32 with warp
//    shuffles; with enough stages a warp takes two blocks of one sequence as one 32-token step.
//    Partial (m, l, o) go to the workspace and a merge kernel combines them by log-sum-exp; a warp
//    that saw a whole sequence writes the bf16 output directly.
//  * In a decode step (pa_decode_step) the kernel overlaps the append launched just before it and
//    waits for it only before the blocks that receive the appended tokens.
//  * With a shared prefix attended apart (pa_decode_attention_shared, shared_prefix.cu) a member
//    sequence's list starts past the prefix, and the merge folds in the prefix's partial rows.
//  * Every wait is bounded; invalid table entries and contexts set error bits and zero rows.

#include <algorithm>
#include <cmath>
#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kTileBytes = 2048;  // one TMA box: 16 slots x 128 bytes
constexpr int kMaxConsumerWarps = 16;
constexpr int kMaxThreads = (kMaxConsumerWarps + 1) * 32;
constexpr int kAutoMaxSeqs = 2048;
constexpr int kFixedFallbackPartition = 512;
// Tuning constants (compile-time; the defaults are the measured best on GB300).
#ifndef PA_CTAS_PER_SM
#define PA_CTAS_PER_SM 1  // balanced mode: resident CTAs per SM
#endif
#ifndef PA_GROUP_BYTES
#define PA_GROUP_BYTES 2048  // KV heads per CTA: as many as fit this many bytes of one slot
#endif
#ifndef PA_MAX_STAGES
#define PA_MAX_STAGES 8
#endif
// INT4: at most this many KV heads per CTA, and this many consumer warps per CTA (blocks per
// stage = warps / heads).  The 4-bit path is bound by its dequantising arithmetic, so it
// trades heads per CTA for more warps in flight.
#ifndef PA_I4_MAX_HG
#define PA_I4_MAX_HG 8
#endif
#ifndef PA_I4_WARPS
#define PA_I4_WARPS 8
#endif
constexpr int kMaxStages = PA_MAX_STAGES;
// shared memory a CTA may use when `ctas` of them share an SM
constexpr int smem_limit(int ctas) { return ctas == 1 ? 227 * 1024 : (228 * 1024) / ctas - 1024; }
constexpr float kNegInf = -INFINITY;

struct DecodeParams {
  int B, H_q, H_kv, G, num_blocks, max_blocks, num_sink, max_ctx;
  int window;  // sliding window in tokens, 0 = whole context
  int hg, nc, nbs, stages, warps_c;
  int block_bytes;  // shared-memory bytes of one block in a stage
  int block_tx;     // bytes the copies of one block deliver (block_bytes less alignment padding)
  int mode;  // 0 balanced, 1 fixed partitions
  int ppb, max_parts;
  int direct_ok;
  int stage_bytes;
  float scale_log2;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  const float* k_scales;
  const float* v_scales;
  const __nv_bfloat16* k_sink;
  const __nv_bfloat16* v_sink;
  float* partials;
  int32_t* ws_meta;
  int32_t* err;
  // Positions of the tokens that the append kernel launched just before this one writes, one per
  // sequence (a decode step), or null.  With them the kernel waits for that kernel only before
  // loading a block that holds such a position; without them it waits before reading anything.
  const int32_t* append_pos;
  // A shared prefix attended apart (pa_decode_attention_shared), or null: a sequence s with
  // shared_flags[s] == kSharedUse starts at position shared_len (a multiple of 16); its positions
  // below it are covered by n_extra partial rows per query head computed by the prefix kernel,
  // extra[((s * n_extra + i) * H_q + h) * (D + 4)], which the merge folds in with its own.
  const int32_t* shared_flags;
  const float* extra;
  int shared_len;
  int n_extra;
};

// Blocks of a sequence with ctx tokens; -1 for an invalid context.
__device__ __forceinline__ int seq_blocks(const DecodeParams& p, int ctx) {
  if (ctx == 0) return 0;
  if (ctx < 0 || ctx > p.max_ctx || ctx > p.max_blocks * PA_BLOCK_SIZE) return -1;
  return (ctx + PA_BLOCK_SIZE - 1) / PA_BLOCK_SIZE;
}

// First position the query attends: the last `window` positions (ldpk §5.3), else 0.
__device__ __forceinline__ int window_lo(const DecodeParams& p, int ctx) {
  return (p.window > 0 && ctx > p.window) ? ctx - p.window : 0;
}

// First position this kernel attends for sequence s (global index): the window's, or past the
// shared prefix attended apart.
__device__ __forceinline__ bool shares_prefix(const DecodeParams& p, int s) {
  return p.shared_flags && p.shared_flags[s] == kSharedUse;
}
__device__ __forceinline__ int seq_lo(const DecodeParams& p, int s, int ctx) {
  const int lo = window_lo(p, ctx);
  return shares_prefix(p, s) ? max(lo, min(p.shared_len, max(ctx, 0))) : lo;
}

// Logical blocks a sequence's query visits (those holding positions seq_lo .. ctx-1); -1 for an
// invalid context.
__device__ __forceinline__ int seq_span(const DecodeParams& p, int s, int ctx) {
  const int nb = seq_blocks(p, ctx);
  return nb <= 0 ? nb : nb - seq_lo(p, s, ctx) / PA_BLOCK_SIZE;
}

// Largest s in [0, n) with cum[s] <= u (cum non-decreasing, cum[0] <= u).
__device__ __forceinline__ int find_seq(const int* cum, int n, int u) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cum[mid] <= u) lo = mid; else hi = mid - 1;
  }
  return lo;
}

struct Smem {
  uint8_t* stages;
  uint64_t* full;
  uint64_t* empty;
  int4* meta;
  int* cum;
  int* ctxs;
  int* los;  // first attended position per sequence
  int* scratch;
};

__device__ __forceinline__ Smem carve(uint8_t* raw, const DecodeParams& p) {
  Smem s;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  s.stages = base;
  s.full = reinterpret_cast<uint64_t*>(base + static_cast<size_t>(p.stages) * p.stage_bytes);
  s.empty = s.full + p.stages;
  s.meta = reinterpret_cast<int4*>(s.empty + p.stages);
  s.cum = reinterpret_cast<int*>(s.meta + p.stages * p.nbs);
  s.ctxs = s.cum + (p.mode == 0 ? p.B + 1 : 2);
  s.los = s.ctxs + (p.mode == 0 ? p.B : 1);
  s.scratch = s.los + (p.mode == 0 ? p.B : 1);
  return s;
}

// ------------------------------------------------------------------------------------
// Consumer: one warp = one KV head x one block slot of every stage.
// ------------------------------------------------------------------------------------
// KIND 0: bf16 K and V; 1: FP8 E4M3 K and INT8 V with per-head scales; 2: INT4 K and V with a
// scale and zero point per 32 dims of every token's head row; 3: as 1, but K with one scale per
// token's head row (the block's scales follow its K and V tiles in the stage).
template <int D, int KIND>
struct Consumer {
  static constexpr bool QUANT = KIND == 1 || KIND == 3;
  static constexpr bool TOKS = KIND == 3;
  static constexpr bool I4 = KIND == 2;
  static constexpr int KT = D / 16;  // k-steps of q·Kᵀ and m-tiles of P·V
  static constexpr int NC = KIND != 0 ? 1 : D * 2 / 128;  // 128-byte chunks per head row
  const DecodeParams& p;
  uint32_t qf[KT][2];
  float o[KT][4];
  float m[2], l[2], sl[2];
  float vsc;
  // INT4 zero points, applied per 32-dim group instead of per code: qz[g][c] = sum of q over
  // group g for query head 2tq + c; cz[g][c] = running sum over tokens of p * s * (128 + z), the
  // part of P·V that the offset codes add to every dim of group g
  float qz[4][2], cz[4][2];
  bool bad;
  int lane, t4, tq, h_kv, j, h_loc;
  uint32_t kofs, vofs, kpofs, vpofs;  // this warp's tiles inside a stage (kpofs: K scales, KIND 3)
  // INT4: this lane's byte offsets inside a stage (they depend only on the lane and the head):
  // K codes of token t4, V codes of tokens 2tq and 2tq+1, K and V group parameters of token t4.
  // The tokens 8 slots further sit i4_dslot (codes: the same swizzle phase) or i4_dprm
  // (parameters) bytes later.
  uint32_t ik0, iv0, iv1, ikp0, ivp0;

  __device__ Consumer(const DecodeParams& p_, int lane_, int h_kv_, int j_, int h_loc_)
      : p(p_), vsc(1.f), lane(lane_), t4(lane_ >> 2), tq(lane_ & 3), h_kv(h_kv_), j(j_), h_loc(h_loc_) {
    sl[0] = sl[1] = p_.scale_log2;
    if constexpr (I4) {
      // block j of a stage: [K codes][V codes] (16 slots x hg/2 rows x 128 B, swizzled), then
      // [K params][V params] (16 slots x hg heads x 16 B)
      kofs = j * p_.block_bytes;
      vofs = kofs + p_.hg * 1024;
      kpofs = kofs + 2 * p_.hg * 1024;
      vpofs = kpofs + p_.hg * 256;
      ik0 = kofs + i4_code_off(t4, tq * 16);
      iv0 = vofs + i4_code_off(2 * tq, t4 * 8);
      iv1 = vofs + i4_code_off(2 * tq + 1, t4 * 8);
      ikp0 = kpofs + (t4 * p_.hg + h_loc_) * 16;
      ivp0 = vpofs + (t4 * p_.hg + h_loc_) * 16;
    } else {
      // block j of a stage: [K tiles][V tiles] (hg heads x nc tiles each), then (KIND 3) the
      // K scales [16 slots][hg heads] fp32
      kofs = j * p_.block_bytes + h_loc_ * p_.nc * kTileBytes;
      vofs = kofs + p_.hg * p_.nc * kTileBytes;
      kpofs = j * p_.block_bytes + 2 * p_.hg * p_.nc * kTileBytes + h_loc_ * 4;
      vpofs = 0;
    }
    reset();
  }

  __device__ __forceinline__ void reset() {
    m[0] = m[1] = kNegInf;
    l[0] = l[1] = 0.f;
    bad = false;
#pragma unroll
    for (int i = 0; i < KT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    if constexpr (I4) {
#pragma unroll
      for (int g = 0; g < 4; ++g) cz[g][0] = cz[g][1] = 0.f;
    }
  }

  // B fragments of q for this KV head's G query heads (N = head, K = head_dim).
  __device__ __forceinline__ void load_q(int s) {
    const bool live = t4 < p.G;
    const __nv_bfloat16* qrow = p.q + (static_cast<size_t>(s) * p.H_q + h_kv * p.G + (live ? t4 : 0)) * D;
    if constexpr (I4) {
      // k-steps 2g and 2g+1 take the dims of 32-dim group g that lane tq's K words hold:
      // 32g + 8tq + {0,4 | 1,5} and {2,6 | 3,7} (the pairs one mask pulls out of a code word)
#pragma unroll
      for (int g = 0; g < D / 32; ++g) {
        const uint4 x = live ? *reinterpret_cast<const uint4*>(qrow + g * 32 + tq * 8) : make_uint4(0, 0, 0, 0);
        qf[2 * g][0] = prmt(x.x, x.z, 0x5410);
        qf[2 * g][1] = prmt(x.x, x.z, 0x7632);
        qf[2 * g + 1][0] = prmt(x.y, x.w, 0x5410);
        qf[2 * g + 1][1] = prmt(x.y, x.w, 0x7632);
        // sum of the group's 32 q values of head t4 (8 here, then over the four tq lanes)
        const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
        float sg = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) sg += __uint_as_float(xw[e] << 16) + __uint_as_float(xw[e] & 0xFFFF0000u);
        sg += __shfl_xor_sync(0xffffffffu, sg, 1);
        sg += __shfl_xor_sync(0xffffffffu, sg, 2);
        // this lane's score columns are heads 2tq, 2tq + 1: lanes 8tq and 8tq + 4 hold them
        qz[g][0] = __shfl_sync(0xffffffffu, sg, 8 * tq);
        qz[g][1] = __shfl_sync(0xffffffffu, sg, 8 * tq + 4);
      }
      sl[0] = sl[1] = p.scale_log2;
      vsc = 1.f;
    } else if constexpr (!QUANT) {
#pragma unroll
      for (int kk = 0; kk < KT; ++kk) {
        qf[kk][0] = live ? *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 2 * tq) : 0u;
        qf[kk][1] = live ? *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 8 + 2 * tq) : 0u;
      }
      sl[0] = sl[1] = p.scale_log2;
      vsc = 1.f;
    } else {
      // fp16 operands: q is scaled by a power of two so that its largest element lands just
      // below 2^15 (every bf16 value in range then converts exactly), and the factor is
      // removed again from the scores.  Dims are taken in the order the 8-bit K fragment
      // delivers them: k-step kk uses d = 16kk + 4tq + {0,1} (b0) and {2,3} (b1).
      float x[KT][4];
      float mx = 0.f;
#pragma unroll
      for (int kk = 0; kk < KT; ++kk) {
        uint2 raw = live ? *reinterpret_cast<const uint2*>(qrow + kk * 16 + 4 * tq) : make_uint2(0, 0);
        x[kk][0] = __uint_as_float(raw.x << 16);
        x[kk][1] = __uint_as_float(raw.x & 0xFFFF0000u);
        x[kk][2] = __uint_as_float(raw.y << 16);
        x[kk][3] = __uint_as_float(raw.y & 0xFFFF0000u);
#pragma unroll
        for (int e = 0; e < 4; ++e) mx = fmaxf(mx, fabsf(x[kk][e]));
      }
      mx = warp_max_xor(mx, 1);
      mx = warp_max_xor(mx, 2);
      int e2 = 0;
      if (mx > 0.f) {
        frexpf(mx, &e2);
        e2 = min(15 - e2, 100);
      }
      const float f = ldexpf(1.f, e2);
#pragma unroll
      for (int kk = 0; kk < KT; ++kk) {
        qf[kk][0] = pack_f16(x[kk][0] * f, x[kk][1] * f);
        qf[kk][1] = pack_f16(x[kk][2] * f, x[kk][3] * f);
      }
      const int e_c0 = __shfl_sync(0xffffffffu, e2, 4 * (2 * tq));
      const int e_c1 = __shfl_sync(0xffffffffu, e2, 4 * (2 * tq + 1));
      // per-token K scales multiply each token's score in scores() instead
      const float base = TOKS ? p.scale_log2 : p.scale_log2 * p.k_scales[h_kv];
      sl[0] = base * ldexpf(1.f, -e_c0);
      sl[1] = base * ldexpf(1.f, -e_c1);
      vsc = p.v_scales[h_kv];
    }
  }

  // INT4: 8 slots further in a codes tile (8 x hg/2 rows of 128 bytes, a multiple of the 8-row
  // swizzle period) and in a parameter tile (8 x hg rows of 16 bytes)
  __device__ __forceinline__ uint32_t i4_dslot() const { return 8 * (p.hg >> 1) * 128; }
  __device__ __forceinline__ uint32_t i4_dprm() const { return 8 * p.hg * 16; }

  // INT4: byte x (0..63) of this warp's head row in slot `slot` of a codes tile, whose 128-byte
  // rows hold two heads each and carry the 128-byte swizzle of the TMA box.
  __device__ __forceinline__ uint32_t i4_code_off(int slot, int x) const {
    const int R = slot * (p.hg >> 1) + (h_loc >> 1);
    const int xb = ((h_loc & 1) << 6) + x;
    return static_cast<uint32_t>(R * 128 + ((((xb >> 4) ^ (R & 7)) << 4) | (xb & 15)));
  }


  // INT4 block.  Codes become exact bf16 integers (128 + n) - (128 + z) = n - z.  Scores: lane
  // tq's K words hold whole 32-dim groups, so the two k-steps of group g accumulate apart and
  // the group's scale multiplies the fp32 sum.  P·V: the MMA sums over tokens, so each token's
  // group scale goes into P before the transpose; the output rows are dims 16mt + t4 (+8).
  __device__ __forceinline__ void scores_i4(const uint8_t* stage, float (&acc)[4]) const {
    const uint4 kw0 = *reinterpret_cast<const uint4*>(stage + ik0);
    const uint4 kw1 = *reinterpret_cast<const uint4*>(stage + ik0 + i4_dslot());
    const uint4 kq0 = *reinterpret_cast<const uint4*>(stage + ikp0);
    const uint4 kq1 = *reinterpret_cast<const uint4*>(stage + ikp0 + i4_dprm());
    const uint32_t w0[4] = {kw0.x, kw0.y, kw0.z, kw0.w}, w1[4] = {kw1.x, kw1.y, kw1.z, kw1.w};
    const uint32_t q0[4] = {kq0.x, kq0.y, kq0.z, kq0.w}, q1[4] = {kq1.x, kq1.y, kq1.z, kq1.w};
    acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      // q·(128 + n) over the group's 32 dims, then - (128 + z) * sum(q) and * scale
      float ag[4] = {0.f, 0.f, 0.f, 0.f};
      mma_bf16(ag, nib_pair(w0[g], 0), nib_pair(w1[g], 0), nib_pair(w0[g], 1), nib_pair(w1[g], 1), qf[2 * g][0],
               qf[2 * g][1]);
      mma_bf16(ag, nib_pair(w0[g], 2), nib_pair(w1[g], 2), nib_pair(w0[g], 3), nib_pair(w1[g], 3),
               qf[2 * g + 1][0], qf[2 * g + 1][1]);
      const float c0 = __uint_as_float(0x43000000u | (q0[g] & 0x00FF0000u));  // 128 + z (z < 16)
      const float c1 = __uint_as_float(0x43000000u | (q1[g] & 0x00FF0000u));
      const float s0 = __uint_as_float(q0[g] << 16), s1 = __uint_as_float(q1[g] << 16);
      acc[0] = fmaf(s0, fmaf(-c0, qz[g][0], ag[0]), acc[0]);
      acc[1] = fmaf(s0, fmaf(-c0, qz[g][1], ag[1]), acc[1]);
      acc[2] = fmaf(s1, fmaf(-c1, qz[g][0], ag[2]), acc[2]);
      acc[3] = fmaf(s1, fmaf(-c1, qz[g][1], ag[3]), acc[3]);
    }
  }

  __device__ __forceinline__ void pv_i4(const uint8_t* stage, const float (&pr)[4], int first, int ntok) {
    const float p00 = pr[0], p01 = pr[1], p10 = pr[2], p11 = pr[3];
    // scales of the P rows (tokens t4, t4 + 8); a masked token's slot may hold any bits, so its
    // scale is replaced by 0 rather than multiplied in
    const bool v0 = t4 < ntok && t4 >= first;
    const bool v1 = t4 + 8 < ntok && t4 + 8 >= first;
    const uint4 vs0 = *reinterpret_cast<const uint4*>(stage + ivp0);
    const uint4 vs1 = *reinterpret_cast<const uint4*>(stage + ivp0 + i4_dprm());
    const uint32_t sv0w[4] = {vs0.x, vs0.y, vs0.z, vs0.w}, sv1w[4] = {vs1.x, vs1.y, vs1.z, vs1.w};
    // codes of the A columns: tokens 2tq, 2tq+1 (a0, a1) and 2tq+8, 2tq+9 (a2, a3)
    const uint2 cA = *reinterpret_cast<const uint2*>(stage + iv0);
    const uint2 cB = *reinterpret_cast<const uint2*>(stage + iv1);
    const uint2 cC = *reinterpret_cast<const uint2*>(stage + iv0 + i4_dslot());
    const uint2 cD = *reinterpret_cast<const uint2*>(stage + iv1 + i4_dslot());
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const float sv0 = v0 ? __uint_as_float(sv0w[g] << 16) : 0.f;
      const float sv1 = v1 ? __uint_as_float(sv1w[g] << 16) : 0.f;
      // P * s as bf16, exactly as the MMA takes it; the offset codes add sum_t p s (128 + z) to
      // every dim of the group, kept in cz and removed when the output is written
      const uint32_t x0 = pack_bf16(p00 * sv0, p01 * sv0), x1 = pack_bf16(p10 * sv1, p11 * sv1);
      const float c0 = __uint_as_float(0x43000000u | (sv0w[g] & 0x00FF0000u));  // 128 + z
      const float c1 = __uint_as_float(0x43000000u | (sv1w[g] & 0x00FF0000u));
      cz[g][0] = fmaf(__uint_as_float(x0 << 16), c0, fmaf(__uint_as_float(x1 << 16), c1, cz[g][0]));
      cz[g][1] = fmaf(__uint_as_float(x0 & 0xFFFF0000u), c0, fmaf(__uint_as_float(x1 & 0xFFFF0000u), c1, cz[g][1]));
      const uint32_t b0 = movmatrix_t(x0), b1 = movmatrix_t(x1);
#pragma unroll
      for (int mm = 0; mm < 2; ++mm) {
        const int mt = 2 * g + mm, k = mt & 3;
        const uint32_t sel = static_cast<uint32_t>(k | ((k + 4) << 8));  // byte k of each token
        const uint32_t tAB = prmt(mt < 4 ? cA.x : cA.y, mt < 4 ? cB.x : cB.y, sel);
        const uint32_t tCD = prmt(mt < 4 ? cC.x : cC.y, mt < 4 ? cD.x : cD.y, sel);
        mma_bf16(o[mt], nib_pair(tAB, 0), nib_pair(tAB, 1), nib_pair(tCD, 0), nib_pair(tCD, 1), b0, b1);
      }
    }
  }

  // q·Kᵀ of one 16-token block for this warp's head: acc rows = tokens t4, t4 + 8, columns =
  // query heads 2tq, 2tq + 1, not yet scaled.  Two independent accumulation chains halve the
  // dependent-MMA latency.
  __device__ __forceinline__ void scores(const uint8_t* stage, float (&acc)[4]) const {
    const uint8_t* kbase = stage + kofs;
    float acc2[4] = {0.f, 0.f, 0.f, 0.f};
    acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
    const int tokA = (lane & 7) + ((lane >> 3) & 1) * 8;
    if constexpr (!QUANT) {
      const int halfA = lane >> 4;
#pragma unroll
      for (int kk = 0; kk < KT; ++kk) {
        const int ch16 = (kk & 3) * 2 + halfA;
        const int row = tokA * NC + (kk >> 2);  // 128-byte row of the swizzled tile
        const uint32_t addr = smem_u32(kbase + row * 128 + ((ch16 ^ (row & 7)) << 4));
        uint32_t a0, a1, a2, a3;
        ldsm_x4(addr, a0, a1, a2, a3);
        mma_bf16((kk & 1) ? acc2 : acc, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
      }
    } else {
#pragma unroll
      for (int kp = 0; kp < KT / 2; ++kp) {
        const int ch16 = 2 * kp + (lane >> 4);
        const uint32_t addr = smem_u32(kbase + tokA * 128 + ((ch16 ^ (tokA & 7)) << 4));
        uint32_t r0, r1, r2, r3;
        ldsm_x4(addr, r0, r1, r2, r3);
        mma_f16(acc, e4m3x2_to_f16x2(r0), e4m3x2_to_f16x2(r1), e4m3x2_to_f16x2(r0 >> 16),
                e4m3x2_to_f16x2(r1 >> 16), qf[2 * kp][0], qf[2 * kp][1]);
        mma_f16(acc2, e4m3x2_to_f16x2(r2), e4m3x2_to_f16x2(r3), e4m3x2_to_f16x2(r2 >> 16),
                e4m3x2_to_f16x2(r3 >> 16), qf[2 * kp + 1][0], qf[2 * kp + 1][1]);
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[e] += acc2[e];
    if constexpr (TOKS) {
      // rows t4 and t4 + 8 of the block: their tokens' K scales ([slot][head] fp32 in the stage)
      const float s0 = *reinterpret_cast<const float*>(stage + kpofs + t4 * p.hg * 4);
      const float s1 = *reinterpret_cast<const float*>(stage + kpofs + (t4 + 8) * p.hg * 4);
      acc[0] *= s0;
      acc[1] *= s0;
      acc[2] *= s1;
      acc[3] *= s1;
    }
  }

  // Online-softmax update over NB blocks' scores at once (one maximum, one rescale check);
  // pr[b] = this lane's unnormalised probabilities {row t4: head 2tq, 2tq+1; row t4+8: same}.
  template <int NB>
  __device__ __forceinline__ void softmax_n(const float (&acc)[NB][4], const int (&first)[NB], const int (&ntok)[NB],
                                            float (&pr)[NB][4]) {
    float s[NB][4];
    float bm0 = kNegInf, bm1 = kNegInf;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const bool v0 = t4 < ntok[b] && t4 >= first[b];
      const bool v1 = t4 + 8 < ntok[b] && t4 + 8 >= first[b];
      s[b][0] = v0 ? acc[b][0] * sl[0] : kNegInf;
      s[b][1] = v0 ? acc[b][1] * sl[1] : kNegInf;
      s[b][2] = v1 ? acc[b][2] * sl[0] : kNegInf;
      s[b][3] = v1 ? acc[b][3] * sl[1] : kNegInf;
      bm0 = fmaxf(bm0, fmaxf(s[b][0], s[b][2]));
      bm1 = fmaxf(bm1, fmaxf(s[b][1], s[b][3]));
    }
#pragma unroll
    for (int mask = 4; mask <= 16; mask <<= 1) {
      bm0 = warp_max_xor(bm0, mask);
      bm1 = warp_max_xor(bm1, mask);
    }
    // The reference maximum only moves when a score exceeds it by more than 2^8 (exact: the
    // final division by l uses the same reference), so most blocks skip the rescale of o.
    const float mn0 = (m[0] == kNegInf || bm0 > m[0] + 8.f) ? fmaxf(m[0], bm0) : m[0];
    const float mn1 = (m[1] == kNegInf || bm1 > m[1] + 8.f) ? fmaxf(m[1], bm1) : m[1];
    const float ms0 = mn0 == kNegInf ? 0.f : mn0;
    const float ms1 = mn1 == kNegInf ? 0.f : mn1;
    float add0 = 0.f, add1 = 0.f;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      pr[b][0] = ex2(s[b][0] - ms0);
      pr[b][1] = ex2(s[b][1] - ms1);
      pr[b][2] = ex2(s[b][2] - ms0);
      pr[b][3] = ex2(s[b][3] - ms1);
      add0 += pr[b][0] + pr[b][2];
      add1 += pr[b][1] + pr[b][3];
    }
    if (__any_sync(0xffffffffu, mn0 != m[0] || mn1 != m[1])) {
      const float al0 = ex2(m[0] - ms0), al1 = ex2(m[1] - ms1);
      l[0] *= al0;
      l[1] *= al1;
#pragma unroll
      for (int mt = 0; mt < KT; ++mt) {
        o[mt][0] *= al0;
        o[mt][1] *= al1;
        o[mt][2] *= al0;
        o[mt][3] *= al1;
      }
      if constexpr (I4) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          cz[g][0] *= al0;
          cz[g][1] *= al1;
        }
      }
    }
    l[0] += add0;
    l[1] += add1;
    m[0] = mn0;
    m[1] = mn1;
  }

  // O += P·V of one block, P = pr (this lane's probabilities, tokens x heads).
  __device__ __forceinline__ void pv(const uint8_t* stage, const float (&pr)[4], int first, int ntok) {
    const uint8_t* vbase = stage + vofs;
    // P (tokens x heads) -> B operand (K = tokens, N = heads) of P·V
    const uint32_t x0 = QUANT ? pack_f16(pr[0], pr[1]) : pack_bf16(pr[0], pr[1]);
    const uint32_t x1 = QUANT ? pack_f16(pr[2], pr[3]) : pack_bf16(pr[2], pr[3]);
    const uint32_t b0 = movmatrix_t(x0), b1 = movmatrix_t(x1);
    if constexpr (!QUANT) {
      // Slots outside the attended range (tail of the last block, sink positions, positions
      // before the window) may hold any bits, NaN included, and 0 * NaN would poison the sum:
      // zero those tokens' V elements.  This lane's A fragments hold tokens 2tq, 2tq+1 (a0, a1)
      // and 2tq+8, 2tq+9 (a2, a3).
      uint32_t mlo = 0xFFFFFFFFu, mhi = 0xFFFFFFFFu;
      if (ntok < PA_BLOCK_SIZE || first > 0) {
        auto keep = [&](int r) { return r < ntok && r >= first; };
        mlo = (keep(2 * tq) ? 0x0000FFFFu : 0u) | (keep(2 * tq + 1) ? 0xFFFF0000u : 0u);
        mhi = (keep(2 * tq + 8) ? 0x0000FFFFu : 0u) | (keep(2 * tq + 9) ? 0xFFFF0000u : 0u);
      }
      const int tokB = (lane & 7) + (lane >> 4) * 8;
      const int halfB = (lane >> 3) & 1;
#pragma unroll
      for (int mt = 0; mt < KT; ++mt) {
        const int ch16 = (mt & 3) * 2 + halfB;
        const int row = tokB * NC + (mt >> 2);
        const uint32_t addr = smem_u32(vbase + row * 128 + ((ch16 ^ (row & 7)) << 4));
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(addr, a0, a1, a2, a3);
        mma_bf16(o[mt], a0 & mlo, a1 & mlo, a2 & mhi, a3 & mhi, b0, b1);
      }
    } else {
      // int8 V: a transposed 8x8 load of 16-bit pairs gives each lane two d values of two
      // tokens; output row m = t4 holds d = 16mt + 2t4 and row m = t4+8 holds d + 1.  Codes are
      // finite, so tokens outside the attended range (P = 0) need no masking.
      const int tokA = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int mp = 0; mp < KT / 2; ++mp) {
        const int ch16 = 2 * mp + (lane >> 4);
        const uint32_t addr = smem_u32(vbase + tokA * 128 + ((ch16 ^ (tokA & 7)) << 4));
        uint32_t r0, r1, r2, r3;
        ldsm_x4_t(addr, r0, r1, r2, r3);
        r0 ^= 0x80808080u;
        r1 ^= 0x80808080u;
        r2 ^= 0x80808080u;
        r3 ^= 0x80808080u;
        mma_f16(o[2 * mp], i8x2_to_f16x2(r0, 0x4240), i8x2_to_f16x2(r0, 0x4341),
                i8x2_to_f16x2(r1, 0x4240), i8x2_to_f16x2(r1, 0x4341), b0, b1);
        mma_f16(o[2 * mp + 1], i8x2_to_f16x2(r2, 0x4240), i8x2_to_f16x2(r2, 0x4341),
                i8x2_to_f16x2(r3, 0x4240), i8x2_to_f16x2(r3, 0x4341), b0, b1);
      }
    }
  }

  // One 16-token block: scores, online softmax update, P·V.
  // Tokens first .. ntok-1 of the block are attended; those below `first` are sink positions
  // (read from the bf16 sink buffer by the merge) or lie before the sliding window.
  __device__ __forceinline__ void block(const uint8_t* stage, int first, int ntok) {
    float acc[1][4], pr[1][4];
    const int f[1] = {first}, n[1] = {ntok};
    if constexpr (I4) {
      scores_i4(stage, acc[0]);
      softmax_n<1>(acc, f, n, pr);
      pv_i4(stage, pr[0], first, ntok);
    } else {
      scores(stage, acc[0]);
      softmax_n<1>(acc, f, n, pr);
      pv(stage, pr[0], first, ntok);
    }
  }

  // Two consecutive blocks of one sequence as one 32-token step: four independent q·Kᵀ chains,
  // one maximum and one rescale check for both, then both P·V products.
  __device__ __forceinline__ void block2(const uint8_t* s0, int f0, int n0, const uint8_t* s1, int f1, int n1) {
    float acc[2][4], pr[2][4];
    const int f[2] = {f0, f1}, n[2] = {n0, n1};
    if constexpr (I4) {
      scores_i4(s0, acc[0]);
      scores_i4(s1, acc[1]);
      softmax_n<2>(acc, f, n, pr);
      pv_i4(s0, pr[0], f0, n0);
      pv_i4(s1, pr[1], f1, n1);
    } else {
      scores(s0, acc[0]);
      scores(s1, acc[1]);
      softmax_n<2>(acc, f, n, pr);
      pv(s0, pr[0], f0, n0);
      pv(s1, pr[1], f1, n1);
    }
  }

  // d index of accumulator element (mt, e): e = 0,1 -> row t4; e = 2,3 -> row t4 + 8.
  __device__ __forceinline__ int dim_of(int mt, int upper) const {
    if constexpr (QUANT) return mt * 16 + 2 * t4 + upper;
    return mt * 16 + t4 + 8 * upper;
  }

  // Emit this warp's state for sequence s (global index).
  __device__ void flush(int s, size_t slot, bool direct) {
    if constexpr (I4) {
      // every token's part of cz, then o[dim][head] -= cz[group of dim][head]
#pragma unroll
      for (int g = 0; g < 4; ++g)
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int mask = 4; mask <= 16; mask <<= 1) cz[g][c] += __shfl_xor_sync(0xffffffffu, cz[g][c], mask);
#pragma unroll
      for (int mt = 0; mt < KT; ++mt) {
        o[mt][0] -= cz[mt >> 1][0];
        o[mt][1] -= cz[mt >> 1][1];
        o[mt][2] -= cz[mt >> 1][0];
        o[mt][3] -= cz[mt >> 1][1];
      }
    }
    float lt0 = l[0], lt1 = l[1];
#pragma unroll
    for (int mask = 4; mask <= 16; mask <<= 1) {
      lt0 += __shfl_xor_sync(0xffffffffu, lt0, mask);
      lt1 += __shfl_xor_sync(0xffffffffu, lt1, mask);
    }
    const int c0 = 2 * tq;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int c = c0 + half;
      if (c >= p.G) continue;
      const int hq = h_kv * p.G + c;
      const float lt = half ? lt1 : lt0;
      if (direct) {
        const float inv = (bad || !(lt > 0.f)) ? 0.f : vsc / lt;
        __nv_bfloat16* orow = p.out + (static_cast<size_t>(s) * p.H_q + hq) * D;
#pragma unroll
        for (int mt = 0; mt < KT; ++mt) {
          orow[dim_of(mt, 0)] = __float2bfloat16_rn(o[mt][half] * inv);
          orow[dim_of(mt, 1)] = __float2bfloat16_rn(o[mt][2 + half] * inv);
        }
      } else {
        float* row = p.partials + ((slot * p.nbs + j) * p.H_q + hq) * static_cast<size_t>(D + 4);
        if (!bad && lt > 0.f) {
#pragma unroll
          for (int mt = 0; mt < KT; ++mt) {
            row[dim_of(mt, 0)] = o[mt][half] * vsc;
            row[dim_of(mt, 1)] = o[mt][2 + half] * vsc;
          }
        }
        if (t4 == 0) {
          row[D] = half ? m[1] : m[0];
          row[D + 1] = bad ? -1.f : lt;
        }
      }
    }
  }

  __device__ void flush_empty(size_t slot) {
    if (t4 != 0) return;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int c = 2 * tq + half;
      if (c >= p.G) continue;
      float* row = p.partials + ((slot * p.nbs + j) * p.H_q + h_kv * p.G + c) * static_cast<size_t>(D + 4);
      row[D] = kNegInf;
      row[D + 1] = 0.f;
    }
  }
};

// ------------------------------------------------------------------------------------
// Producer: streams the CTA's blocks into the stage ring.  Every lane owns one block of the
// current 32-block chunk: its table entry is loaded one chunk ahead and its stage metadata is
// packed once when the chunk becomes current, so a stage costs one shuffle, one shared store and
// one TMA per box.  A block takes one box per tensor: the whole head rows of the group's heads for
// the block's 16 slots, head-major.  (Measured, issuing a box costs about 90 cycles whatever its
// size, so fewer, larger boxes keep the producer ahead of HBM.)  INT4 stages take four boxes per
// block: K and V codes of all the group's heads (128-byte rows of two heads), then K and V group
// parameters.  With per-token K scales a third box per block carries the block's [16 slots][hg
// heads] scales.  Run by a warp of its own, or (INT4) by consumer warp 0 between its blocks.
// ------------------------------------------------------------------------------------
template <int KIND>
struct Producer {
  static constexpr int kOps = KIND == 2 ? 4 : (KIND == 3 ? 3 : 2);  // boxes per block
  // Where the CTA's list lives: sequences [seq_base, seq_base + nseq), entries [u0, u1).
  struct Range {
    int seq_base, nseq, u0, u1;
  };
  // what persists from stage to stage: the current 32-block chunk (first entry `base`), this
  // lane's table entries of it and of the next chunk, its block's metadata, the chunk's live and
  // append-wait masks, and whether the append has been waited for
  int base, cur_pb, nxt_pb;
  int4 my_meta;
  unsigned live_mask, wait_mask;
  bool waited;

  // logical block of list entry u of sequence s (the visited blocks start at the window)
  static __device__ __forceinline__ int logical(const DecodeParams& p, const Smem& sm, int s, int u) {
    return sm.los[s] / PA_BLOCK_SIZE + (u - sm.cum[s]);
  }
  static __device__ __forceinline__ int load_entry(const DecodeParams& p, const Smem& sm, const Range& r, int u) {
    if (u >= r.u1) return -1;
    const int s = find_seq(sm.cum, r.nseq, u);
    return p.block_tables[static_cast<size_t>(r.seq_base + s) * p.max_blocks + logical(p, sm, s, u)];
  }

  __device__ __forceinline__ void init(const DecodeParams& p, const Smem& sm, const Range& r, int lane, bool step) {
    waited = !step;
    base = r.u0;
    cur_pb = load_entry(p, sm, r, base + lane);
    nxt_pb = load_entry(p, sm, r, base + 32 + lane);
    pack(p, sm, r, lane, step);
  }

  __device__ __forceinline__ void pack(const DecodeParams& p, const Smem& sm, const Range& r, int lane, bool step) {
    const int u = base + lane;
    const bool valid = u < r.u1;
    const int s = valid ? find_seq(sm.cum, r.nseq, u) : 0;
    const int lb = valid ? logical(p, sm, s, u) : 0;
    const bool bad = valid && (cur_pb < 0 || cur_pb >= p.num_blocks);
    if (bad) set_error(p.err, PA_EFLAG_BAD_BLOCK_ID);
    // first attended token of the block: sinks and positions before the window are skipped
    const int first =
        valid ? min(PA_BLOCK_SIZE, max(0, max(p.num_sink, sm.los[s]) - lb * PA_BLOCK_SIZE)) : 0;
    my_meta = valid ? make_int4(s, first, min(PA_BLOCK_SIZE, sm.ctxs[s] - lb * PA_BLOCK_SIZE), bad ? 1 : 0)
                    : make_int4(-1, 0, 0, 1);
    live_mask = __ballot_sync(0xffffffffu, valid && !bad);
    // blocks that receive this step's appended token (the append's position of the sequence)
    const int ap = (valid && step) ? p.append_pos[r.seq_base + s] : -1;
    wait_mask = __ballot_sync(0xffffffffu, ap >= 0 && ap / PA_BLOCK_SIZE == lb);
  }

  // Fill the stage of iteration k (its previous use must have been released).
  __device__ __forceinline__ void issue(const DecodeParams& p, const Smem& sm, const Range& r, int lane, bool step,
                                        int hgi, int k, const CUtensorMap* tmK, const CUtensorMap* tmV,
                                        const CUtensorMap* tmKp, const CUtensorMap* tmVp) {
    const int S = p.stages, nbs = p.nbs;
    int i = k * nbs - (base - r.u0);
    if (i >= 32) {
      base += 32;
      i -= 32;
      cur_pb = nxt_pb;
      nxt_pb = load_entry(p, sm, r, base + 32 + lane);
      pack(p, sm, r, lane, step);
    }
    // this lane's op: block jj of the stage, tensor (and parameters) of the box
    const int my_jj = lane / kOps, my_op = lane - my_jj * kOps;
    const int st = k % S;
    const unsigned stage_bits = (1u << nbs) - 1u;
    const int pb = __shfl_sync(0xffffffffu, cur_pb, (i + my_jj) & 31);
    const unsigned live = (live_mask >> i) & stage_bits;  // i + nbs <= 32 since nbs divides 32
    if (!waited && ((wait_mask >> i) & stage_bits)) {   // a block the append writes: wait for it
      grid_dep_wait();
      waited = true;
    }
    if (lane >= i && lane < i + nbs) sm.meta[st * nbs + (lane - i)] = my_meta;
    if (lane == 0) {
      const uint32_t bytes = __popc(live) * static_cast<uint32_t>(p.block_tx);
      if (bytes) mbar_arrive_expect_tx(&sm.full[st], bytes);
      else mbar_arrive(&sm.full[st]);
    }
    __syncwarp();
    if (lane < nbs * kOps && ((live >> my_jj) & 1u)) {
      const uint64_t policy = l2_evict_first_policy();
      uint8_t* stage = sm.stages + static_cast<size_t>(st) * p.stage_bytes + static_cast<size_t>(my_jj) * p.block_bytes;
      if constexpr (KIND == 2) {
        const int t = my_op & 1, prm = my_op >> 1;
        tma_load_3d(stage + (prm ? 2 * p.hg * 1024 + t * p.hg * 256 : t * p.hg * 1024),
                    prm ? (t ? tmVp : tmKp) : (t ? tmV : tmK), &sm.full[st], 0, prm ? hgi * p.hg : hgi * (p.hg >> 1),
                    pb * PA_BLOCK_SIZE, policy);
      } else if (KIND == 3 && my_op == 2) {  // the block's per-token K scales
        tma_load_2d(stage + 2 * p.hg * p.nc * kTileBytes, tmKp, &sm.full[st], hgi * p.hg, pb * PA_BLOCK_SIZE, policy);
      } else {  // K (op 0) or V (op 1): every head of the group, head-major
        tma_load_4d(stage + static_cast<size_t>(my_op) * p.hg * p.nc * kTileBytes, my_op ? tmV : tmK, &sm.full[st], 0,
                    0, pb * PA_BLOCK_SIZE, hgi * p.hg, policy);
      }
    }
  }

  // The grid must not complete before the append it overlaps (a decode step).
  __device__ __forceinline__ void finish() {
    if (!waited) grid_dep_wait();
  }
};

// Wait (bounded) until the copies of iterations [from, to) have landed in their stages.
__device__ __forceinline__ void drain_copies(const Smem& sm, int S, int from, int to, int lane, int32_t* err) {
  for (int k = max(from, to - S); k < to; ++k) {
    if (!mbar_wait(&sm.full[k % S], static_cast<uint32_t>(k / S) & 1u)) {
      if (lane == 0) set_error(err, PA_EFLAG_TIMEOUT);
    }
  }
}

template <int D, int KIND, int MAXW>
__global__ void __launch_bounds__((MAXW + 1) * 32, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmKp, const __grid_constant__ CUtensorMap tmVp,
                  const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  const Smem sm = carve(smem_raw, p);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nthreads = blockDim.x;
  // The merge kernel may be scheduled now; it waits for this grid before reading its output.
  grid_dep_launch_dependents();
  // This kernel may have been launched while the previous kernel of the stream still runs
  // (programmatic dependent launch); whatever that kernel is, it may have produced any input
  // read below (q, context lengths, tables, the cache), so wait for it first.  What overlaps is
  // the launch and the CTA set-up.  In a decode step the previous kernel is the append of one
  // token per sequence (append_pos), which writes only the block holding each new position: the
  // producer waits before loading such a block, so the append runs alongside the streaming of
  // every other block, and every CTA waits before it leaves, so that this grid never completes
  // before the append.
  const bool step = p.append_pos != nullptr;
  if (!step) grid_dep_wait();

  // ---- this CTA's range [u0, u1) of the (sequence, logical block) list ----
  int hgi, seq_base, nseq, u0, u1;
  if (p.mode == 0) {
    hgi = blockIdx.y;
    seq_base = 0;
    nseq = p.B;
    const bool reporter = blockIdx.x == 0 && blockIdx.y == 0;
    // exclusive scan of per-sequence block counts (every CTA computes it for itself)
    const int per = (p.B + nthreads - 1) / nthreads;
    const int lo = min(p.B, tid * per), hi = min(p.B, lo + per);
    int local = 0;
    for (int i = lo; i < hi; ++i) {
      const int ctx = p.context_lens[i];
      const int nb = seq_span(p, i, ctx);
      if (nb < 0 && reporter) set_error(p.err, PA_EFLAG_CTX_OVERFLOW);
      local += max(nb, 0);
    }
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    if (lane == 31) sm.scratch[warp] = incl;
    __syncthreads();
    if (tid == 0) {
      int run = 0;
      for (int w = 0; w < nthreads / 32; ++w) {
        const int t = sm.scratch[w];
        sm.scratch[w] = run;
        run += t;
      }
      sm.cum[0] = 0;
    }
    __syncthreads();
    int run = sm.scratch[warp] + incl - local;
    for (int i = lo; i < hi; ++i) {
      const int ctx = p.context_lens[i];
      const int nb = seq_span(p, i, ctx);
      run += max(nb, 0);
      sm.cum[i + 1] = run;
      sm.ctxs[i] = nb < 0 ? 0 : ctx;
      sm.los[i] = nb < 0 ? 0 : seq_lo(p, i, ctx);
    }
    __syncthreads();
    const int T = sm.cum[p.B];
    if (reporter) {
      for (int i = tid; i <= p.B; i += nthreads) p.ws_meta[i] = sm.cum[i];
      if (tid == 0) p.ws_meta[p.B + 1] = T;
    }
    const int W = (T + gridDim.x - 1) / gridDim.x;
    u0 = blockIdx.x * W;
    u1 = min(T, u0 + W);
    if (T == 0 || u0 >= u1) {
      if (step) grid_dep_wait();
      return;
    }
  } else {
    hgi = blockIdx.z;
    seq_base = blockIdx.y;
    nseq = 1;
    const int ctx = p.context_lens[seq_base];
    const int nb = seq_span(p, seq_base, ctx);
    if (nb < 0 && blockIdx.x == 0 && blockIdx.z == 0 && tid == 0) set_error(p.err, PA_EFLAG_CTX_OVERFLOW);
    const int nbv = max(nb, 0);
    if (tid == 0) {
      sm.cum[0] = 0;
      sm.cum[1] = nbv;
      sm.ctxs[0] = nb < 0 ? 0 : ctx;
      sm.los[0] = nb < 0 ? 0 : seq_lo(p, seq_base, ctx);
    }
    u0 = blockIdx.x * p.ppb;
    u1 = min(nbv, u0 + p.ppb);
    if (u0 >= u1) {
      if (step) grid_dep_wait();
      return;
    }
  }

  if (tid == 0) {
    for (int i = 0; i < p.stages; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], p.warps_c);
    }
    fence_mbar_init();
  }
  __syncthreads();

  const int S = p.stages, nbs = p.nbs;
  const int n_iters = (u1 - u0 + nbs - 1) / nbs;
  const typename Producer<KIND>::Range range{seq_base, nseq, u0, u1};
  if (warp == p.warps_c) {
    // ------------------------------- producer warp -------------------------------
    Producer<KIND> pr;
    pr.init(p, sm, range, lane, step);
    int k = 0;
    for (; k < n_iters; ++k) {
      if (!mbar_wait(&sm.empty[k % S], (static_cast<uint32_t>(k / S) & 1u) ^ 1u)) {
        if (lane == 0) set_error(p.err, PA_EFLAG_TIMEOUT);
        break;
      }
      pr.issue(p, sm, range, lane, step, hgi, k, &tmK, &tmV, &tmKp, &tmVp);
    }
    // do not leave while a copy into this CTA's shared memory may still be in flight
    drain_copies(sm, S, 0, k, lane, p.err);
    pr.finish();  // nor before the append of this step has completed
    return;
  }
  if (warp > p.warps_c) return;

  // ------------------------------- consumers -------------------------------
  const int j = warp / p.hg;
  const int h_loc = warp - j * p.hg;
  Consumer<D, KIND> c(p, lane, hgi * p.hg + h_loc, j, h_loc);
  const int s_first = find_seq(sm.cum, nseq, u0);
  const int s_last = find_seq(sm.cum, nseq, u1 - 1);
  const int cta = blockIdx.x;
  auto slot_of = [&](int s_rel) -> size_t {
    const int s = seq_base + s_rel;
    return p.mode == 0 ? static_cast<size_t>(s + cta) : static_cast<size_t>(s) * p.max_parts + cta;
  };
  auto covers = [&](int s_rel) -> bool { return sm.cum[s_rel] >= u0 && sm.cum[s_rel + 1] <= u1; };
  int cur = s_first;
  bool q_loaded = false;
  for (int k = 0; k < n_iters; ++k) {
    const int st = k % S;
    const uint32_t ph = static_cast<uint32_t>(k / S) & 1u;
    if (!mbar_wait(&sm.full[st], ph)) {
      if (lane == 0) set_error(p.err, PA_EFLAG_TIMEOUT);
      return;
    }
    const int u = u0 + k * nbs + j;
    bool paired = false;
    if (u < u1) {
      const int4 mt = sm.meta[st * nbs + j];
      if (mt.x != cur) {
        c.flush(seq_base + cur, slot_of(cur), p.direct_ok && covers(cur));
        for (int s = cur + 1; s < mt.x; ++s) c.flush_empty(slot_of(s));
        cur = mt.x;
        c.reset();
        q_loaded = false;
      }
      if (!q_loaded) {
        c.load_q(seq_base + cur);
        q_loaded = true;
      }
      if (mt.w) {
        c.bad = true;
      } else {
        const uint8_t* stage = sm.stages + static_cast<size_t>(st) * p.stage_bytes;
        if constexpr (MAXW <= 8) {
          // one block per stage: take the next stage too when its block belongs to the same
          // sequence, and run both as one 32-token step (every warp decides alike: the
          // metadata is the stage's).  Only with 4 or more stages, so that holding two still
          // leaves the copies room ahead (measured: with 3 stages of 64 KiB it is slower); wider
          // CTAs lack the registers for it.
          if (nbs == 1 && S >= 4 && k + 1 < n_iters) {
            const int st1 = (k + 1) % S;
            if (!mbar_wait(&sm.full[st1], static_cast<uint32_t>((k + 1) / S) & 1u)) {
              if (lane == 0) set_error(p.err, PA_EFLAG_TIMEOUT);
              return;
            }
            const int4 mt1 = sm.meta[st1];
            if (mt1.x == mt.x && !mt1.w) {
              c.block2(stage, mt.y, mt.z, sm.stages + static_cast<size_t>(st1) * p.stage_bytes, mt1.y, mt1.z);
              paired = true;
            }
          }
        }
        if (!paired) c.block(stage, mt.y, mt.z);
      }
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&sm.empty[st]);
      if (paired) mbar_arrive(&sm.empty[(k + 1) % S]);
    }
    if (paired) ++k;
  }
  c.flush(seq_base + cur, slot_of(cur), p.direct_ok && covers(cur) && q_loaded);
  for (int s = cur + 1; s <= s_last; ++s) c.flush_empty(slot_of(s));
}

// ------------------------------------------------------------------------------------
// Merge: out = Σ_p e^{m_p - M} o_p / Σ_p e^{m_p - M} l_p (plus the bf16 sink tokens).
// WPR = 1: one warp per (sequence, query head).  WPR = 4, for launches with few (sequence, head)
// rows: four warps per row, each merging a quarter of the partials (the first also the sinks),
// combined through shared memory by the same log-sum-exp rule.  CH partials are loaded per
// round: 8, or 16 when a shared prefix adds its rows (one round for both kinds).
// ------------------------------------------------------------------------------------
template <int D, int WPR, int CH>
__global__ void __launch_bounds__(128) merge_kernel(const DecodeParams p, int grid_x) {
  constexpr int E = D / 32;  // dims per lane
  const int s = blockIdx.x;
  const int wid = threadIdx.x >> 5;
  const int h = WPR == 1 ? blockIdx.y * 4 + wid : blockIdx.y;
  const int part = WPR == 1 ? 0 : wid;  // this warp's share of the row's partials
  const int lane = threadIdx.x & 31;
  if (h >= p.H_q) return;  // (WPR = 4: h is the CTA's, so the CTA leaves together)
  const int h_kv = h / p.G;
  // Every input is read after the wait: this launch may begin while the decode kernel (and, through
  // it, whatever kernel wrote q or the context lengths) still runs; the wait covers them all.
  grid_dep_wait();  // the decode kernel's partials and prefix sums are complete from here on
  // the row's extent in the balanced split does not depend on the context length: its loads go
  // out together with it (one round trip before the partials, not two)
  int cs = 0, ce = 0, T = 0;
  if (p.mode == 0) {
    cs = p.ws_meta[s];
    ce = p.ws_meta[s + 1];
    T = p.ws_meta[p.B + 1];
  }
  const int ctx = p.context_lens[s];
  const int nb = seq_span(p, s, ctx);
  // sink positions inside the attended range [seq_lo, ctx)
  const int sink_lo = seq_lo(p, s, ctx);
  // partial rows of a shared prefix attended apart (only when this sequence has one)
  const int n_x = (nb < 0 || !shares_prefix(p, s)) ? 0 : p.n_extra;
  const int n_sink = (nb < 0 || part != 0) ? 0 : min(p.num_sink, ctx);
  float qv[E];
  if (n_sink > sink_lo) {
    const __nv_bfloat16* qrow = p.q + (static_cast<size_t>(s) * p.H_q + h) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) qv[e] = __bfloat162float(qrow[e]);
  }
  __nv_bfloat16* orow = p.out + (static_cast<size_t>(s) * p.H_q + h) * D;

  int c_first = 0, c_last = -1;
  if (nb > 0) {
    if (p.mode == 0) {
      const int W = (T + grid_x - 1) / grid_x;
      c_first = cs / W;
      c_last = (ce - 1) / W;
    } else {
      c_last = (nb + p.ppb - 1) / p.ppb - 1;
    }
    if (p.direct_ok && c_first == c_last) return;  // the main kernel wrote this row
  }
  const int n_own = (c_last - c_first + 1) * p.nbs;  // this call's own partials, then the prefix's
  const int n_parts = n_own + n_x;
  const int share = (n_parts + WPR - 1) / WPR;
  const int i_begin = min(n_parts, part * share), i_end = min(n_parts, i_begin + share);
  auto row_of = [&](int i) -> const float* {
    if (i >= n_own)
      return p.extra + ((static_cast<size_t>(s) * p.n_extra + (i - n_own)) * p.H_q + h) * static_cast<size_t>(D + 4);
    const int c = c_first + i / p.nbs, jj = i % p.nbs;
    const size_t slot = p.mode == 0 ? static_cast<size_t>(s + c) : static_cast<size_t>(s) * p.max_parts + c;
    return p.partials + ((slot * p.nbs + jj) * p.H_q + h) * static_cast<size_t>(D + 4);
  };

  // Partials are merged CH at a time: lane i holds partial i's (m, l), every lane loads its E
  // dims of all CH partials in the same round, and rows of empty partials (never written) are
  // masked out by their zero weight through a select, never multiplied.
  float M = kNegInf, L = 0.f;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  bool bad = false;
  for (int base = i_begin; base < i_end; base += CH) {
    const int n = min(CH, i_end - base);
    float mi = kNegInf, li = 0.f;
    if (lane < n) {
      const float* r = row_of(base + lane);
      mi = r[D];
      li = r[D + 1];
    }
    float v[CH][E];
#pragma unroll
    for (int j = 0; j < CH; ++j) {
      if (j < n) {
        const float* r = row_of(base + j) + lane * E;
        if constexpr (E == 4) {
          const float4 t = *reinterpret_cast<const float4*>(r);
          v[j][0] = t.x; v[j][1] = t.y; v[j][2] = t.z; v[j][3] = t.w;
        } else {
          const float2 t = *reinterpret_cast<const float2*>(r);
          v[j][0] = t.x; v[j][1] = t.y;
        }
      }
    }
    bad = bad || li < 0.f;
    float mc = li > 0.f ? mi : kNegInf;
#pragma unroll
    for (int mask = 1; mask < 32; mask <<= 1) mc = warp_max_xor(mc, mask);
    const float newM = fmaxf(M, mc);
    if (newM == kNegInf) continue;
    const float sc = ex2(M - newM);
    L *= sc;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] *= sc;
    M = newM;
    const float wi = li > 0.f ? ex2(mi - M) : 0.f;
    float wl = wi * li;
#pragma unroll
    for (int mask = 1; mask < 32; mask <<= 1) wl += __shfl_xor_sync(0xffffffffu, wl, mask);
    L += wl;
#pragma unroll
    for (int j = 0; j < CH; ++j) {
      const float wj = __shfl_sync(0xffffffffu, wi, j);
      if (j < n) {
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] += wj != 0.f ? wj * v[j][e] : 0.f;
      }
    }
  }
  bad = __any_sync(0xffffffffu, bad);

  for (int t = sink_lo; t < n_sink; ++t) {  // bf16 sink tokens join the merge as single-token partials
    const size_t off = ((static_cast<size_t>(s) * p.num_sink + t) * p.H_kv + h_kv) * D + lane * E;
    float dot = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) dot += qv[e] * __bfloat162float(p.k_sink[off + e]);
#pragma unroll
    for (int mask = 1; mask < 32; mask <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, mask);
    const float st = dot * p.scale_log2;
    const float newM = fmaxf(M, st);
    const float sc = ex2(M - newM), w = ex2(st - newM);
    L = L * sc + w;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = acc[e] * sc + w * __bfloat162float(p.v_sink[off + e]);
    M = newM;
  }
  if constexpr (WPR > 1) {
    // the warps' (M, L, acc) -> one row: weights e^{M_w - max M}, warps without a partial weigh 0
    __shared__ float sh_m[WPR], sh_l[WPR], sh_acc[WPR][D];
    __shared__ int sh_bad[WPR];
    if (lane == 0) {
      sh_m[wid] = M;
      sh_l[wid] = L;
      sh_bad[wid] = bad ? 1 : 0;
    }
#pragma unroll
    for (int e = 0; e < E; ++e) sh_acc[wid][lane * E + e] = acc[e];
    __syncthreads();
    if (wid != 0) return;
    float Mt = kNegInf;
#pragma unroll
    for (int w = 0; w < WPR; ++w) Mt = fmaxf(Mt, sh_m[w]);
    L = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    bad = false;
#pragma unroll
    for (int w = 0; w < WPR; ++w) {
      bad = bad || sh_bad[w] != 0;
      if (sh_m[w] == kNegInf) continue;
      const float sc = ex2(sh_m[w] - Mt);
      L += sc * sh_l[w];
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] += sc * sh_acc[w][lane * E + e];
    }
  }
  const float inv = (bad || nb < 0 || !(L > 0.f)) ? 0.f : 1.f / L;
#pragma unroll
  for (int e = 0; e < E; ++e) orow[lane * E + e] = __float2bfloat16_rn(acc[e] * inv);
}

// ------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------
struct Plan {
  int hg, n_hg, nc, nbs, warps_c, threads, stages;
  int mode, ppb, max_parts, grid_x;
  int stage_bytes, block_bytes, block_tx;
  size_t smem_bytes, meta_bytes, ws_bytes, n_slots;
};


pa_status make_plan(const pa_cache_desc* d, int max_ctx, int partition_size, Plan* pl) {
  pa_status st = validate_desc(d);
  if (st != PA_OK) return st;
  if (max_ctx < 0 || partition_size < 0 || partition_size % PA_BLOCK_SIZE != 0) return PA_ERR_INVALID_ARG;
  const bool int4 = is_int4(d), tok = has_token_scales(d);
  const int e = dtype_bytes(d->k_dtype);
  const int row_bytes = int4 ? d->head_dim / 2 : d->head_dim * e;  // 64, 128 or 256
  pl->nc = int4 ? 1 : row_bytes / 128;
  // per-token K scales travel as a [16 slots][hg heads] fp32 box: hg x 4 bytes a multiple of 16
  int hg = 1;
  for (int c = 1; c <= d->num_kv_heads; ++c)
    if (d->num_kv_heads % c == 0 && c * row_bytes <= PA_GROUP_BYTES && (!int4 || (c % 2 == 0 && c <= PA_I4_MAX_HG)) &&
        (!tok || c % 4 == 0))
      hg = c;
  if (int4 && hg % 2 != 0) return PA_ERR_UNSUPPORTED;
  if (tok && hg % 4 != 0) return PA_ERR_UNSUPPORTED;
  pl->hg = hg;
  pl->n_hg = d->num_kv_heads / hg;
  // Blocks per stage: a power of two, so that a stage never straddles the 32-entry chunks in
  // which the producer warp resolves table entries (one lane per block).
  int nbs = std::max(1, (int4 ? PA_I4_WARPS : 8) / hg);
  while (32 % nbs != 0) --nbs;
  pl->nbs = nbs;
  pl->warps_c = hg * pl->nbs;
  if (pl->warps_c > kMaxConsumerWarps) return PA_ERR_UNSUPPORTED;
  pl->threads = (pl->warps_c + 1) * 32;
  // int4 block: K and V codes (hg x 1 KiB each) and group parameters (hg x 256 B each); a
  // per-token block: K and V tiles, then the K scales padded to 1 KiB, so that the next block's
  // swizzled tiles stay 1024-byte aligned
  pl->block_tx = int4 ? 2560 * hg : 2 * hg * pl->nc * kTileBytes + (tok ? 64 * hg : 0);
  pl->block_bytes = tok ? 2 * hg * pl->nc * kTileBytes + (64 * hg + 1023) / 1024 * 1024 : pl->block_tx;
  pl->stage_bytes = pl->nbs * pl->block_bytes;
  const int B = d->num_seqs;
  if (B > 65535) return PA_ERR_UNSUPPORTED;  // grid.y of the fixed-partition launch
  if (partition_size == 0 && B <= kAutoMaxSeqs) {
    pl->mode = 0;
    pl->ppb = 0;
    pl->max_parts = 0;
    // one wave: every head group gets an equal share of the resident CTAs
    const int sms = sm_count_current();
    if (sms <= 0) return PA_ERR_CUDA;
    pl->grid_x = std::max(1, sms * PA_CTAS_PER_SM / pl->n_hg);
    pl->n_slots = static_cast<size_t>(B) + pl->grid_x;
    pl->meta_bytes = ((static_cast<size_t>(B) + 2) * 4 + 255) / 256 * 256;
  } else {
    const int part = partition_size ? partition_size : kFixedFallbackPartition;
    pl->mode = 1;
    pl->ppb = part / PA_BLOCK_SIZE;
    int max_blk = (max_ctx + PA_BLOCK_SIZE - 1) / PA_BLOCK_SIZE;
    // a window of W positions spans at most ceil((W-1)/16) + 1 blocks
    if (d->sliding_window > 0) max_blk = std::min(max_blk, (d->sliding_window + 14) / PA_BLOCK_SIZE + 1);
    pl->max_parts = std::max(1, (max_blk + pl->ppb - 1) / pl->ppb);
    pl->grid_x = pl->max_parts;
    pl->n_slots = static_cast<size_t>(B) * pl->max_parts;
    pl->meta_bytes = 256;
  }
  const size_t kSmemLimit = smem_limit(PA_CTAS_PER_SM);
  const size_t cum_ints = pl->mode == 0 ? (3 * static_cast<size_t>(B) + 1) : 4;  // cum, ctxs, los
  const size_t fixed_bytes = 1024 + (cum_ints + 32) * 4;
  const size_t per_stage = pl->stage_bytes + 16 + static_cast<size_t>(pl->nbs) * 16;
  if (fixed_bytes + 2 * per_stage > kSmemLimit) return PA_ERR_UNSUPPORTED;
  pl->stages = static_cast<int>(std::min<size_t>(kMaxStages, (kSmemLimit - fixed_bytes) / per_stage));
  pl->smem_bytes = fixed_bytes + pl->stages * per_stage;
  const size_t partial_bytes =
      pl->n_slots * pl->nbs * static_cast<size_t>(d->num_q_heads) * (d->head_dim + 4) * sizeof(float);
  pl->ws_bytes = pl->meta_bytes + partial_bytes;
  return PA_OK;
}

template <int D, int KIND>
pa_status launch(const Plan& pl, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mkp,
                 const CUtensorMap& mvp, const DecodeParams& p, cudaStream_t stream) {
  // 9-warp CTAs get the register budget of a 288-thread launch; wider ones a 416-thread (INT4
  // only: four warps per scheduler, 128 registers) or a 544-thread one
  auto kern = decode_kernel<D, KIND, kMaxConsumerWarps>;
  if (pl.warps_c <= 8) {
    kern = decode_kernel<D, KIND, 8>;
  } else if constexpr (KIND == 2) {
    if (pl.warps_c <= 12) kern = decode_kernel<D, KIND, 12>;
  }
  if (!ensure_dynamic_smem(reinterpret_cast<const void*>(kern), pl.smem_bytes)) return PA_ERR_CUDA;
  const dim3 grid = p.mode == 0 ? dim3(pl.grid_x, pl.n_hg, 1) : dim3(pl.max_parts, p.B, pl.n_hg);
  // Both kernels may start while their predecessor drains (the decode prologue overlaps the
  // append; the merge launch overlaps the decode tail); each waits before reading its inputs.
  if (launch_overlapped(kern, grid, dim3(pl.threads), pl.smem_bytes, stream, mk, mv, mkp, mvp, p) != PA_OK)
    return PA_ERR_CUDA;
  // few (sequence, head) rows for the SMs (long contexts, small batches): four warps per row
  if (static_cast<long long>(p.B) * p.H_q < 4LL * std::max(1, sm_count_current()))
    return launch_overlapped(merge_kernel<D, 4, 8>, dim3(p.B, p.H_q), dim3(128), 0, stream, p, pl.grid_x);
  if (p.n_extra > 0)
    return launch_overlapped(merge_kernel<D, 1, 16>, dim3(p.B, (p.H_q + 3) / 4), dim3(128), 0, stream, p, pl.grid_x);
  return launch_overlapped(merge_kernel<D, 1, 8>, dim3(p.B, (p.H_q + 3) / 4), dim3(128), 0, stream, p, pl.grid_x);
}

}  // namespace
}  // namespace pa

extern "C" size_t pa_decode_workspace_size(const pa_cache_desc* desc, int max_context_len,
                                           int partition_size) {
  pa::Plan pl;
  if (pa::make_plan(desc, max_context_len, partition_size, &pl) != PA_OK) return 0;
  return pl.ws_bytes;
}

namespace pa {
namespace {
// The prefix part of pa_decode_attention_shared, already enqueued: flags and rows as DecodeParams'.
struct SharedPart {
  const int32_t* flags;
  const float* extra;
  int shared_len;
  int n_extra;
};

// pa_decode_attention, the attention half of pa_decode_step (append_pos non-null) and the
// decode half of pa_decode_attention_shared (shared non-null).
pa_status decode_attention_impl(const pa_cache_desc* desc, void* out, const void* q, const void* k_cache,
                                const void* v_cache, const int32_t* block_tables, const int32_t* context_lens,
                                int max_context_len, float scale, int partition_size, void* workspace,
                                size_t workspace_bytes, int32_t* err_flag, void* stream, const int32_t* append_pos,
                                const SharedPart* shared = nullptr) {
  pa::Plan pl;
  pa_status st = pa::make_plan(desc, max_context_len, partition_size, &pl);
  if (st != PA_OK) return st;
  if (desc->num_seqs == 0) return PA_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !workspace)
    return PA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache) |
       reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 15u)
    return PA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return PA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return PA_ERR_INVALID_ARG;
  if (workspace_bytes < pl.ws_bytes) return PA_ERR_WORKSPACE_TOO_SMALL;

  const int e = pa::dtype_bytes(desc->k_dtype);
  const long long slots = static_cast<long long>(desc->num_blocks) * PA_BLOCK_SIZE;
  const bool int4 = pa::is_int4(desc);
  CUtensorMap mk, mv, mkp, mvp;
  if (int4) {
    // codes: 128-byte rows of two heads; parameters: 16-byte rows of one head
    const size_t po = pa::int4_params_offset(desc);
    if (!pa::encode_cache_map(&mk, k_cache, 1, desc->num_kv_heads / 2, pl.hg / 2, slots) ||
        !pa::encode_cache_map(&mv, v_cache, 1, desc->num_kv_heads / 2, pl.hg / 2, slots) ||
        !pa::encode_param_map(&mkp, static_cast<const uint8_t*>(k_cache) + po, desc->num_kv_heads, pl.hg, slots) ||
        !pa::encode_param_map(&mvp, static_cast<const uint8_t*>(v_cache) + po, desc->num_kv_heads, pl.hg, slots))
      return PA_ERR_CUDA;
  } else {
    if (!pa::encode_cache_map_heads(&mk, k_cache, e, desc->num_kv_heads, pl.nc, pl.hg, slots) ||
        !pa::encode_cache_map_heads(&mv, v_cache, e, desc->num_kv_heads, pl.nc, pl.hg, slots))
      return PA_ERR_CUDA;
    mkp = mk;  // unused by the bf16 and per-head 8-bit kernels
    mvp = mv;
    if (pa::has_token_scales(desc) &&
        !pa::encode_scale_map(&mkp, static_cast<const uint8_t*>(k_cache) + pa::token_scales_offset(desc),
                              desc->num_kv_heads, pl.hg, slots))
      return PA_ERR_CUDA;
  }

  pa::DecodeParams p;
  p.B = desc->num_seqs;
  p.H_q = desc->num_q_heads;
  p.H_kv = desc->num_kv_heads;
  p.G = desc->num_q_heads / desc->num_kv_heads;
  p.num_blocks = desc->num_blocks;
  p.max_blocks = desc->max_blocks_per_seq;
  p.num_sink = desc->num_sink;
  p.window = desc->sliding_window;
  p.max_ctx = max_context_len;
  p.hg = pl.hg;
  p.nc = pl.nc;
  p.nbs = pl.nbs;
  p.stages = pl.stages;
  p.warps_c = pl.warps_c;
  p.mode = pl.mode;
  p.ppb = pl.ppb;
  p.max_parts = pl.max_parts;
  // a row that one CTA covers is written by it, unless a shared prefix's rows are still to come
  p.direct_ok = (pl.nbs == 1 && desc->num_sink == 0 && !shared) ? 1 : 0;
  p.stage_bytes = pl.stage_bytes;
  p.block_bytes = pl.block_bytes;
  p.block_tx = pl.block_tx;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.k_scales = desc->k_scales;
  p.v_scales = desc->v_scales;
  p.k_sink = static_cast<const __nv_bfloat16*>(desc->k_sink);
  p.v_sink = static_cast<const __nv_bfloat16*>(desc->v_sink);
  p.ws_meta = static_cast<int32_t*>(workspace);
  p.partials = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + pl.meta_bytes);
  p.err = err_flag;
  p.append_pos = append_pos;
  p.shared_flags = shared ? shared->flags : nullptr;
  p.extra = shared ? shared->extra : nullptr;
  p.shared_len = shared ? shared->shared_len : 0;
  p.n_extra = shared ? shared->n_extra : 0;

  cudaStream_t s = pa::as_stream(stream);
  const bool quant = pa::is_quantized(desc);
  if (desc->head_dim == 128)
    return int4                         ? pa::launch<128, 2>(pl, mk, mv, mkp, mvp, p, s)
           : pa::has_token_scales(desc) ? pa::launch<128, 3>(pl, mk, mv, mkp, mvp, p, s)
           : quant                      ? pa::launch<128, 1>(pl, mk, mv, mkp, mvp, p, s)
                                        : pa::launch<128, 0>(pl, mk, mv, mkp, mvp, p, s);
  return pa::launch<64, 0>(pl, mk, mv, mkp, mvp, p, s);
}
}  // namespace
}  // namespace pa

extern "C" pa_status pa_decode_attention(const pa_cache_desc* desc, void* out, const void* q,
                                         const void* k_cache, const void* v_cache,
                                         const int32_t* block_tables, const int32_t* context_lens,
                                         int max_context_len, float scale, int partition_size,
                                         void* workspace, size_t workspace_bytes, int32_t* err_flag,
                                         void* stream) {
  return pa::decode_attention_impl(desc, out, q, k_cache, v_cache, block_tables, context_lens, max_context_len,
                                   scale, partition_size, workspace, workspace_bytes, err_flag, stream, nullptr);
}

extern "C" pa_status pa_decode_step(const pa_cache_desc* desc, void* out, const void* q, void* k_cache,
                                    void* v_cache, const void* k_new, const void* v_new,
                                    const int32_t* block_tables, const int32_t* positions,
                                    const int32_t* context_lens, int max_context_len, float scale,
                                    int partition_size, void* workspace, size_t workspace_bytes,
                                    int32_t* err_flag, void* stream) {
  // every argument of the attention half is checked before anything is enqueued
  pa::Plan pl;
  pa_status st = pa::make_plan(desc, max_context_len, partition_size, &pl);
  if (st != PA_OK) return st;
  if (desc->num_seqs == 0) return PA_OK;
  if (!positions || !workspace || !out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
    return PA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache) |
       reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 15u)
    return PA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) || !std::isfinite(scale)) return PA_ERR_INVALID_ARG;
  if (workspace_bytes < pl.ws_bytes) return PA_ERR_WORKSPACE_TOO_SMALL;
  st = pa_kv_append(desc, k_cache, v_cache, k_new, v_new, block_tables, positions, err_flag, stream);
  if (st != PA_OK) return st;
  return pa::decode_attention_impl(desc, out, q, k_cache, v_cache, block_tables, context_lens, max_context_len,
                                   scale, partition_size, workspace, workspace_bytes, err_flag, stream, positions);
}

// ------------------------------------------------------------------------------------
// Shared-prefix decode: the prefix kernel (shared_prefix.cu), then the decode kernel from each
// member's first position past the prefix, its merge folding the prefix rows in.
// ------------------------------------------------------------------------------------
namespace pa {
namespace {
struct SharedLayout {
  size_t flags_off, extra_off, total;
};

bool shared_layout(const pa_cache_desc* desc, int max_context_len, int partition_size, int shared_len,
                   Plan* pl, SharedLayout* lay) {
  if (make_plan(desc, max_context_len, partition_size, pl) != PA_OK) return false;
  if (shared_len < 0 || shared_len % PA_BLOCK_SIZE != 0 || shared_len > max_context_len) return false;
  auto up = [](size_t b) { return (b + 255) / 256 * 256; };
  const size_t B = static_cast<size_t>(desc->num_seqs);
  lay->flags_off = up(pl->ws_bytes);
  lay->extra_off = lay->flags_off + up(B * sizeof(int32_t));
  lay->total = lay->extra_off + B * shared_prefix_chunks(shared_len) * static_cast<size_t>(desc->num_q_heads) *
                                    (desc->head_dim + 4) * sizeof(float);
  return true;
}
}  // namespace
}  // namespace pa

extern "C" size_t pa_decode_shared_workspace_size(const pa_cache_desc* desc, int max_context_len,
                                                  int partition_size, int shared_len) {
  pa::Plan pl;
  pa::SharedLayout lay;
  return pa::shared_layout(desc, max_context_len, partition_size, shared_len, &pl, &lay) ? lay.total : 0;
}

extern "C" pa_status pa_decode_attention_shared(const pa_cache_desc* desc, void* out, const void* q,
                                                const void* k_cache, const void* v_cache,
                                                const int32_t* block_tables, const int32_t* context_lens,
                                                int max_context_len, float scale, int partition_size,
                                                const int32_t* shared_seqs, int n_shared, int shared_len,
                                                void* workspace, size_t workspace_bytes, int32_t* err_flag,
                                                void* stream) {
  pa::Plan pl;
  pa_status st = pa::make_plan(desc, max_context_len, partition_size, &pl);
  if (st != PA_OK) return st;
  if (pa::is_quantized(desc) || desc->num_sink > 0 || desc->sliding_window > 0) return PA_ERR_UNSUPPORTED;
  pa::SharedLayout lay;
  if (!pa::shared_layout(desc, max_context_len, partition_size, shared_len, &pl, &lay)) return PA_ERR_INVALID_ARG;
  if (n_shared < 0 || n_shared > desc->num_seqs || (n_shared > 0 && !shared_seqs)) return PA_ERR_INVALID_ARG;
  if (desc->num_seqs == 0) return PA_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !workspace)
    return PA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache) |
       reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 15u)
    return PA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) || !std::isfinite(scale)) return PA_ERR_INVALID_ARG;
  if (workspace_bytes < lay.total) return PA_ERR_WORKSPACE_TOO_SMALL;
  if (n_shared == 0 || shared_len == 0)  // nothing to share: the plain decode
    return pa::decode_attention_impl(desc, out, q, k_cache, v_cache, block_tables, context_lens, max_context_len,
                                     scale, partition_size, workspace, workspace_bytes, err_flag, stream, nullptr);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* flags = reinterpret_cast<int32_t*>(ws + lay.flags_off);
  float* extra = reinterpret_cast<float*>(ws + lay.extra_off);
  st = pa::launch_shared_prefix(desc, q, k_cache, v_cache, block_tables, context_lens, max_context_len, scale,
                                shared_seqs, n_shared, shared_len, flags, extra, err_flag, pa::as_stream(stream));
  if (st != PA_OK) return st;
  const pa::SharedPart part{flags, extra, shared_len, pa::shared_prefix_chunks(shared_len)};
  return pa::decode_attention_impl(desc, out, q, k_cache, v_cache, block_tables, context_lens, max_context_len,
                                   scale, partition_size, workspace, lay.flags_off, err_flag, stream, nullptr, &part);
}

// ------------------------------------------------------------------------------------
// Allocation-free variant: the same kernels with their scratch in a static device array.
// ------------------------------------------------------------------------------------
namespace pa {
namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB on every device that loads the library
constexpr int kMaxDevices = 64;

// Loaded with the module on each device and held until the process exits.  Kernels may name
// it directly; host code must not (the host symbol is only a stand-in for the device address).
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
struct ScratchAddr {
  unsigned long long ctx_id;  // the context the address belongs to
  void* ptr;
};
ScratchAddr g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array in the current context of the current device.  It is looked
// up (cudaGetSymbolAddress, with the device current) the first time a context is seen and kept
// under that context's id, so a new context on the device (after cudaDeviceReset, or another
// context made current) gets a fresh lookup rather than an address of a module that is gone.
pa_status static_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  const unsigned long long id = current_ctx_id();
  if (id != 0 && g_scratch_addr[dev].ptr && g_scratch_addr[dev].ctx_id == id) {
    *out = g_scratch_addr[dev].ptr;
    return PA_OK;
  }
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || !ptr) return PA_ERR_CUDA;
  // the lookup makes the device's primary context current if none was: ask again
  const unsigned long long id_now = id != 0 ? id : current_ctx_id();
  g_scratch_addr[dev] = {id_now, id_now != 0 ? ptr : nullptr};
  *out = ptr;
  return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_decode_attention_noalloc(const pa_cache_desc* desc, void* out, const void* q,
                                                 const void* k_cache, const void* v_cache,
                                                 const int32_t* block_tables, const int32_t* context_lens,
                                                 int max_context_len, float scale, int partition_size,
                                                 int32_t* err_flag, void* stream) {
  pa::Plan pl;
  const pa_status st = pa::make_plan(desc, max_context_len, partition_size, &pl);
  if (st != PA_OK) return st;
  if (pl.ws_bytes > pa::kStaticScratchBytes) return PA_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const pa_status ss = pa::static_scratch(&scratch);
  if (ss != PA_OK) return ss;
  return pa_decode_attention(desc, out, q, k_cache, v_cache, block_tables, context_lens, max_context_len,
                             scale, partition_size, scratch, pa::kStaticScratchBytes, err_flag, stream);
}

/*
 * pa.h — paged KV-cache decode attention on NVIDIA GB300 (sm_103a), C ABI.
 *
 * What the library computes, and where the pages define it:
 *   - The KV cache is a pool of fixed-size physical blocks of 16 token slots; every
 *     sequence owns a block table mapping logical block pos/16 to a physical block, and
 *     a token's flat slot is table[pos/16]*16 + pos%16
 *     ("KV Cache 的显存账本：PagedAttention 与连续批处理", §四, the locate() sketch).
 *   - A decode step appends the new token's K and V at its slot (untitled article at
 *     ldpk.cn/news/58971, §2.3), copying a shared block first when other sequences still
 *     reference it (显存账本 §四; "大模型推理KV Cache显存优化：从PagedAttention到AI内存系统
 *     演进", §3.2 reference counts and copy-on-write).
 *   - It then computes one query per head against every cached token:
 *     out = softmax(q·Kᵀ · scale) · V with scale = 1/sqrt(d_head) (ldpk §2.1), where query
 *     head h reads KV head h / G, G = num_q_heads / num_kv_heads (显存账本 §二, GQA).
 *   - Optional 8-bit caches store K as FP8 E4M3 and V as INT8 with one fp32 scale per KV
 *     head, and keep the first num_sink positions of every sequence in bf16 (显存账本 §七).
 *   - Optionally K keeps one fp32 scale per token's head row instead of one per KV head
 *     (PA_FP8_E4M3_TOKEN; ldpk §5.2: K develops outlier channels, so per-tensor or per-head
 *     scales fail on long contexts and finer granularity is needed).
 *   - Optional 4-bit caches store K and V as INT4 codes with a scale and a zero point per
 *     group of 32 dims of every token's head row (ldpk §5.2: int4 keeps a scale and a zero
 *     point, about 0.55-0.65 bytes per element; per-token granularity against K's outlier
 *     channels).
 *   - Optional sliding window of W tokens (ldpk §5.3): each query attends only the most
 *     recent W positions, its own included, and blocks that fall wholly before the window
 *     go back to the pool (pa_bm_slide_window), so a sequence holds O(W) cache.
 *   - Sequences that share a prompt prefix point their tables at one copy of its whole blocks
 *     (AI内存系统 §3.1, §3.3); pa_decode_attention_shared attends those blocks once for all of
 *     them and merges that part with each sequence's own positions.
 *
 * Memory layout (all row-major, all device memory unless stated otherwise):
 *   k_cache, v_cache  [num_blocks * 16][num_kv_heads][head_dim]  element type per k/v_dtype
 *                     (slot-major: one physical block is one contiguous chunk holding all
 *                     KV heads of its 16 slots)
 *   block_tables      int32 [num_seqs][max_blocks_per_seq]; entries past a sequence's last
 *                     logical block are ignored and may be -1
 *   context_lens      int32 [num_seqs]  tokens attended, including the new token
 *   positions         int32 [num_seqs]  slot position of the appended token (= old length)
 *   q, out            bf16  [num_seqs][num_q_heads][head_dim]
 *   k_new, v_new      bf16  [rows][num_kv_heads][head_dim]
 *   k_sink, v_sink    bf16  [num_seqs][num_sink][num_kv_heads][head_dim]
 *   k_scales,v_scales fp32  [num_kv_heads]
 *   INT4 pools        [num_blocks * 16][num_kv_heads][64] code bytes, then (at byte offset
 *                     num_blocks*16*num_kv_heads*64 of the same allocation)
 *                     [num_blocks * 16][num_kv_heads][4] uint32 group parameters; see PA_INT4.
 *   PA_FP8_E4M3_TOKEN K pools  [num_blocks * 16][num_kv_heads][head_dim] E4M3 codes, then (at
 *                     byte offset num_blocks*16*num_kv_heads*head_dim of the same allocation)
 *                     [num_blocks * 16][num_kv_heads] fp32 scales, one per token's head row.
 *
 * Conventions:
 *   - The caller owns every buffer; apart from the static scratch array behind
 *     pa_decode_attention_noalloc, the library allocates no device memory and keeps no
 *     per-call state.  Calls are stream-ordered on the given stream (a cudaStream_t passed
 *     as void*; NULL is the legacy default stream) and return after enqueueing.
 *   - Errors the host can see (null pointers, unsupported shapes, small workspace) are
 *     returned synchronously and nothing is enqueued.
 *   - Errors in device data (a block id out of range, a context longer than the table or
 *     than max_context_len, a sequence index out of range) set bits in the optional device
 *     word *err_flag (atomicOr, never cleared by the library), skip the affected work and,
 *     for attention, write zeros to the affected output rows.  No kernel traps.
 *   - Every wait inside a kernel is bounded (about two seconds); on expiry the kernel sets
 *     PA_EFLAG_TIMEOUT and returns instead of hanging.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PA_BLOCK_SIZE 16

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,          /* null pointer, negative size, inconsistent shapes */
  PA_ERR_UNSUPPORTED = 2,          /* valid but not implemented (head_dim, block size, dtypes) */
  PA_ERR_WORKSPACE_TOO_SMALL = 3,  /* workspace_bytes < pa_decode_workspace_size(...) */
  PA_ERR_CUDA = 4,                 /* a CUDA runtime/driver call failed (launch, attribute) */
  PA_ERR_OUT_OF_BLOCKS = 5         /* block manager: no free physical block */
} pa_status;

typedef enum {
  PA_BF16 = 0,
  PA_FP8_E4M3 = 1, /* OCP FP8 E4M3, round-to-nearest-even, saturating at +-448 */
  PA_INT8 = 2,     /* symmetric int8, round-half-even, clamped to [-127, 127] */
  PA_INT4 = 3,     /* asymmetric 4-bit codes with a bf16 scale and a zero point per 32 dims:
                    * for each group x[0..31] of a token's head row (head_dim 128: 4 groups)
                    *   lo = min(0, min x), hi = max(0, max x)           (fp32)
                    *   s  = bf16(rn((hi - lo) / 15)), 1.0 if that is +-0
                    *   z  = clamp(rint(-lo / s), 0, 15)
                    *   q  = clamp(rint(x / s) + z, 0, 15)               (IEEE fp32 divisions)
                    * and a code decodes to s * (q - z).  Parameter word of a group: bits 0-15
                    * the bf16 scale, bits 16-23 z, bits 24-31 zero.  Code bytes of one
                    * (slot, head) row, little-endian:
                    *   K: uint32 word 4c + g (c, g in 0..3) holds dim 32g + 8c + i in bits
                    *      4i .. 4i+3 (i in 0..7);
                    *   V: byte 8r + m (r, m in 0..7) holds dim 16m + r in bits 0-3 and dim
                    *      16m + r + 8 in bits 4-7.
                    * 64 code bytes + 16 parameter bytes per row: 0.625 bytes per element. */
  PA_FP8_E4M3_TOKEN = 4 /* K only: OCP FP8 E4M3 codes with one fp32 scale per (token, KV head)
                         * row: s = max|x| / 448 over the row's head_dim values in IEEE fp32 (NaN
                         * elements left out of the maximum, which starts from 0; a row whose
                         * maximum is 0 takes s = 1), code = e4m3(x / s) rounded and saturated as
                         * PA_FP8_E4M3, value = code * s.  The scale follows the codes in the same
                         * allocation (see the layout above): head_dim + 4 bytes per row. */
} pa_dtype;

/* Bits OR-ed into *err_flag by the kernels. */
#define PA_EFLAG_BAD_BLOCK_ID 1 /* a table entry or copy pair outside [0, num_blocks) */
#define PA_EFLAG_CTX_OVERFLOW 2 /* position/context beyond max_blocks_per_seq*16 or max_context_len */
#define PA_EFLAG_BAD_SEQ 4      /* a token's sequence index outside [0, num_seqs) */
#define PA_EFLAG_TIMEOUT 8      /* a bounded in-kernel wait expired */

/* One layer's cache description.  Supported: block_size == 16; head_dim 64 or 128;
 * num_q_heads % num_kv_heads == 0 with G = num_q_heads/num_kv_heads <= 8;
 * (k_dtype, v_dtype) = (PA_BF16, PA_BF16), (PA_FP8_E4M3, PA_INT8), (PA_FP8_E4M3_TOKEN, PA_INT8)
 * or (PA_INT4, PA_INT4), the 8-bit and 4-bit ones with head_dim 128, the 4-bit one with an even
 * num_kv_heads, the per-token one with num_kv_heads a multiple of 4.  k_scales/v_scales are
 * required for 8-bit dtypes (k_scales is ignored with PA_FP8_E4M3_TOKEN) and ignored otherwise.
 * num_sink > 0 keeps positions < num_sink in k_sink/v_sink (bf16) for any dtype.
 * sliding_window = W > 0 restricts every query to the W most recent positions (ldpk §5.3):
 * a decode query of a ctx-token sequence reads positions max(0, ctx-W) .. ctx-1, a prefill
 * query at position p reads max(0, p-W+1) .. p.  Table entries of logical blocks that lie
 * wholly before those positions are never read (they may be -1 after pa_bm_slide_window);
 * sink positions take part only when they fall inside the window.  0 = whole context. */
typedef struct {
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int head_dim;
  int block_size;
  int num_blocks;
  int max_blocks_per_seq;
  pa_dtype k_dtype;
  pa_dtype v_dtype;
  const float* k_scales; /* device fp32 [num_kv_heads], this layer */
  const float* v_scales; /* device fp32 [num_kv_heads], this layer */
  void* k_sink;          /* device bf16 [num_seqs][num_sink][num_kv_heads][head_dim] or NULL */
  void* v_sink;
  int num_sink;          /* 0 when unused */
  int sliding_window;    /* W > 0: attend the last W positions only; 0 = whole context */
} pa_cache_desc;

/* Human-readable name of a status code (static string, never NULL). */
const char* pa_status_string(pa_status status);

/* ---------------------------------------------------------------------------------
 * Append (decode): write the new token of every sequence into its slot.
 * ldpk §2.3 (write the new K and V at the current length); 显存账本 §四 (locate());
 * 显存账本 §七 (per-head scales, K in FP8 and V in INT8, sinks kept in bf16).
 *
 * Row s writes k_new[s], v_new[s] at position positions[s] of sequence s:
 *   positions[s] < 0                   -> row skipped (padding), no flag;
 *   positions[s] < num_sink            -> bf16 copy into k_sink[s][pos], v_sink[s][pos]; the
 *                                         paged slot is not touched;
 *   pos/16 >= max_blocks_per_seq       -> PA_EFLAG_CTX_OVERFLOW, row skipped;
 *   table entry outside [0,num_blocks) -> PA_EFLAG_BAD_BLOCK_ID, row skipped;
 *   otherwise the slot table[s][pos/16]*16 + pos%16 receives the bf16 bits unchanged, or
 *   for 8-bit caches code = round(x / scale[kv_head]) with the division in IEEE fp32 (with
 *   PA_FP8_E4M3_TOKEN the K row's own scale, stored beside it), or for 4-bit caches the
 *   PA_INT4 codes and group parameters of the row.
 * The caller makes the slot writable first (pa_bm_prepare_step + pa_block_copy) and passes
 * context_lens = positions + 1 to the following pa_decode_attention.
 * Host errors: PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_CUDA. */
pa_status pa_kv_append(const pa_cache_desc* desc, void* k_cache, void* v_cache,
                       const void* k_new, const void* v_new,
                       const int32_t* block_tables, const int32_t* positions,
                       int32_t* err_flag, void* stream);

/* Bulk append (prefill / chunked fill): num_tokens rows, row i going to sequence
 * token_seq[i] at position token_pos[i]; same rules as pa_kv_append, plus
 * PA_EFLAG_BAD_SEQ for token_seq[i] outside [0, num_seqs).  Rows must target distinct
 * slots.  k_new/v_new are bf16 [num_tokens][num_kv_heads][head_dim]. */
pa_status pa_kv_append_tokens(const pa_cache_desc* desc, void* k_cache, void* v_cache,
                              const void* k_new, const void* v_new, int num_tokens,
                              const int32_t* token_seq, const int32_t* token_pos,
                              const int32_t* block_tables, int32_t* err_flag, void* stream);

/* ---------------------------------------------------------------------------------
 * Copy-on-write block copy: for each pair i, physical block dst = src_dst_pairs[2i+1]
 * receives every byte of block src = src_dst_pairs[2i] in both k_cache and v_cache
 * (显存账本 §四 copy only at the fork; AI内存系统 §3.2 copy before writing a shared block).
 * src_dst_pairs: device int32 [n_pairs][2].  A pair with an id outside [0, num_blocks)
 * sets PA_EFLAG_BAD_BLOCK_ID and is skipped.  Destinations must be distinct and must not
 * be a source of the same call.  n_pairs == 0 enqueues nothing. */
pa_status pa_block_copy(const pa_cache_desc* desc, void* k_cache, void* v_cache,
                        const int32_t* src_dst_pairs, int n_pairs,
                        int32_t* err_flag, void* stream);

/* ---------------------------------------------------------------------------------
 * Decode attention over the paged cache (ldpk §2.1 formula; ldpk §4.3: the kernel fetches
 * K and V from non-contiguous places through the block table; 显存账本 §二 GQA).
 *
 * For every sequence s and query head h (KV head h/G), over positions 0..ctx-1 with
 * ctx = context_lens[s]:  out[s][h] = sum_t softmax_t(scale * q[s][h]·K_t) V_t, with
 * fp32 accumulation and the result rounded to bf16.  K_t/V_t are the bf16 values, or
 * code*scale for 8-bit caches, or the sink rows for t < num_sink.  ctx == 0 gives zeros.
 * With desc->sliding_window = W > 0 the positions are max(0, ctx-W) .. ctx-1 instead, and
 * only the table entries of the logical blocks holding them are read.
 *
 * partition_size: 0 = automatic (the cached blocks of all sequences are split evenly over
 * the GPU's SMs; partial results are merged by a second kernel); a positive multiple of 16
 * = fixed context partitions of that many tokens per CTA plus the merge kernel (a value
 * >= max_context_len gives one pass per sequence).
 * max_context_len bounds every context_lens[s] (larger ones set PA_EFLAG_CTX_OVERFLOW
 * and give a zero row).  workspace: device memory of at least
 * pa_decode_workspace_size(desc, max_context_len, partition_size) bytes, 256-byte
 * aligned, used as scratch by this call only (its contents need not be initialised).
 * k_cache and v_cache must be 16-byte aligned.
 * Host errors: PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE_TOO_SMALL,
 * PA_ERR_CUDA. */
size_t pa_decode_workspace_size(const pa_cache_desc* desc, int max_context_len, int partition_size);

pa_status pa_decode_attention(const pa_cache_desc* desc, void* out, const void* q,
                              const void* k_cache, const void* v_cache,
                              const int32_t* block_tables, const int32_t* context_lens,
                              int max_context_len, float scale, int partition_size,
                              void* workspace, size_t workspace_bytes,
                              int32_t* err_flag, void* stream);

/* ---------------------------------------------------------------------------------
 * Decode attention with a shared prompt prefix attended once (AI内存系统 §3.1: requests with the
 * same prefix point their block tables at one copy of its blocks; §3.3: only whole blocks are
 * shared; ldpk §2.1 formula).
 *
 * The result is pa_decode_attention's, up to the order of the fp32 sums.  The first shared_len
 * positions of the listed sequences are attended together: for each KV head and each 128 of
 * those positions, one product takes the queries of all listed sequences (G heads each) against
 * the prefix keys read once, and leaves a softmax partial (running max, sum, unnormalised output)
 * per row; the decode kernel then visits only positions shared_len .. ctx-1 of those sequences,
 * and its merge combines both parts by the log-sum-exp rule.
 *   shared_seqs   device int32 [n_shared], 0 <= n_shared <= num_seqs: the sequences to share; the
 *                 first one's table supplies the prefix blocks.  Duplicates are harmless.
 *   shared_len    a multiple of 16 with 0 <= shared_len <= max_context_len: the prefix length.
 * The list is checked, not trusted: a listed sequence takes the shared part only when its
 * context covers shared_len and its table holds the first listed sequence's physical block for
 * every prefix block; every other sequence is attended in full as by pa_decode_attention.  An
 * entry outside [0, num_seqs) sets PA_EFLAG_BAD_SEQ and is ignored (the first one: nothing is
 * shared); a prefix block id outside [0, num_blocks) sets PA_EFLAG_BAD_BLOCK_ID and zeroes the
 * rows of the sequences that share it.  n_shared == 0 or shared_len == 0 is pa_decode_attention.
 * bf16 caches without sinks or sliding window only (PA_ERR_UNSUPPORTED otherwise), head_dim 64
 * or 128.
 *   workspace     at least pa_decode_shared_workspace_size(desc, max_context_len, partition_size,
 *                 shared_len) bytes, 256-byte aligned, scratch for this call only.  The size is 0
 *                 when an argument is invalid.
 * Other arguments, device errors and host errors as pa_decode_attention. */
size_t pa_decode_shared_workspace_size(const pa_cache_desc* desc, int max_context_len, int partition_size,
                                       int shared_len);

pa_status pa_decode_attention_shared(const pa_cache_desc* desc, void* out, const void* q,
                                     const void* k_cache, const void* v_cache,
                                     const int32_t* block_tables, const int32_t* context_lens,
                                     int max_context_len, float scale, int partition_size,
                                     const int32_t* shared_seqs, int n_shared, int shared_len,
                                     void* workspace, size_t workspace_bytes,
                                     int32_t* err_flag, void* stream);

/* ---------------------------------------------------------------------------------
 * Chunked-prefill (extend) attention over the paged cache (ldpk §2.2: under the causal mask the
 * query of position i attends to positions up to i; ldpk §7: long prompts are prefilled in
 * chunks).  Sequence s contributes the query rows q_start[s] .. q_start[s+1]-1 of q: they are its
 * last n_s = q_start[s+1] - q_start[s] positions, ctx-n_s .. ctx-1 with ctx = context_lens[s],
 * and their K/V must already be in the cache (pa_kv_append_tokens).  The query at position p
 * attends to positions 0..p of its sequence, or max(0, p-W+1) .. p under a sliding window W
 * (desc->sliding_window, ldpk §5.3).
 *   q, out            bf16 [T][num_q_heads][head_dim], T >= q_start[num_seqs]
 *   q_start           device int32 [num_seqs + 1], non-decreasing
 *   max_query_len     bounds every n_s (it sizes the grid)
 * Every cache kind is supported.  bf16 caches without sinks run on the tensor-core paths as they
 * are; 8-bit, per-token-scaled and INT4 caches and caches with sinks (显存账本 §七) are decoded block
 * by block (code times scale as fp32, rounded to bf16; sink positions from the sink buffers) and
 * then take the same bf16 products, so their results carry that extra bf16 rounding of K and V.
 * A sequence with n_s < 0, n_s > ctx, n_s > max_query_len or ctx beyond its table sets
 * PA_EFLAG_CTX_OVERFLOW and gets zero rows; a table entry outside [0, num_blocks) sets
 * PA_EFLAG_BAD_BLOCK_ID and zeroes the rows of every query tile whose keys include it.
 * Host errors: PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_CUDA. */
pa_status pa_prefill_attention(const pa_cache_desc* desc, void* out, const void* q,
                               const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, const int32_t* q_start,
                               const int32_t* context_lens, int max_query_len, float scale,
                               int32_t* err_flag, void* stream);

/* One chunked-prefill step: pa_kv_append_tokens of the chunk's K/V, then pa_prefill_attention,
 * enqueued together (ldpk §7: a chunk's K/V join the cache and its queries attend over it).  The
 * result is what the two calls give one after the other.  What differs is the overlap: on the
 * tensor-core path the attention kernel's set-up (work ranking, query loads) runs while the
 * append does, and only its K/V copies wait for the append.  That is exact because the append
 * writes only the K/V slots of the chunk's tokens, and nothing but those copies reads them.
 *   Arguments: those of pa_kv_append_tokens (k_new, v_new, num_tokens, token_seq, token_pos) and
 *   of pa_prefill_attention, with the same meaning, layouts and rules; out must not overlap
 *   k_new, v_new, token_seq or token_pos.  Every argument is checked before anything is
 *   enqueued.
 * Host errors: those of pa_kv_append_tokens and pa_prefill_attention. */
pa_status pa_prefill_step(const pa_cache_desc* desc, void* out, const void* q, void* k_cache,
                          void* v_cache, const void* k_new, const void* v_new, int num_tokens,
                          const int32_t* token_seq, const int32_t* token_pos,
                          const int32_t* block_tables, const int32_t* q_start,
                          const int32_t* context_lens, int max_query_len, float scale,
                          int32_t* err_flag, void* stream);

/* Chunked-prefill attention with a workspace: the computation, layouts, rules and device errors
 * of pa_prefill_attention, for caches that are decoded (8-bit, per-token-scaled and INT4 caches,
 * and caches with sinks; 显存账本 §七, ldpk §5.2).  Each logical block that the chunk's queries can
 * attend (from the first query's window start to the end of the context) is decoded once, into
 * a bf16 copy in the workspace laid out as a bf16 cache of num_seqs * ceil(max_context_len / 16)
 * blocks (code times scale in fp32 rounded to bf16, sink positions from the sink buffers: the
 * values pa_prefill_attention takes), and the tensor-core kernel of bf16 caches then runs over
 * that copy, instead of every 16-token query tile decoding each block it reads for itself.
 * Results equal pa_prefill_attention's up to the order in which the products are summed.
 *   max_context_len   bounds every context_lens[s]; 0 <= max_context_len <= max_blocks_per_seq*16.
 *                     A sequence with a longer context sets PA_EFLAG_CTX_OVERFLOW and gets zero
 *                     rows.
 *   workspace         device memory of at least pa_prefill_workspace_size(desc, max_context_len)
 *                     bytes, 256-byte aligned, scratch for this call only (its contents need not
 *                     be initialised).
 * pa_prefill_workspace_size returns 0 when the call needs no workspace (a bf16 cache without
 * sinks, head_dim 64, a G that is not a power of two, or more than 2^31 slots in the copy: the
 * call is then pa_prefill_attention, and workspace may be NULL) and when desc or
 * max_context_len is invalid (the call then reports the error).
 * Host errors: those of pa_prefill_attention, PA_ERR_INVALID_ARG for max_context_len out of range
 * or a missing or misaligned workspace, PA_ERR_WORKSPACE_TOO_SMALL. */
size_t pa_prefill_workspace_size(const pa_cache_desc* desc, int max_context_len);

pa_status pa_prefill_attention_ws(const pa_cache_desc* desc, void* out, const void* q,
                                  const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, const int32_t* q_start,
                                  const int32_t* context_lens, int max_query_len, int max_context_len,
                                  float scale, void* workspace, size_t workspace_bytes,
                                  int32_t* err_flag, void* stream);

/* One chunked-prefill step with the workspace path: pa_kv_append_tokens of the chunk's K/V, then
 * pa_prefill_attention_ws, enqueued together (ldpk §7).  The result is what the two calls give
 * one after the other.  Arguments: those of pa_kv_append_tokens and of pa_prefill_attention_ws,
 * with the same meaning, layouts and rules; out must not overlap k_new, v_new, token_seq or
 * token_pos.  Every argument is checked before anything is enqueued.
 * Host errors: those of pa_kv_append_tokens and pa_prefill_attention_ws. */
pa_status pa_prefill_step_ws(const pa_cache_desc* desc, void* out, const void* q, void* k_cache,
                             void* v_cache, const void* k_new, const void* v_new, int num_tokens,
                             const int32_t* token_seq, const int32_t* token_pos,
                             const int32_t* block_tables, const int32_t* q_start,
                             const int32_t* context_lens, int max_query_len, int max_context_len,
                             float scale, void* workspace, size_t workspace_bytes, int32_t* err_flag,
                             void* stream);

/* Allocation-free decode attention.  The pages have no counterpart to this entry point: it is
 * pa_decode_attention for callers that cannot allocate device memory when they call it, for
 * example a plugin running inside a host framework that owns every byte of device memory, a
 * latency-critical path where cudaMalloc/cudaFree could synchronise the device and stall other
 * work, or a caller that has no way to recover from an out-of-memory failure in the middle of a
 * decode step.  It takes the same arguments minus the workspace, and runs the same kernels with
 * their scratch in a static 8 MiB device array that every GPU which loads this library holds
 * until the process exits.
 *   - The first call in a context looks the array's address up (cudaGetSymbolAddress, with that
 *     device current) and keeps it under the context's unique id; make that first call before any
 *     stream capture on the device.  A new context on the device (after cudaDeviceReset, or
 *     another context made current) gets its own lookup on its first call, never an address
 *     kept from an earlier one.
 *   - A problem whose pa_decode_workspace_size() exceeds 8 MiB (8388608 bytes) is rejected
 *     with PA_ERR_WORKSPACE_TOO_SMALL and nothing is enqueued.
 *   - Nothing is allocated: no cudaMalloc, no cudaFree, no allocating library routine.
 *   - Every call on a device shares the array and leaves its contents behind; the kernels write
 *     every scratch byte before reading it, so nothing needs clearing, but calls that overlap on
 *     the GPU (e.g. on two streams at once) race on it: serialise them.
 * Host errors: as pa_decode_attention, plus PA_ERR_CUDA if the address lookup fails. */
pa_status pa_decode_attention_noalloc(const pa_cache_desc* desc, void* out, const void* q,
                                      const void* k_cache, const void* v_cache,
                                      const int32_t* block_tables, const int32_t* context_lens,
                                      int max_context_len, float scale, int partition_size,
                                      int32_t* err_flag, void* stream);

/* One decode step: pa_kv_append of one token per sequence, then pa_decode_attention, enqueued
 * together (显存账本 §四: the step appends the new token's K/V into the sequence's last block and
 * attends over the context; ldpk §4.3).  The result is what the two calls give one after the
 * other.  What differs is the overlap: the attention kernel waits for the append only before it
 * loads a block that holds one of `positions`, so the append runs while every other block
 * streams.  That is exact because the append writes nothing else the attention reads: it writes
 * the K/V (and for 8-bit or INT4 caches the codes and parameters) of slot positions[s], and the
 * bf16 sink rows when positions[s] < num_sink, which the attention reads only after the step's
 * kernels have all waited for the append.
 *   Arguments: those of pa_kv_append (k_new, v_new, positions) and of pa_decode_attention,
 *   with the same meaning, layouts and rules; q, block_tables, positions and context_lens must
 *   not be written by the append (they are not).  Every argument is checked before anything is
 *   enqueued.
 * Host errors: those of pa_kv_append and pa_decode_attention. */
pa_status pa_decode_step(const pa_cache_desc* desc, void* out, const void* q, void* k_cache,
                         void* v_cache, const void* k_new, const void* v_new,
                         const int32_t* block_tables, const int32_t* positions,
                         const int32_t* context_lens, int max_context_len, float scale,
                         int partition_size, void* workspace, size_t workspace_bytes,
                         int32_t* err_flag, void* stream);

/* ---------------------------------------------------------------------------------
 * Host block manager: the physical block pool with a free list and reference counts
 * (显存账本 §四: equal-size blocks, any free one usable; AI内存系统 §3.2: reference counts,
 * recycle at zero, copy-on-write; AI内存系统 §2.3: blocks return to the pool on every exit
 * path).  Host memory only; every function is thread-safe (one internal mutex).
 * Allocation hands out the lowest-numbered free block. */
typedef struct pa_bm pa_bm;

/* NULL if num_blocks <= 0 or block_size <= 0 or on allocation failure. */
pa_bm* pa_bm_create(int num_blocks, int block_size);
void pa_bm_destroy(pa_bm* bm);
/* A free block with refcount 1, or -1 when none is free. */
int pa_bm_alloc(pa_bm* bm);
/* Take a specific free block (refcount 0 -> 1): 0 on success, -1 if not free/invalid. */
int pa_bm_claim(pa_bm* bm, int blk);
/* New refcount, or -1 if blk is not allocated. */
int pa_bm_incref(pa_bm* bm, int blk);
/* New refcount (0 = returned to the free list), or -1 if blk is not allocated. */
int pa_bm_decref(pa_bm* bm, int blk);
int pa_bm_refcount(const pa_bm* bm, int blk); /* 0 for free blocks, -1 if out of range */
int pa_bm_num_free(const pa_bm* bm);
/* dst_row[i] = src_row[i] with incref, for i < n_blocks (prefix sharing). */
pa_status pa_bm_fork(pa_bm* bm, const int32_t* src_row, int32_t* dst_row, int n_blocks);
/* decref row[i] and set it to -1 for i < n_blocks; returns the number of blocks freed
 * (entries already -1 are skipped), or -1 on invalid arguments. */
int pa_bm_release(pa_bm* bm, int32_t* row, int n_blocks);

/* Make the slot of positions[s] writable for every sequence s (host tables, in place):
 *   entry table[s][pos/16] < 0      -> allocate a block and store it (no copy);
 *   refcount(entry) > 1 (shared)    -> allocate dst, decref the shared block, repoint the
 *                                      entry, and emit the pair (src, dst) to cow_pairs;
 *   otherwise                       -> nothing.
 * Rows with positions[s] < 0 are skipped.  cow_pairs: host int32 [num_seqs][2] output,
 * *n_pairs receives the count; *n_changed (may be NULL) receives the number of table
 * entries changed.  On PA_ERR_OUT_OF_BLOCKS the rows handled before the failure keep their
 * changes (and their pairs are reported); PA_ERR_INVALID_ARG for a position beyond the
 * table. */
pa_status pa_bm_prepare_step(pa_bm* bm, int32_t* block_tables, int num_seqs,
                             int max_blocks_per_seq, const int32_t* positions,
                             int32_t* cow_pairs, int* n_pairs, int* n_changed);

/* Sliding-window release (ldpk §5.3: only the most recent W positions are kept, so the cache
 * stays O(W)).  For every sequence s with c = context_lens[s] > window > 0, each logical block
 * lying wholly before position c - window (blocks 0 .. (c-window)/16 - 1) that still holds a
 * physical block is decref-ed (freed at zero; a shared block stays with its other holders)
 * and its host table entry set to -1.  Call it after the attention that used context_lens;
 * later queries of those sequences never reach the released positions.  Entries already -1
 * and sequences with c <= window are left alone.  Returns the number of table entries
 * released, and *n_freed (may be NULL) the number of blocks that went back to the free list;
 * -1 on invalid arguments (nothing changed) or on a table entry the pool does not hold (the
 * sequences before it keep their changes). */
int pa_bm_slide_window(pa_bm* bm, int32_t* block_tables, int num_seqs, int max_blocks_per_seq,
                       const int32_t* context_lens, int window, int* n_freed);

/* ---------------------------------------------------------------------------------
 * Prefix cache ("大模型推理KV Cache显存优化：从PagedAttention到AI内存系统演进", prefix-cache
 * section, and §7.2): which physical blocks of a pool already hold the K/V of a token prefix, so a
 * new request reuses them and computes only what follows.  Host memory only; thread-safe (its
 * own mutex, then the pool's).
 *
 * Block identity: only full 16-token blocks are cached.  Block i of a request is identified by
 *   h_i = SHA-256(h_{i-1} || tokens[16i .. 16i+15] as little-endian int32 || extra_key as
 *                 little-endian uint64),   h_{-1} = SHA-256(salt as little-endian uint64)
 * (FIPS 180-4), so it covers the whole prefix, the request's extra inputs (e.g. an adapter or a
 * multimodal input id in extra_key) and the tenant's cache salt: different salts never share.
 *
 * The cache holds one reference of its own on every registered block (so a cached block survives
 * its request) and orders entries by last use; eviction returns to the pool the least recently
 * used blocks that no sequence holds (refcount 1), deeper blocks first among equally recent ones.
 * A matched block is full and shared, so the pool's copy-on-write keeps it unmodified. */
#define PA_PC_DIGEST_BYTES 32
typedef struct pa_pc pa_pc;

/* Digests of the n_tokens/16 full blocks of a token sequence (a partial tail block gets none)
 * into digests [n_tokens/16][32].  Returns n_tokens/16, or -1 on invalid arguments. */
int pa_pc_block_hashes(const int32_t* tokens, int n_tokens, uint64_t salt, uint64_t extra_key,
                       uint8_t* digests);
/* A cache over pool bm (which must outlive it); capacity = maximum entries, 0 = bounded by the
 * pool only.  NULL on invalid arguments or allocation failure. */
pa_pc* pa_pc_create(pa_bm* bm, int capacity);
/* Drops the cache's references (pa_pc_clear) and frees the cache. */
void pa_pc_destroy(pa_pc* pc);
/* Longest cached leading run of digests[0 .. n_blocks-1]: its physical blocks go to
 * table_row[0 .. n-1], each gains one reference for the request, the entries count as used now.
 * Returns n (0 = no hit), or -1 on invalid arguments.  An engine passes at most
 * (prompt_tokens - 1) / 16 digests so that at least one prompt token is still computed. */
int pa_pc_match(pa_pc* pc, const uint8_t* digests, int n_blocks, int32_t* table_row);
/* Register blocks table_row[0 .. n_blocks-1] (their K/V written) under digests[0 .. n_blocks-1].
 * A new entry takes the cache's own reference; a digest already cached keeps its block and is
 * only marked used.  At capacity, the LRU evictable entry makes room; registration stops when
 * none can.  Returns the number of new entries, or -1 on invalid arguments or on a block the pool
 * does not hold (the entries registered before it stay). */
int pa_pc_insert(pa_pc* pc, const uint8_t* digests, const int32_t* table_row, int n_blocks);
/* Return up to n least recently used entries whose block no sequence holds to the pool; returns
 * how many went, or -1 on invalid arguments. */
int pa_pc_evict(pa_pc* pc, int n);
/* Number of cached entries (-1 for NULL). */
int pa_pc_size(const pa_pc* pc);
/* Drop every entry and the cache's reference on its block; returns the number dropped. */
int pa_pc_clear(pa_pc* pc);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */

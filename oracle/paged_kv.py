"""The oracle: what paged decode attention computes, written out plainly.

Pages cited (title, or address where the page has no title line):
  * "KV Cache 的显存账本：PagedAttention 与连续批处理" (gcssc.sfwss.com kv-cache-budget),
    cited as  显存账本 §一 .. §七
  * "大模型推理KV Cache显存优化：从PagedAttention到AI内存系统演进" (wmrh.cn/news/79784),
    cited as  AI内存系统 §1.1 .. §7.4
  * untitled KV-cache article at ldpk.cn/news/58971, cited as  ldpk §1.1 .. §7
  * untitled memory-planning article at pptc.cn/news/143802, cited as  pptc §3.2 ..
  * "面试官皱眉：KV Cache为什么占显存？PagedAttention解决什么问题？" (yfxerp.com/news/121119),
    cited as  面试官皱眉

Readings taken where the pages are silent (each repeated where it is used):
  * the new token is appended first and then attends to itself (ctx = old_len + 1);
  * cache layout is slot-major: slot = locate(...), element [slot][kv_head][dim];
  * query head h reads KV head h // G (contiguous grouping);
  * e4m3 = OCP FP8 E4M3 (no infinities, max 448), round-to-nearest-even, saturating;
    int8 = symmetric, zero-point 0, range [-127, 127], round-half-even;
  * the quantiser divides in IEEE fp32 (x_fp32 / scale_fp32) before rounding;
  * sink positions (pos < num_sink) live in a separate bf16 buffer and the paged slot
    is left untouched;
  * the block pool hands out the lowest-numbered free block;
  * int4 (ldpk §5.2: int4 stores a scale and a zero point besides the codes, about 0.55-0.65
    bytes per element; K develops outlier channels, so per-tensor scales fail and finer
    granularity is needed): asymmetric 4-bit codes per group of 32 consecutive dims of one
    (token, KV head) row; the group's range [min(0, min x), max(0, max x)] gives
    s = bf16((hi - lo) / 15) (1 if that is 0), z = clamp(rint(-lo / s), 0, 15) and
    q = clamp(rint(x / s) + z, 0, 15), divisions in IEEE fp32; a code decodes to s * (q - z);
    with a bf16 scale and the zero point in one 32-bit word that is 0.625 bytes per element;
  * per-token K scales (ldpk §5.2: K develops outlier channels, so one scale per tensor or per
    head fails on long contexts and finer granularity is needed): "e4m3_tok" K stores E4M3 codes
    with one fp32 scale per (token, KV head), s = max|x| / 448 over the token's head row in IEEE
    fp32 (NaN elements left out of the maximum, an all-zero row takes 1), and codes
    e4m3(x / s); a code decodes to its value times s;
  * sliding window W (ldpk §5.3): the query at position p attends positions
    max(0, p - W + 1) .. p, i.e. the most recent W tokens with itself included, and W = 0
    means no window; a block is freed once all its positions lie before the window of the
    sequence's latest query (the block is the pool's unit, 显存账本 §四).

Everything is numpy; floating point is fp64 except the fp32 quantiser division.
"""

from __future__ import annotations

import heapq
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "BLOCK_SIZE",
    "kv_bytes_per_token",
    "kv_bytes_total",
    "locate",
    "slots_of_sequence",
    "blocks_needed",
    "window_start",
    "bf16_bits_to_f64",
    "f32_to_bf16_bits",
    "E4M3_MAX",
    "INT8_MAX",
    "e4m3_decode",
    "e4m3_encode",
    "e4m3_encode_bruteforce",
    "int8_encode",
    "int8_decode",
    "quantize_row",
    "e4m3_token_scale",
    "quantize_token_rows",
    "INT4_GROUP",
    "int4_encode_group",
    "int4_encode_row",
    "int4_decode_row",
    "BlockPool",
    "PagedKVCache",
    "ContiguousKVCache",
    "decode_attention",
    "decode_attention_partials",
    "merge_partials",
    "decode_attention_split",
    "softmax_weights",
    "prefill_attention",
]

# 显存账本 §四: "典型 16 个 token 一块" — the typical block holds 16 tokens.
BLOCK_SIZE = 16


# ----------------------------------------------------------------------------------
# Capacity arithmetic
# ----------------------------------------------------------------------------------
def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int, dtype_bytes: float) -> float:
    """Bytes of K and V cached per token over the whole model.

    ldpk §3.1 and 显存账本 §一: the factor 2 is one copy each of K and V, multiplied by
    the number of layers, the number of *KV* heads (not attention heads), the head
    dimension and the bytes per element.
    """
    return 2 * num_layers * num_kv_heads * head_dim * dtype_bytes


def kv_bytes_total(num_layers, num_kv_heads, head_dim, dtype_bytes, seq_len, batch):
    """Total cache bytes: the per-token figure times sequence length times batch (ldpk §3.1)."""
    return kv_bytes_per_token(num_layers, num_kv_heads, head_dim, dtype_bytes) * seq_len * batch


def blocks_needed(num_tokens: int, block_size: int = BLOCK_SIZE) -> int:
    """Physical blocks a sequence of ``num_tokens`` occupies: ceil(n / block_size).

    显存账本 §四: internal fragmentation is at most one block (the tail block).
    """
    return -(-int(num_tokens) // block_size)


# ----------------------------------------------------------------------------------
# Logical -> physical mapping
# ----------------------------------------------------------------------------------
def locate(block_table_row, pos: int, block_size: int = BLOCK_SIZE) -> int:
    """Flat physical slot of logical position ``pos``.

    显存账本 §四 (the locate() sketch): the logical block is pos // block_size, the
    block table maps it to a physical block number, and the slot is
    physical * block_size + pos % block_size.  The sketch has no bounds check; the
    oracle raises on a position beyond the table or an unassigned (negative) entry.
    """
    lb = pos // block_size
    if pos < 0 or lb >= len(block_table_row):
        raise IndexError(f"position {pos} outside the block table")
    pb = int(block_table_row[lb])
    if pb < 0:
        raise IndexError(f"logical block {lb} has no physical block")
    return pb * block_size + pos % block_size


def slots_of_sequence(block_table_row, ctx: int, block_size: int = BLOCK_SIZE) -> np.ndarray:
    """locate() applied to every position 0..ctx-1 of one sequence, as an index array."""
    return np.array([locate(block_table_row, p, block_size) for p in range(ctx)], dtype=np.int64)


# ----------------------------------------------------------------------------------
# Number formats
# ----------------------------------------------------------------------------------
def bf16_bits_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float64 values (bf16 is the top half of fp32)."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def f32_to_bf16_bits(x) -> np.ndarray:
    """fp32 values -> bf16 bits, round to nearest, ties to even; NaN -> 0x7FC0 (sign kept)."""
    x = np.asarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    upper = u >> np.uint64(16)
    lower = u & np.uint64(0xFFFF)
    round_up = (lower > 0x8000) | ((lower == 0x8000) & ((upper & np.uint64(1)) == 1))
    out = (upper + round_up.astype(np.uint64)).astype(np.uint32)
    nan = np.isnan(x)
    out = np.where(nan, (upper & np.uint64(0x8000)).astype(np.uint32) | np.uint32(0x7FC0), out)
    return out.astype(np.uint16)


# OCP FP8 E4M3 ("E4M3FN"): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, no
# infinities, S.1111.111 is NaN, so the largest finite magnitude is 1.75 * 2^8 = 448.
E4M3_MAX = 448.0
INT8_MAX = 127


def e4m3_decode(codes) -> np.ndarray:
    """e4m3 code (uint8) -> float64 value, from the format definition."""
    c = np.asarray(codes).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((e == 0xF) & ((c & 0x7) == 0x7), np.nan, mag)
    return sign * mag


# The 127 finite non-negative magnitudes, in code order 0x00..0x7E.  Code order is
# value order, and "even code" is "even mantissa" (consecutive codes step the last
# mantissa bit), which is what ties-to-even picks.
_E4M3_MAGNITUDES = e4m3_decode(np.arange(0x7F, dtype=np.uint8))


def e4m3_encode(x) -> np.ndarray:
    """fp32 value -> e4m3 code: round to nearest (ties to the even code), saturate.

    显存账本 §七 and 面试官皱眉 name FP8 for K; the variant (E4M3), saturation at the
    largest finite value and round-to-nearest-even are this oracle's reading.  The sign
    is kept for zero results (negative underflow gives 0x80).  NaN gives 0x7F / 0xFF.
    """
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x).astype(np.float64)
    neg = np.signbit(x)
    idx = np.clip(np.searchsorted(_E4M3_MAGNITUDES, a, side="left"), 1, 0x7E)
    lo, hi = idx - 1, idx
    d_lo = a - _E4M3_MAGNITUDES[lo]
    d_hi = _E4M3_MAGNITUDES[hi] - a
    pick = np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi, np.where(lo % 2 == 0, lo, hi)))
    pick = np.where(a >= E4M3_MAX, 0x7E, pick)  # satfinite, including +-inf
    pick = np.where(np.isnan(x), 0x7F, pick)
    return (pick | (neg.astype(np.int64) << 7)).astype(np.uint8)


def e4m3_encode_bruteforce(x: float) -> int:
    """Reference for the reference: scan all 127 magnitudes for the nearest (small inputs)."""
    xf = float(np.float32(x))
    if np.isnan(xf):
        return 0xFF if np.signbit(np.float32(x)) else 0x7F
    a = abs(xf)
    best, best_d = 0, None
    for code in range(0x7F):
        d = abs(float(_E4M3_MAGNITUDES[code]) - a)
        if best_d is None or d < best_d or (d == best_d and code % 2 == 0):
            best, best_d = code, d
    if a >= E4M3_MAX:
        best = 0x7E
    return best | (0x80 if np.signbit(np.float32(x)) else 0)


def int8_encode(x) -> np.ndarray:
    """fp32 value -> symmetric int8 code: round half to even, clamp to [-127, 127].

    显存账本 §七 names INT8 for V; symmetric with range +-127 and zero-point 0 is this
    oracle's reading.  NaN gives 0.  Written with floor() so that numpy's rint can pin it.
    """
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    f = np.floor(x)
    r = x - f
    f_odd = np.mod(f, 2.0) == 1.0
    q = f + ((r > 0.5) | ((r == 0.5) & f_odd)).astype(np.float64)
    q = np.clip(q, -INT8_MAX, INT8_MAX)
    q = np.where(np.isnan(x), 0.0, q)
    return q.astype(np.int8)


def int8_decode(codes) -> np.ndarray:
    return np.asarray(codes).astype(np.int8).astype(np.float64)


def quantize_row(x_bf16_bits, scale: np.float32, kind: str) -> np.ndarray:
    """One K or V row (bf16 bits) -> codes with one per-head scale.

    The value divided is the fp32 value of the bf16 input, divided by the fp32 scale
    in IEEE fp32 (correctly rounded), then rounded to the code (显存账本 §七: one scale
    per head, not per tensor).
    """
    xf = bf16_bits_to_f64(x_bf16_bits).astype(np.float32)
    e = (xf / np.float32(scale)).astype(np.float32)
    if kind == "e4m3":
        return e4m3_encode(e)
    if kind == "int8":
        return int8_encode(e).view(np.uint8)
    raise ValueError(kind)


def e4m3_token_scale(x_bf16_bits):
    """Per-token K scale of head rows [..., d] (bf16 bits) -> fp32 [...].

    ldpk §5.2: K carries outlier channels, so a scale shared by a whole tensor or head leaves
    most tokens with a fraction of the code range; one scale per token's head row adapts to each
    token.  s = max|x| / 448 (the largest finite E4M3 value) in IEEE fp32, so that the row's
    largest element maps to the top of the code range; NaN elements are left out of the maximum
    (it starts from 0), and a row whose maximum is 0 takes s = 1 (any scale encodes it exactly).
    """
    x = bf16_bits_to_f64(np.asarray(x_bf16_bits, dtype=np.uint16)).astype(np.float32)
    a = np.fmax.reduce(np.abs(x), axis=-1, initial=np.float32(0)).astype(np.float32)
    s = (a / np.float32(E4M3_MAX)).astype(np.float32)
    return np.where(s == 0, np.float32(1), s).astype(np.float32)


def quantize_token_rows(x_bf16_bits):
    """Head rows [..., d] (bf16 bits) -> (E4M3 codes uint8 [..., d], fp32 scales [...]): each row
    is divided by its own per-token scale in IEEE fp32 and rounded to E4M3 (nearest, ties to
    even, saturating), as quantize_row does with a per-head scale."""
    x = np.asarray(x_bf16_bits, dtype=np.uint16)
    sc = e4m3_token_scale(x)
    xf = bf16_bits_to_f64(x).astype(np.float32)
    with np.errstate(invalid="ignore"):  # inf / inf (a row holding an infinity) is NaN, as in IEEE
        e = (xf / sc[..., None]).astype(np.float32)
    return e4m3_encode(e), sc


INT4_GROUP = 32   # dims per scale / zero-point group
INT4_LEVELS = 15  # codes 0 .. 15


def int4_encode_group(x_bf16_bits):
    """Groups of 32 bf16 values [..., 32] -> (codes uint8 [..., 32] in 0..15, bf16 scale bits
    [...], zero points [...]); one group (a 1-D input) gives the scale bits and the zero point
    as Python ints.

    ldpk §5.2: int4 keeps a scale and a zero point per quantisation group; the group here is
    32 consecutive dims of one token's head row (per-token granularity, so an outlier channel
    of another token cannot squeeze this one).  The range always contains 0, so 0 encodes
    exactly (q = z).  Every arithmetic step is IEEE fp32 and the scale is rounded to bf16
    before it is used, so that encoding and decoding use the same stored scale.  Each group is
    encoded on its own; the leading axes only batch independent groups.
    """
    bits = np.asarray(x_bf16_bits, dtype=np.uint16)
    x = bf16_bits_to_f64(bits).astype(np.float32)
    lo = np.minimum(np.float32(0), x.min(axis=-1))
    hi = np.maximum(np.float32(0), x.max(axis=-1))
    s = (np.asarray(hi - lo, dtype=np.float32) / np.float32(INT4_LEVELS)).astype(np.float32)
    sb = f32_to_bf16_bits(s).astype(np.uint16)
    sb = np.where((sb & 0x7FFF) == 0, np.uint16(0x3F80), sb)  # an all-zero group: any scale works, take 1
    sf = bf16_bits_to_f64(sb).astype(np.float32)
    z = np.clip(np.rint((np.asarray(-lo, dtype=np.float32) / sf).astype(np.float32)), 0, INT4_LEVELS)
    q = np.clip(np.rint((x / sf[..., None]).astype(np.float32)) + z[..., None], 0, INT4_LEVELS).astype(np.uint8)
    z = z.astype(np.int64)
    if bits.ndim == 1:
        return q, int(sb), int(z)
    return q, sb, z


def int4_encode_row(x_bf16_bits):
    """Head rows [..., d] -> (codes uint8 [..., d], params uint32 [..., d / 32]) with each params
    word holding its group's bf16 scale in bits 0-15 and its zero point in bits 16-23; the groups
    are dims 32g .. 32g + 31 of each row."""
    x = np.asarray(x_bf16_bits, dtype=np.uint16)
    d = x.shape[-1]
    groups = x.reshape(x.shape[:-1] + (d // INT4_GROUP, INT4_GROUP))
    q, sb, z = int4_encode_group(groups)
    codes = q.reshape(x.shape)
    params = (np.asarray(sb).astype(np.uint32) | (np.asarray(z).astype(np.uint32) << np.uint32(16))).astype(np.uint32)
    return codes, params


def int4_decode_row(codes, params):
    """Codes [..., d] and params [..., d / 32] -> fp64 values s * (q - z)."""
    codes = np.asarray(codes).astype(np.float64)
    params = np.asarray(params, dtype=np.uint32)
    scale = bf16_bits_to_f64((params & 0xFFFF).astype(np.uint16))
    zero = ((params >> 16) & 0xFF).astype(np.float64)
    scale = np.repeat(scale, INT4_GROUP, axis=-1)
    zero = np.repeat(zero, INT4_GROUP, axis=-1)
    return scale * (codes - zero)


# ----------------------------------------------------------------------------------
# Host block pool: free list, reference counts, copy-on-write decision
# ----------------------------------------------------------------------------------
class BlockPool:
    """Fixed-size physical blocks with reference counts.

    显存账本 §四: all blocks have the same size and any free one can be used.
    AI内存系统 §3.2: a shared block carries a reference count; finishing a sequence
    decrements it and the block is recycled only at zero; a sequence that must write
    into a shared block first copies it (copy-on-write).
    Allocation policy (a reading; the pages do not fix one): the lowest-numbered free
    block is handed out first.
    """

    def __init__(self, num_blocks: int, block_size: int = BLOCK_SIZE):
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        self.refcount = np.zeros(self.num_blocks, dtype=np.int64)
        self._free = list(range(self.num_blocks))
        heapq.heapify(self._free)

    # -- primitive operations ------------------------------------------------------
    def num_free(self) -> int:
        return len(self._free)

    def alloc(self) -> int:
        if not self._free:
            return -1
        b = heapq.heappop(self._free)
        self.refcount[b] = 1
        return b

    def claim(self, blk: int) -> bool:
        """Take a specific free block (used to register a pre-placed layout)."""
        if not (0 <= blk < self.num_blocks) or self.refcount[blk] != 0:
            return False
        self._free.remove(blk)
        heapq.heapify(self._free)
        self.refcount[blk] = 1
        return True

    def incref(self, blk: int) -> int:
        if not (0 <= blk < self.num_blocks) or self.refcount[blk] <= 0:
            return -1
        self.refcount[blk] += 1
        return int(self.refcount[blk])

    def decref(self, blk: int) -> int:
        if not (0 <= blk < self.num_blocks) or self.refcount[blk] <= 0:
            return -1
        self.refcount[blk] -= 1
        if self.refcount[blk] == 0:
            heapq.heappush(self._free, blk)
        return int(self.refcount[blk])

    # -- sequence-level operations ---------------------------------------------------
    def fork(self, src_row, n_blocks: int):
        """A new table row sharing the first n_blocks of src_row (prefix sharing)."""
        row = np.full(len(src_row), -1, dtype=np.int64)
        for i in range(n_blocks):
            row[i] = src_row[i]
            self.incref(int(src_row[i]))
        return row

    def release(self, row, n_blocks: int) -> int:
        freed = 0
        for i in range(n_blocks):
            if row[i] >= 0:
                if self.decref(int(row[i])) == 0:
                    freed += 1
                row[i] = -1
        return freed

    def slide_window(self, row, ctx: int, window: int) -> int:
        """Release the blocks of one sequence that no later query can reach.

        ldpk §5.3: under a sliding window of W tokens only the K and V of the most recent W
        positions are kept and older ones are dropped, so the cache stays O(W).  The pool's unit
        is the block (显存账本 §四), so a block goes only when every one of its positions lies
        before ctx - W, the window start of the sequence's latest query.  Its table entry
        becomes -1 and it loses one reference (a shared block stays with its other holders).
        Returns the number of blocks that went back to the free list.
        """
        if window <= 0 or ctx <= window:
            return 0
        freed = 0
        for lb in range((ctx - window) // self.block_size):
            if row[lb] >= 0:
                if self.decref(int(row[lb])) == 0:
                    freed += 1
                row[lb] = -1
        return freed

    def prepare_append(self, row, pos: int):
        """Make the slot of ``pos`` writable for this sequence.

        Returns ("ok",), ("alloc", new) when the logical block had no physical block,
        or ("copy", src, dst) when the block was shared (refcount > 1): a fresh block is
        allocated, the table entry is repointed to it and the shared block loses one
        reference (AI内存系统 §3.2; 显存账本 §四 "只在分叉时才复制").  The caller copies
        the block contents src -> dst before writing.
        """
        lb = pos // self.block_size
        if pos < 0 or lb >= len(row):
            raise IndexError("position outside the table")
        pb = int(row[lb])
        if pb < 0:
            new = self.alloc()
            if new < 0:
                raise MemoryError("block pool exhausted")
            row[lb] = new
            return ("alloc", new)
        if self.refcount[pb] > 1:
            new = self.alloc()
            if new < 0:
                raise MemoryError("block pool exhausted")
            self.decref(pb)
            row[lb] = new
            return ("copy", pb, new)
        return ("ok",)


# ----------------------------------------------------------------------------------
# Cache state
# ----------------------------------------------------------------------------------
@dataclass
class PagedKVCache:
    """One layer's paged K and V pools, stored as codes.

    Layout (a reading: the pages give only the flat slot of locate()):
    ``k[slot][kv_head][dim]`` with slot = physical_block * block_size + offset.
    bf16 pools hold uint16 bit patterns; e4m3 / int8 pools hold uint8 codes; int4 pools hold
    one uint8 code (0..15) per element in natural order plus ``k_params`` / ``v_params``
    [slot][kv_head][dim / 32] uint32 (bf16 scale | zero point << 16); an "e4m3_tok" K pool holds
    E4M3 codes plus ``k_tscale`` [slot][kv_head] fp32, one scale per token's head row.
    ``k_sink`` / ``v_sink`` hold the bf16 rows of positions < num_sink per sequence
    (显存账本 §七: attention-sink tokens keep their original precision).
    """

    num_blocks: int
    num_kv_heads: int
    head_dim: int
    block_size: int = BLOCK_SIZE
    k_dtype: str = "bf16"  # "bf16" | "e4m3" | "e4m3_tok" | "int4"
    v_dtype: str = "bf16"  # "bf16" | "int8" | "int4"
    k_scales: np.ndarray | None = None  # fp32 [num_kv_heads]
    v_scales: np.ndarray | None = None
    num_seqs: int = 0
    num_sink: int = 0
    k: np.ndarray = field(init=False)
    v: np.ndarray = field(init=False)
    k_sink: np.ndarray = field(init=False)
    v_sink: np.ndarray = field(init=False)

    def __post_init__(self):
        n_slots = self.num_blocks * self.block_size
        kt = np.uint16 if self.k_dtype == "bf16" else np.uint8
        vt = np.uint16 if self.v_dtype == "bf16" else np.uint8
        self.k = np.zeros((n_slots, self.num_kv_heads, self.head_dim), dtype=kt)
        self.v = np.zeros((n_slots, self.num_kv_heads, self.head_dim), dtype=vt)
        pshape = (n_slots, self.num_kv_heads, self.head_dim // INT4_GROUP)
        self.k_params = np.zeros(pshape, dtype=np.uint32) if self.k_dtype == "int4" else None
        self.v_params = np.zeros(pshape, dtype=np.uint32) if self.v_dtype == "int4" else None
        self.k_tscale = (np.zeros((n_slots, self.num_kv_heads), dtype=np.float32) if self.k_dtype == "e4m3_tok"
                         else None)
        shape = (self.num_seqs, self.num_sink, self.num_kv_heads, self.head_dim)
        self.k_sink = np.zeros(shape, dtype=np.uint16)
        self.v_sink = np.zeros(shape, dtype=np.uint16)

    def _encode(self, bits, kind, scales):
        """Codes of one token's rows [kv_heads][dim], and its int4 params or per-token scales
        (else None)."""
        if kind == "bf16":
            return np.asarray(bits, dtype=np.uint16), None
        if kind == "e4m3_tok":
            return quantize_token_rows(bits)
        out = np.empty(bits.shape, dtype=np.uint8)
        if kind == "int4":
            params = np.empty((self.num_kv_heads, self.head_dim // INT4_GROUP), dtype=np.uint32)
            for h in range(self.num_kv_heads):
                out[h], params[h] = int4_encode_row(bits[h])
            return out, params
        for h in range(self.num_kv_heads):
            out[h] = quantize_row(bits[h], np.float32(scales[h]), kind)
        return out, None

    def append(self, seq: int, table_row, pos: int, k_bits, v_bits):
        """Write one token's K and V rows (bf16 bits [kv_heads][dim]) at ``pos``.

        ldpk §2.3: each generated token's K and V are written at the current length.
        Paged: the slot is locate(table_row, pos) (显存账本 §四).  Quantised pools store
        the per-head codes (显存账本 §七); sink positions go to the bf16 sink buffer and
        leave the paged slot untouched.
        """
        k_bits = np.asarray(k_bits, dtype=np.uint16)
        v_bits = np.asarray(v_bits, dtype=np.uint16)
        if pos < self.num_sink:
            self.k_sink[seq, pos] = k_bits
            self.v_sink[seq, pos] = v_bits
            return
        slot = locate(table_row, pos, self.block_size)
        self.k[slot], kp = self._encode(k_bits, self.k_dtype, self.k_scales)
        self.v[slot], vp = self._encode(v_bits, self.v_dtype, self.v_scales)
        if kp is not None and self.k_dtype == "e4m3_tok":
            self.k_tscale[slot] = kp
        elif kp is not None:
            self.k_params[slot] = kp
        if vp is not None:
            self.v_params[slot] = vp

    def block_copy(self, src: int, dst: int):
        """Copy-on-write: the destination block receives the source block's bytes."""
        bs = self.block_size
        self.k[dst * bs:(dst + 1) * bs] = self.k[src * bs:(src + 1) * bs]
        self.v[dst * bs:(dst + 1) * bs] = self.v[src * bs:(src + 1) * bs]
        for prm in (self.k_params, self.v_params, self.k_tscale):
            if prm is not None:
                prm[dst * bs:(dst + 1) * bs] = prm[src * bs:(src + 1) * bs]

    def _decode_k(self, codes, heads=None, slots=None):
        if self.k_dtype == "bf16":
            return bf16_bits_to_f64(codes)
        if self.k_dtype == "int4":
            return int4_decode_row(codes, self.k_params[slots])
        if self.k_dtype == "e4m3_tok":
            return e4m3_decode(codes) * self.k_tscale[slots].astype(np.float64)[..., None]
        vals = e4m3_decode(codes)
        sc = np.asarray(self.k_scales, dtype=np.float32).astype(np.float64)
        return vals * (sc if heads is None else sc[heads])[..., :, None]

    def _decode_v(self, codes, heads=None, slots=None):
        if self.v_dtype == "bf16":
            return bf16_bits_to_f64(codes)
        if self.v_dtype == "int4":
            return int4_decode_row(codes, self.v_params[slots])
        vals = int8_decode(codes)
        sc = np.asarray(self.v_scales, dtype=np.float32).astype(np.float64)
        return vals * (sc if heads is None else sc[heads])[..., :, None]

    def gather(self, seq: int, table_row, ctx: int, start: int = 0):
        """K and V of positions start..ctx-1 as contiguous fp64 arrays [ctx - start][kv_heads][dim].

        ldpk §4.3: the attention path fetches K and V from non-contiguous places through
        the block table.  Codes are decoded exactly and multiplied by their per-head
        scale in fp64; sink positions come from the sink buffer.  Positions before
        ``start`` (outside a sliding window) are never looked up, so their table entries may
        already be released (-1).
        """
        n = max(0, ctx - start)
        K = np.zeros((n, self.num_kv_heads, self.head_dim))
        V = np.zeros((n, self.num_kv_heads, self.head_dim))
        for i, p in enumerate(range(start, ctx)):
            if p < self.num_sink:
                K[i] = bf16_bits_to_f64(self.k_sink[seq, p])
                V[i] = bf16_bits_to_f64(self.v_sink[seq, p])
        paged = [p for p in range(start, ctx) if p >= self.num_sink]
        if paged:
            slots = np.array([locate(table_row, p, self.block_size) for p in paged])
            K[n - len(paged):] = self._decode_k(self.k[slots], slots=slots)
            V[n - len(paged):] = self._decode_v(self.v[slots], slots=slots)
        return K, V


class ContiguousKVCache:
    """The unpaged layout that paging replaces: [B][kv_heads][max_seq_len][dim] plus a
    current-length counter per sequence (ldpk §2.3).  Used only to pin the paged oracle."""

    def __init__(self, num_seqs, num_kv_heads, max_seq_len, head_dim):
        self.k = np.zeros((num_seqs, num_kv_heads, max_seq_len, head_dim))
        self.v = np.zeros((num_seqs, num_kv_heads, max_seq_len, head_dim))
        self.current_len = np.zeros(num_seqs, dtype=np.int64)

    def append(self, seq, k_row, v_row):
        t = self.current_len[seq]
        self.k[seq, :, t] = k_row
        self.v[seq, :, t] = v_row
        self.current_len[seq] = t + 1

    def view(self, seq):
        n = self.current_len[seq]
        return self.k[seq, :, :n].transpose(1, 0, 2), self.v[seq, :, :n].transpose(1, 0, 2)


# ----------------------------------------------------------------------------------
# Attention
# ----------------------------------------------------------------------------------
def window_start(ctx: int, window: int) -> int:
    """First position a decode query of a ctx-token sequence attends (ldpk §5.3: only the most
    recent W tokens, the query's own included); window <= 0 means the whole context."""
    return max(0, ctx - window) if window > 0 else 0


def softmax_weights(scores) -> np.ndarray:
    """softmax with the maximum subtracted before exp (fp64)."""
    s = np.asarray(scores, dtype=np.float64)
    w = np.exp(s - s.max())
    return w / w.sum()


def decode_attention(q, K, V, scale: float, window: int = 0) -> np.ndarray:
    """One decode query per head against the cached tokens of one sequence.

    ldpk §2.1: Attention(Q, K, V) = softmax(Q K^T / sqrt(d_head)) V; in decode there is
    one query row per head (ldpk §2.2).  显存账本 §二: under GQA every g query heads share
    one KV head; the grouping is contiguous (query head h reads KV head h // g).
    ldpk §5.3: with a sliding window of W tokens the query (at position ctx - 1) attends only
    positions ctx - W .. ctx - 1.

    q: [H_q][d], K and V: [ctx][H_kv][d], all fp64.  ctx == 0 gives zeros.
    """
    q = np.asarray(q, dtype=np.float64)
    H_q, d = q.shape
    ctx, H_kv, _ = K.shape
    out = np.zeros((H_q, d))
    if ctx == 0:
        return out
    G = H_q // H_kv
    a = window_start(ctx, window)
    for h in range(H_q):
        kv = h // G
        scores = scale * (K[a:, kv, :] @ q[h])
        w = softmax_weights(scores)
        out[h] = w @ V[a:, kv, :]
    return out


def decode_attention_partials(q, K, V, scale: float, bounds):
    """Split the context at ``bounds`` (partition edges) and return, per partition and
    head, the unnormalised (m, l, o): m = max score, l = sum exp(s - m),
    o = sum exp(s - m) V.  Empty partitions give (-inf, 0, 0)."""
    q = np.asarray(q, dtype=np.float64)
    H_q, d = q.shape
    _, H_kv, _ = K.shape
    G = H_q // H_kv
    parts = []
    for a, b in zip(bounds[:-1], bounds[1:]):
        m = np.full(H_q, -np.inf)
        l = np.zeros(H_q)
        o = np.zeros((H_q, d))
        if b > a:
            for h in range(H_q):
                kv = h // G
                s = scale * (K[a:b, kv, :] @ q[h])
                m[h] = s.max()
                e = np.exp(s - m[h])
                l[h] = e.sum()
                o[h] = e @ V[a:b, kv, :]
        parts.append((m, l, o))
    return parts


def merge_partials(parts):
    """log-sum-exp merge: out = sum_p e^{m_p - M} o_p / sum_p e^{m_p - M} l_p, M = max m_p."""
    ms = np.stack([p[0] for p in parts])
    ls = np.stack([p[1] for p in parts])
    os_ = np.stack([p[2] for p in parts])
    M = ms.max(axis=0)
    safe_M = np.where(np.isfinite(M), M, 0.0)
    w = np.where(np.isfinite(ms), np.exp(ms - safe_M), 0.0)
    L = (w * ls).sum(axis=0)
    O = (w[:, :, None] * os_).sum(axis=0)
    out = np.zeros_like(O)
    nz = L > 0
    out[nz] = O[nz] / L[nz, None]
    return out


def decode_attention_split(q, K, V, scale: float, partition_tokens: int):
    """Decode attention computed over fixed-size context partitions and merged."""
    ctx = K.shape[0]
    if ctx == 0:
        return np.zeros(np.asarray(q).shape)
    bounds = list(range(0, ctx, partition_tokens)) + [ctx]
    return merge_partials(decode_attention_partials(q, K, V, scale, bounds))


def prefill_attention(q, K, V, scale: float, first_pos: int, window: int = 0) -> np.ndarray:
    """Causal attention of a chunk of new query tokens over one sequence's cached K/V.

    ldpk §2.2: during prefill every position's query attends to the keys of positions 1..i under
    the causal mask, and only K and V are kept; ldpk §7 splits a long prompt into chunks.  The
    chunk's queries sit at positions first_pos .. first_pos + n - 1 (their own K/V are already in
    the cache), and the query at position p reads keys 0..p.  GQA grouping as in
    decode_attention.  With a sliding window of W tokens (ldpk §5.3) the query at position p
    reads keys max(0, p - W + 1) .. p instead.
    q: [n][H_q][d], K and V: [ctx][H_kv][d] with ctx >= first_pos + n (fp64).
    """
    q = np.asarray(q, dtype=np.float64)
    n, H_q, d = q.shape
    ctx, H_kv, _ = K.shape
    G = H_q // H_kv
    out = np.zeros((n, H_q, d))
    for i in range(n):
        p = first_pos + i
        a = window_start(p + 1, window)
        for h in range(H_q):
            kv = h // G
            scores = scale * (K[a:p + 1, kv, :] @ q[i, h])
            out[i, h] = softmax_weights(scores) @ V[a:p + 1, kv, :]
    return out

"""Seeded synthetic decode workloads shaped like the pages' examples.

This module only draws random numbers and lays out shapes: context lengths, a random
placement of every sequence's logical blocks in the physical pool, bf16 N(0,1) token data
and the per-KV-head calibration scales of 8-bit caches (absmax / code range).  It holds none
of the method's arithmetic (no slot computation, no quantisation, no attention): the library
and the oracle each do that themselves from these same inputs.

Workloads (seed = 20260 + index):
  1 "tiny"        4 sequences, cached lengths {1, 17, 100, 256}, 8 query / 2 KV heads, d 64,
                  pool of 64 blocks, scale 1/8.
  2 "8b"          64 sequences, cached lengths uniform in [512, 4096], 32 / 8 heads, d 128,
                  pool = total need + 10 %.
  3 "70b"         32 sequences of 4096 cached tokens, 64 / 8 heads (GQA-8), d 128.
  4 "prefix_cow"  64 sequences sharing a 1208-token prefix (76 blocks, the last one half
                  full), private suffixes uniform in [200, 2000] tokens, 32 / 8 heads, d 128.
  5 "long_quant"  4 sequences of 131072 cached tokens, 32 / 8 heads, d 128, K stored FP8 E4M3
                  and V INT8 with per-KV-head scales from the absmax of the data, the first 4
                  positions kept in bf16 (sinks).
  6 "prefill_chunk"  8 sequences with cached lengths uniform in [0, 3584] each receiving a chunk
                  of 512 new tokens (queries + their K/V), 32 / 8 heads, d 128
                  (make_prefill_workload).
  7 "swa"         64 sequences, cached lengths uniform in [4096, 16384], 32 / 8 heads, d 128,
                  sliding window of 4096 tokens: only the blocks holding the first step's window
                  are in the pool (earlier table entries are -1, already released), and only the
                  window's positions are written.
  8 "int4_8b"     the 8b shape (64 sequences, cached U[512, 4096], 32 / 8 heads, d 128) with K and V
                  stored as INT4 codes with a scale and zero point per 32 dims of every row.
  9 "long_quant_tok"  the long_quant shape with K stored FP8 E4M3 with one scale per token's head
                  row (computed by the cache from each row, so no K calibration scales are
                  drawn), V INT8 with per-KV-head scales, 4 bf16 sinks.
Every step appends one token per sequence at position = cached length, then attends over
cached length + 1 tokens.  All tensors are produced on the CPU with a torch.Generator.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

BLOCK = 16

CONFIGS = {
    "tiny": dict(index=1, B=4, H_q=8, H_kv=2, D=64, ctx_list=[1, 17, 100, 256], pool_blocks=64),
    "8b": dict(index=2, B=64, H_q=32, H_kv=8, D=128, ctx_range=(512, 4096)),
    "70b": dict(index=3, B=32, H_q=64, H_kv=8, D=128, ctx_fixed=4096),
    "prefix_cow": dict(index=4, B=64, H_q=32, H_kv=8, D=128, prefix=1208, suffix_range=(200, 2000)),
    "long_quant": dict(index=5, B=4, H_q=32, H_kv=8, D=128, ctx_fixed=131072, quant=True, num_sink=4),
    "swa": dict(index=7, B=64, H_q=32, H_kv=8, D=128, ctx_range=(4096, 16384), window=4096),
    "int4_8b": dict(index=8, B=64, H_q=32, H_kv=8, D=128, ctx_range=(512, 4096), kv="int4"),
    "long_quant_tok": dict(index=9, B=4, H_q=32, H_kv=8, D=128, ctx_fixed=131072, quant=True, num_sink=4,
                           kv="e4m3_tok"),
}

# Calibration code ranges of the 8-bit formats (largest finite E4M3 value; symmetric int8).
E4M3_RANGE = 448.0
INT8_RANGE = 127.0


@dataclass
class Workload:
    name: str
    seed: int
    B: int
    H_q: int
    H_kv: int
    D: int
    k_dtype: str
    v_dtype: str
    num_sink: int
    scale: float
    num_blocks: int
    max_blocks: int
    steps: int
    ctx_old: np.ndarray            # int32 [B] tokens cached before step 0
    tables: np.ndarray             # int32 [B][max_blocks] placement of cached blocks, -1 = none
    fill_k: torch.Tensor           # bf16 [N][H_kv][D] cached tokens (CPU)
    fill_v: torch.Tensor
    fill_seq: np.ndarray           # int32 [N] sequence of each cached token
    fill_pos: np.ndarray           # int32 [N] position of each cached token
    q: torch.Tensor                # bf16 [steps][B][H_q][D]
    k_new: torch.Tensor            # bf16 [steps][B][H_kv][D]
    v_new: torch.Tensor
    k_scales: torch.Tensor | None = None  # fp32 [H_kv]
    v_scales: torch.Tensor | None = None
    prefix: int = 0                # shared prefix tokens (prefix_cow), cached once via sequence 0
    suffix_len: np.ndarray | None = None  # int32 [B] private tokens after the prefix
    suffix_k: torch.Tensor | None = None  # bf16 [sum(suffix_len)][H_kv][D], sequence-major
    suffix_v: torch.Tensor | None = None
    window: int = 0                # sliding window in tokens (0 = whole context)
    extra: dict = field(default_factory=dict)

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv

    def positions(self, step: int) -> np.ndarray:
        return (self.ctx_old + step).astype(np.int32)

    def context_lens(self, step: int) -> np.ndarray:
        return (self.ctx_old + step + 1).astype(np.int32)

    def kv_elem_bytes(self) -> int:
        return 1 if self.k_dtype != "bf16" else 2

    def kv_row_bytes(self) -> int:
        """Cache bytes of one (token, KV head) row of V (and of K, except with per-token K
        scales): int4 holds 4-bit codes plus one 32-bit scale / zero-point word per 32 dims."""
        if self.k_dtype == "int4":
            return self.D // 2 + self.D // 32 * 4
        return self.D * self.kv_elem_bytes()

    def k_row_bytes(self) -> int:
        """Cache bytes of one (token, KV head) row of K: per-token K scales add a 4-byte scale."""
        return self.kv_row_bytes() + (4 if self.k_dtype == "e4m3_tok" else 0)


def _randn_bf16(g, shape, chunk_rows=1 << 16):
    """N(0,1) drawn in fp32 and rounded to bf16 (round to nearest even), in row chunks."""
    out = torch.empty(shape, dtype=torch.bfloat16)
    if out.numel() == 0:
        return out
    flat = out.view(shape[0], -1)
    for a in range(0, shape[0], chunk_rows):
        b = min(shape[0], a + chunk_rows)
        flat[a:b] = torch.randn((b - a, flat.shape[1]), generator=g, dtype=torch.float32).to(torch.bfloat16)
    return out


def _blocks(n):
    return -(-int(n) // BLOCK)


def make_workload(name: str, steps: int = 1, **overrides) -> Workload:
    """Draw the named workload.  ``overrides`` shrink it for tests (e.g. B=8, ctx_range=(16, 300)).
    ``horizon`` (default: steps) sizes the tables and the pool for that many steps of appends while
    only ``steps`` steps of inputs are drawn; ``window`` > 0 makes it a sliding-window workload."""
    cfg = dict(CONFIGS[name])
    cfg.update(overrides)
    seed = cfg.get("seed", 20260 + cfg["index"])
    g = torch.Generator().manual_seed(seed)
    B, H_q, H_kv, D = cfg["B"], cfg["H_q"], cfg["H_kv"], cfg["D"]
    quant = cfg.get("quant", False)
    num_sink = cfg.get("num_sink", 0)
    prefix = cfg.get("prefix", 0)
    window = int(cfg.get("window", 0))
    horizon = int(cfg.get("horizon", steps))
    assert not (window and prefix), "sliding-window workloads have no shared prefix"

    if "ctx_list" in cfg:
        ctx = np.array(cfg["ctx_list"], dtype=np.int64)
        assert len(ctx) == B
    elif "ctx_range" in cfg:
        lo, hi = cfg["ctx_range"]
        ctx = torch.randint(lo, hi + 1, (B,), generator=g).numpy().astype(np.int64)
    elif prefix:
        ctx = np.full(B, prefix, dtype=np.int64)
    else:
        ctx = np.full(B, cfg["ctx_fixed"], dtype=np.int64)

    suffix_len = None
    if prefix:
        lo, hi = cfg["suffix_range"]
        suffix_len = torch.randint(lo, hi + 1, (B,), generator=g).numpy().astype(np.int64)
        final = prefix + suffix_len + steps
        need = _blocks(prefix) + sum(_blocks(f) - (_blocks(prefix) - 1) for f in final)
        max_blocks = int(max(_blocks(f) for f in final))
    else:
        final = ctx + horizon
        # first position kept: under a window only the first step's window is cached
        keep_from = np.maximum(0, ctx + 1 - window) if window else np.zeros(B, dtype=np.int64)
        need = int(sum(_blocks(f) - k // BLOCK for f, k in zip(final, keep_from)))
        max_blocks = int(max(_blocks(f) for f in final))
    num_blocks = int(cfg.get("pool_blocks") or math.ceil(1.1 * need))
    max_blocks = int(cfg.get("max_blocks", max_blocks))

    perm = torch.randperm(num_blocks, generator=g).numpy().astype(np.int32)
    tables = np.full((B, max_blocks), -1, dtype=np.int32)
    if prefix:
        shared = perm[:_blocks(prefix)]
        tables[:, :len(shared)] = shared
        fill_seq = np.zeros(prefix, dtype=np.int32)
        fill_pos = np.arange(prefix, dtype=np.int32)
    else:
        k = 0
        for s in range(B):
            b0, n = int(keep_from[s]) // BLOCK, _blocks(ctx[s])
            tables[s, b0:n] = perm[k:k + n - b0]
            k += n - b0
        fill_seq = np.repeat(np.arange(B, dtype=np.int32), ctx - keep_from)
        fill_pos = (np.concatenate([np.arange(a, c, dtype=np.int32) for a, c in zip(keep_from, ctx)])
                    if B else np.zeros(0, np.int32))

    N = len(fill_seq)
    fill_k = _randn_bf16(g, (N, H_kv, D))
    fill_v = _randn_bf16(g, (N, H_kv, D))
    suffix_k = suffix_v = None
    if prefix:
        ns = int(suffix_len.sum())
        suffix_k = _randn_bf16(g, (ns, H_kv, D))
        suffix_v = _randn_bf16(g, (ns, H_kv, D))
    q = _randn_bf16(g, (steps * B, H_q, D)).view(steps, B, H_q, D)
    k_new = _randn_bf16(g, (steps * B, H_kv, D)).view(steps, B, H_kv, D)
    v_new = _randn_bf16(g, (steps * B, H_kv, D)).view(steps, B, H_kv, D)

    k_scales = v_scales = None
    kv = cfg.get("kv")
    if quant:
        keep = torch.from_numpy(fill_pos >= num_sink)
        k_abs = torch.zeros(H_kv)
        v_abs = torch.zeros(H_kv)
        chunk = 1 << 20
        for a in range(0, N, chunk):
            m = keep[a:a + chunk]
            if m.any():
                k_abs = torch.maximum(k_abs, fill_k[a:a + chunk][m].float().abs().amax(dim=(0, 2)))
                v_abs = torch.maximum(v_abs, fill_v[a:a + chunk][m].float().abs().amax(dim=(0, 2)))
        k_scales = None if kv == "e4m3_tok" else (k_abs / E4M3_RANGE).to(torch.float32)
        v_scales = (v_abs / INT8_RANGE).to(torch.float32)

    int4 = kv == "int4"
    return Workload(
        name=name, seed=seed, B=B, H_q=H_q, H_kv=H_kv, D=D,
        k_dtype="int4" if int4 else (("e4m3_tok" if kv == "e4m3_tok" else "e4m3") if quant else "bf16"),
        v_dtype="int4" if int4 else ("int8" if quant else "bf16"),
        num_sink=num_sink, scale=1.0 / math.sqrt(D), num_blocks=num_blocks, max_blocks=max_blocks,
        steps=steps, ctx_old=ctx.astype(np.int32), tables=tables, fill_k=fill_k, fill_v=fill_v,
        fill_seq=fill_seq, fill_pos=fill_pos, q=q, k_new=k_new, v_new=v_new,
        k_scales=k_scales, v_scales=v_scales, prefix=prefix,
        suffix_len=None if suffix_len is None else suffix_len.astype(np.int32),
        suffix_k=suffix_k, suffix_v=suffix_v, window=window,
    )


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The raw bit patterns of a bf16 tensor as uint16 (for the oracle's exact decoding)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


@dataclass
class PrefillWorkload:
    """A chunk of new tokens per sequence on top of an already cached prefix."""
    name: str
    seed: int
    B: int
    H_q: int
    H_kv: int
    D: int
    scale: float
    num_blocks: int
    max_blocks: int
    ctx_old: np.ndarray        # int32 [B] cached tokens before the chunk
    chunk: np.ndarray          # int32 [B] new tokens per sequence
    tables: np.ndarray         # int32 [B][max_blocks], blocks for cached + chunk positions
    fill_k: torch.Tensor       # bf16 [N][H_kv][D] cached tokens
    fill_v: torch.Tensor
    fill_seq: np.ndarray
    fill_pos: np.ndarray
    new_k: torch.Tensor        # bf16 [T][H_kv][D] the chunk's tokens, sequence-major
    new_v: torch.Tensor
    new_seq: np.ndarray        # int32 [T]
    new_pos: np.ndarray        # int32 [T]
    q: torch.Tensor            # bf16 [T][H_q][D]

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv

    def q_start(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.chunk)]).astype(np.int32)

    def context_lens(self) -> np.ndarray:
        return (self.ctx_old + self.chunk).astype(np.int32)


def make_prefill_workload(B=8, H_q=32, H_kv=8, D=128, cached_range=(0, 3584), chunk=512,
                          cached_list=None, chunk_list=None, seed=20266, name="prefill_chunk"):
    g = torch.Generator().manual_seed(seed)
    if cached_list is not None:
        ctx = np.array(cached_list, dtype=np.int64)
        B = len(ctx)
    else:
        lo, hi = cached_range
        ctx = torch.randint(lo, hi + 1, (B,), generator=g).numpy().astype(np.int64)
    n = np.array(chunk_list if chunk_list is not None else [chunk] * B, dtype=np.int64)
    total = ctx + n
    need = int(sum(_blocks(t) for t in total))
    num_blocks = max(1, int(math.ceil(1.1 * need)))
    max_blocks = max(1, int(max(_blocks(t) for t in total)))
    perm = torch.randperm(num_blocks, generator=g).numpy().astype(np.int32)
    tables = np.full((B, max_blocks), -1, dtype=np.int32)
    k = 0
    for s in range(B):
        m = _blocks(total[s])
        tables[s, :m] = perm[k:k + m]
        k += m
    fill_seq = np.repeat(np.arange(B, dtype=np.int32), ctx)
    fill_pos = np.concatenate([np.arange(c, dtype=np.int32) for c in ctx]) if B else np.zeros(0, np.int32)
    new_seq = np.repeat(np.arange(B, dtype=np.int32), n)
    new_pos = np.concatenate([np.arange(c, c + m, dtype=np.int32) for c, m in zip(ctx, n)])
    fill_k = _randn_bf16(g, (len(fill_seq), H_kv, D))
    fill_v = _randn_bf16(g, (len(fill_seq), H_kv, D))
    T = int(n.sum())
    new_k = _randn_bf16(g, (T, H_kv, D))
    new_v = _randn_bf16(g, (T, H_kv, D))
    q = _randn_bf16(g, (T, H_q, D))
    return PrefillWorkload(name=name, seed=seed, B=B, H_q=H_q, H_kv=H_kv, D=D, scale=1.0 / math.sqrt(D),
                           num_blocks=num_blocks, max_blocks=max_blocks, ctx_old=ctx.astype(np.int32),
                           chunk=n.astype(np.int32), tables=tables, fill_k=fill_k, fill_v=fill_v,
                           fill_seq=fill_seq, fill_pos=fill_pos, new_k=new_k, new_v=new_v,
                           new_seq=new_seq, new_pos=new_pos, q=q)

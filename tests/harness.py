"""Test infrastructure: build the same decode state twice — once on the GPU through the C ABI,
once in the CPU oracle — from one seeded workload, and compare.

The GPU side calls only the library (block manager, bulk append, block copy, append, decode
attention).  The oracle side calls only ``oracle``.  They share nothing but the workload's
random inputs.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle as O
import paged_kv_cache_table_gb300 as P
from paged_kv_cache_table_gb300.workloads import Workload, bf16_bits

# Fill patterns for never-written slots: NaN in bf16 pools (0x7FC0) and in e4m3 K pools
# (0x7F); -128 in int8 V pools (outside the encoder's range).  Attention must never let them
# reach the output.
BF16_NAN = 0x7FC0
E4M3_NAN = 0x7F
INT8_OUTSIDE = 0x80
# int4 pools: every code nibble 15 and every group parameter word all ones (a NaN scale, zero
# point 255)
INT4_FILL = 0xFF
# per-token K pools: every byte 0x7F, i.e. NaN codes and never-written scales of 0x7F7F7F7F
# (3.4e38); an attention that read either would not stay finite
TOK_FILL = 0x7F

ATOL_MAX = 2e-2   # attention: max |gpu - oracle|
ATOL_MEAN = 2e-3  # attention: mean |gpu - oracle|


def _refcounts_from_tables(w: Workload):
    blocks, counts = np.unique(w.tables[w.tables >= 0], return_counts=True)
    extra = 1 if w.prefix else 0  # the cached prefix itself holds one reference
    return blocks, counts + extra


class GpuState:
    """One layer's paged cache on the GPU, driven only through the C ABI."""

    def __init__(self, w: Workload, device="cuda", fill=True):
        self.w = w
        self.dev = device
        n_slots = w.num_blocks * 16
        shape = (n_slots, w.H_kv, w.D)
        if w.k_dtype == "bf16":
            self.k = torch.full(shape, BF16_NAN, dtype=torch.int16, device=device).view(torch.bfloat16)
            self.v = torch.full(shape, BF16_NAN, dtype=torch.int16, device=device).view(torch.bfloat16)
        elif w.k_dtype == "int4":
            nbytes = n_slots * w.H_kv * w.kv_row_bytes()
            self.k = torch.full((nbytes,), INT4_FILL, dtype=torch.uint8, device=device)
            self.v = torch.full((nbytes,), INT4_FILL, dtype=torch.uint8, device=device)
        elif w.k_dtype == "e4m3_tok":
            self.k = torch.full((n_slots * w.H_kv * w.k_row_bytes(),), TOK_FILL, dtype=torch.uint8, device=device)
            self.v = torch.full(shape, INT8_OUTSIDE, dtype=torch.uint8, device=device)
        else:
            self.k = torch.full(shape, E4M3_NAN, dtype=torch.uint8, device=device)
            self.v = torch.full(shape, INT8_OUTSIDE, dtype=torch.uint8, device=device)
        self.k_scales = None if w.k_scales is None else w.k_scales.to(device)
        self.v_scales = None if w.v_scales is None else w.v_scales.to(device)
        self.k_sink = self.v_sink = None
        if w.num_sink:
            sshape = (w.B, w.num_sink, w.H_kv, w.D)
            self.k_sink = torch.full(sshape, BF16_NAN, dtype=torch.int16, device=device).view(torch.bfloat16)
            self.v_sink = torch.full(sshape, BF16_NAN, dtype=torch.int16, device=device).view(torch.bfloat16)
        self.desc = P.make_desc(w.B, w.H_q, w.H_kv, w.D, w.num_blocks, w.max_blocks, w.k_dtype, w.v_dtype,
                                self.k_scales, self.v_scales, self.k_sink, self.v_sink, w.num_sink,
                                sliding_window=w.window)
        self.tables = w.tables.copy()
        self.tables_dev = torch.from_numpy(self.tables).to(device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.bm = P.BlockManager(w.num_blocks)
        blocks, counts = _refcounts_from_tables(w)
        for b, c in zip(blocks, counts):
            assert self.bm.claim(int(b))
            for _ in range(int(c) - 1):
                self.bm.incref(int(b))
        if fill:
            self.bulk_append(w.fill_k, w.fill_v, w.fill_seq, w.fill_pos)

    def bulk_append(self, k, v, seq, pos):
        n = len(seq)
        if n == 0:
            return
        P.pa_kv_append_tokens(self.desc, self.k, self.v, k.to(self.dev), v.to(self.dev), n,
                              torch.from_numpy(np.ascontiguousarray(seq, dtype=np.int32)).to(self.dev),
                              torch.from_numpy(np.ascontiguousarray(pos, dtype=np.int32)).to(self.dev),
                              self.tables_dev, self.err)

    def prepare(self, positions):
        pairs, _ = self.bm.prepare_step(self.tables, np.ascontiguousarray(positions, dtype=np.int32))
        self.tables_dev.copy_(torch.from_numpy(self.tables))
        if len(pairs):
            P.pa_block_copy(self.desc, self.k, self.v, torch.from_numpy(pairs).to(self.dev), len(pairs), self.err)
        return pairs

    def append(self, k_new, v_new, positions):
        P.pa_kv_append(self.desc, self.k, self.v, k_new.to(self.dev), v_new.to(self.dev), self.tables_dev,
                       torch.from_numpy(np.ascontiguousarray(positions, dtype=np.int32)).to(self.dev), self.err)

    def attend(self, q, context_lens, partition=0, max_ctx=None):
        w = self.w
        ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
        max_ctx = int(ctx.max()) if max_ctx is None else int(max_ctx)
        out = torch.full((w.B, w.H_q, w.D), float("nan"), dtype=torch.bfloat16, device=self.dev)
        nbytes = P.pa_decode_workspace_size(self.desc, max_ctx, partition)
        assert nbytes > 0
        ws = torch.empty(nbytes, dtype=torch.uint8, device=self.dev)
        P.pa_decode_attention(self.desc, out, q.to(self.dev), self.k, self.v, self.tables_dev,
                              torch.from_numpy(ctx).to(self.dev), max_ctx, w.scale, partition, ws, nbytes,
                              self.err)
        return out

    def decode_step(self, k_new, v_new, q, positions, context_lens, partition=0, max_ctx=None):
        """pa_decode_step: the append of one token per sequence and the attention in one call
        (the entry point the benchmark times).  The slots must be writable (prepare first)."""
        w = self.w
        pos = np.ascontiguousarray(positions, dtype=np.int32)
        ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
        max_ctx = int(ctx.max()) if max_ctx is None else int(max_ctx)
        out = torch.full((w.B, w.H_q, w.D), float("nan"), dtype=torch.bfloat16, device=self.dev)
        nbytes = P.pa_decode_workspace_size(self.desc, max_ctx, partition)
        assert nbytes > 0
        ws = torch.empty(nbytes, dtype=torch.uint8, device=self.dev)
        P.pa_decode_step(self.desc, out, q.to(self.dev), self.k, self.v, k_new.to(self.dev), v_new.to(self.dev),
                         self.tables_dev, torch.from_numpy(pos).to(self.dev), torch.from_numpy(ctx).to(self.dev),
                         max_ctx, w.scale, partition, ws, nbytes, self.err)
        return out

    def attend_shared(self, q, context_lens, shared_seqs, shared_len, partition=0, max_ctx=None, ws_fill=None):
        """pa_decode_attention_shared: the listed sequences' first shared_len positions attended
        once for all of them.  ws_fill: a byte the workspace is filled with first (else empty)."""
        w = self.w
        ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
        max_ctx = int(ctx.max()) if max_ctx is None else int(max_ctx)
        out = torch.full((w.B, w.H_q, w.D), float("nan"), dtype=torch.bfloat16, device=self.dev)
        nbytes = P.pa_decode_shared_workspace_size(self.desc, max_ctx, partition, shared_len)
        assert nbytes > 0
        if ws_fill is None:
            ws = torch.empty(nbytes, dtype=torch.uint8, device=self.dev)
        else:
            ws = torch.full((nbytes,), ws_fill, dtype=torch.uint8, device=self.dev)
        seqs = torch.tensor(np.asarray(shared_seqs, dtype=np.int32), device=self.dev)
        P.pa_decode_attention_shared(self.desc, out, q.to(self.dev), self.k, self.v, self.tables_dev,
                                     torch.from_numpy(ctx).to(self.dev), max_ctx, w.scale, partition, seqs,
                                     len(shared_seqs), shared_len, ws, nbytes, self.err)
        return out

    def attend_noalloc(self, q, context_lens, partition=0, max_ctx=None):
        """pa_decode_attention_noalloc: the same attention with the library's static scratch."""
        w = self.w
        ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
        max_ctx = int(ctx.max()) if max_ctx is None else int(max_ctx)
        out = torch.full((w.B, w.H_q, w.D), float("nan"), dtype=torch.bfloat16, device=self.dev)
        P.pa_decode_attention_noalloc(self.desc, out, q.to(self.dev), self.k, self.v, self.tables_dev,
                                      torch.from_numpy(ctx).to(self.dev), max_ctx, w.scale, partition, self.err)
        return out

    def slide(self, context_lens):
        """Sliding window: release the blocks behind every sequence's window (host tables, then
        the device copy)."""
        released, freed = self.bm.slide_window(self.tables, context_lens, self.w.window)
        if released:
            self.tables_dev.copy_(torch.from_numpy(self.tables))
        return freed

    def step(self, i, partition=0):
        w = self.w
        pos = w.positions(i)
        pairs = self.prepare(pos)
        self.append(w.k_new[i], w.v_new[i], pos)
        out = self.attend(w.q[i], w.context_lens(i), partition)
        if w.window:
            self.slide(w.context_lens(i))
        return out, pairs

    def err_bits(self) -> int:
        torch.cuda.synchronize()
        return int(self.err.item())

    def pools(self):
        """Host copies of the raw pools (uint16 bf16 bits or uint8 codes) and sink buffers."""
        torch.cuda.synchronize()
        def raw(t):
            if t is None:
                return None
            if t.dtype == torch.bfloat16:
                return t.view(torch.int16).cpu().numpy().view(np.uint16)
            return t.cpu().numpy()
        return raw(self.k), raw(self.v), raw(self.k_sink), raw(self.v_sink)


class OracleState:
    """The same layer in the oracle: pool, tables, refcounts, codes."""

    def __init__(self, w: Workload, fill=True):
        self.w = w
        ks = None if w.k_scales is None else w.k_scales.numpy().astype(np.float32)
        vs = None if w.v_scales is None else w.v_scales.numpy().astype(np.float32)
        self.cache = O.PagedKVCache(w.num_blocks, w.H_kv, w.D, k_dtype=w.k_dtype, v_dtype=w.v_dtype,
                                    k_scales=ks, v_scales=vs, num_seqs=w.B, num_sink=w.num_sink)
        if w.k_dtype == "bf16":
            self.cache.k[:] = BF16_NAN
            self.cache.v[:] = BF16_NAN
        elif w.k_dtype == "int4":  # what the GPU fill reads as
            self.cache.k[:] = 15
            self.cache.v[:] = 15
            self.cache.k_params[:] = 0xFFFFFFFF
            self.cache.v_params[:] = 0xFFFFFFFF
        elif w.k_dtype == "e4m3_tok":
            self.cache.k[:] = TOK_FILL
            self.cache.k_tscale.view(np.uint32)[:] = 0x7F7F7F7F
            self.cache.v[:] = INT8_OUTSIDE
        else:
            self.cache.k[:] = E4M3_NAN
            self.cache.v[:] = INT8_OUTSIDE
        self.cache.k_sink[:] = BF16_NAN
        self.cache.v_sink[:] = BF16_NAN
        self.pool = O.BlockPool(w.num_blocks)
        blocks, counts = _refcounts_from_tables(w)
        for b, c in zip(blocks, counts):
            assert self.pool.claim(int(b))
            for _ in range(int(c) - 1):
                self.pool.incref(int(b))
        self.tables = w.tables.astype(np.int64).copy()
        if fill:
            self.bulk_append(w.fill_k, w.fill_v, w.fill_seq, w.fill_pos)

    def bulk_append(self, k, v, seq, pos):
        kb, vb = bf16_bits(k), bf16_bits(v)
        for i in range(len(seq)):
            s = int(seq[i])
            self.cache.append(s, self.tables[s], int(pos[i]), kb[i], vb[i])

    def prepare(self, positions):
        pairs = []
        for s, p in enumerate(positions):
            if p < 0:
                continue
            act = self.pool.prepare_append(self.tables[s], int(p))
            if act[0] == "copy":
                self.cache.block_copy(act[1], act[2])
                pairs.append((act[1], act[2]))
        return pairs

    def append(self, k_new, v_new, positions):
        kb, vb = bf16_bits(k_new), bf16_bits(v_new)
        for s, p in enumerate(positions):
            if p >= 0:
                self.cache.append(s, self.tables[s], int(p), kb[s], vb[s])

    def attend(self, q, context_lens):
        w = self.w
        qv = O.bf16_bits_to_f64(bf16_bits(q))
        out = np.zeros((w.B, w.H_q, w.D))
        for s in range(w.B):
            c = int(context_lens[s])
            # positions before the window are never gathered (their blocks may be released)
            K, V = self.cache.gather(s, self.tables[s], c, O.window_start(c, w.window))
            out[s] = O.decode_attention(qv[s], K, V, w.scale)
        return out

    def slide(self, context_lens):
        return sum(self.pool.slide_window(self.tables[s], int(context_lens[s]), self.w.window)
                   for s in range(self.w.B))

    def step(self, i):
        w = self.w
        pos = w.positions(i)
        pairs = self.prepare(pos)
        self.append(w.k_new[i], w.v_new[i], pos)
        out = self.attend(w.q[i], w.context_lens(i))
        if w.window:
            self.slide(w.context_lens(i))
        return out, pairs


def to_f64(out: torch.Tensor) -> np.ndarray:
    return out.float().cpu().numpy().astype(np.float64)


def assert_attention_close(gpu: np.ndarray, ref: np.ndarray, what=""):
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite output"
    err = np.abs(gpu - ref)
    assert err.max() <= ATOL_MAX, f"{what}: max abs err {err.max():.3e}"
    assert err.mean() <= ATOL_MEAN, f"{what}: mean abs err {err.mean():.3e}"
    return float(err.max()), float(err.mean())


def unpack_int4_pool(raw: np.ndarray, n_slots: int, H: int, D: int, tensor: str):
    """Natural-order codes [slot][head][dim] and params [slot][head][dim/32] of a GPU int4 pool,
    read by the byte layout the library documents for PA_INT4 (K: word 4c + g holds dims
    32g + 8c + i at bits 4i; V: byte 8r + m holds dims 16m + r and 16m + r + 8)."""
    code_bytes = n_slots * H * (D // 2)
    rows = raw[:code_bytes].reshape(n_slots, H, D // 2)
    params = raw[code_bytes:code_bytes + n_slots * H * (D // 32) * 4].view(np.uint32).reshape(n_slots, H, D // 32)
    codes = np.empty((n_slots, H, D), dtype=np.uint8)
    if tensor == "k":
        words = rows.view(np.uint32)  # [slot][head][16]
        for c in range(4):
            for g in range(D // 32):
                w = words[:, :, 4 * c + g]
                for i in range(8):
                    codes[:, :, 32 * g + 8 * c + i] = (w >> (4 * i)) & 0xF
    else:
        for r in range(8):
            for m in range(D // 16):
                b = rows[:, :, 8 * r + m]
                codes[:, :, 16 * m + r] = b & 0xF
                codes[:, :, 16 * m + r + 8] = b >> 4
    return codes, params


def unpack_tok_pool(raw: np.ndarray, n_slots: int, H: int, D: int):
    """Codes [slot][head][D] and fp32 scales [slot][head] of a GPU per-token K pool, read by the
    layout the library documents for PA_FP8_E4M3_TOKEN (codes of every slot, then the scales)."""
    code_bytes = n_slots * H * D
    codes = raw[:code_bytes].reshape(n_slots, H, D)
    scales = raw[code_bytes:code_bytes + n_slots * H * 4].view(np.float32).reshape(n_slots, H)
    return codes, scales


def assert_pools_equal(gpu: GpuState, ora: OracleState):
    gk, gv, gks, gvs = gpu.pools()
    assert np.array_equal(gpu.tables, ora.tables.astype(np.int32)), "block tables differ"
    if gpu.w.k_dtype == "e4m3_tok":
        w = gpu.w
        kc, ks = unpack_tok_pool(gk, w.num_blocks * 16, w.H_kv, w.D)
        assert np.array_equal(kc, ora.cache.k), "K codes differ"
        assert np.array_equal(ks.view(np.uint32), ora.cache.k_tscale.view(np.uint32)), "K token scales differ"
        assert np.array_equal(gv, ora.cache.v), "V pool differs"
    elif gpu.w.k_dtype == "int4":
        w = gpu.w
        n_slots = w.num_blocks * 16
        kc, kp = unpack_int4_pool(gk, n_slots, w.H_kv, w.D, "k")
        vc, vp = unpack_int4_pool(gv, n_slots, w.H_kv, w.D, "v")
        assert np.array_equal(kc, ora.cache.k), "K codes differ"
        assert np.array_equal(kp, ora.cache.k_params), "K group parameters differ"
        assert np.array_equal(vc, ora.cache.v), "V codes differ"
        assert np.array_equal(vp, ora.cache.v_params), "V group parameters differ"
    else:
        assert np.array_equal(gk, ora.cache.k), "K pool differs"
        assert np.array_equal(gv, ora.cache.v), "V pool differs"
    if gks is not None:
        assert np.array_equal(gks, ora.cache.k_sink), "K sink buffer differs"
        assert np.array_equal(gvs, ora.cache.v_sink), "V sink buffer differs"


# ----------------------------------------------------------------------------------
# Full-size checks: the oracle computes each sequence's rows from the workload's logical token
# stream (the K/V rows of the positions a step attends, in position order), without building a
# whole pool.
# ----------------------------------------------------------------------------------
def logical_tokens(w: Workload, s: int, step: int):
    """bf16 bit rows [n][H_kv][D] of the positions sequence s attends at `step`, in order, and the
    position of the first one.  Positions a workload never wrote (before a sliding window) are
    not part of it: the rows start at the first cached position."""
    parts_k, parts_v = [], []
    if w.prefix:
        pos0 = 0
        parts_k.append(bf16_bits(w.fill_k))
        parts_v.append(bf16_bits(w.fill_v))
        off = int(w.suffix_len[:s].sum())
        n = int(w.suffix_len[s])
        parts_k.append(bf16_bits(w.suffix_k[off:off + n]))
        parts_v.append(bf16_bits(w.suffix_v[off:off + n]))
    else:
        idx = np.nonzero(w.fill_seq == s)[0]
        order = idx[np.argsort(w.fill_pos[idx])]
        pos0 = int(w.fill_pos[order[0]]) if len(order) else int(w.ctx_old[s])
        parts_k.append(bf16_bits(w.fill_k[torch.from_numpy(order)]))
        parts_v.append(bf16_bits(w.fill_v[torch.from_numpy(order)]))
    for i in range(step + 1):
        parts_k.append(bf16_bits(w.k_new[i, s:s + 1]))
        parts_v.append(bf16_bits(w.v_new[i, s:s + 1]))
    return np.concatenate(parts_k), np.concatenate(parts_v), pos0


def _decode_head(k_dtype, num_sink, ks, vs, kb, vb, pos0):
    """fp64 K and V [n][D] of one KV head's logical rows kb/vb (positions pos0 ..) as the cache
    stores them: sink positions in bf16, the others through the oracle's encoder and decoder for
    the cache kind (ks/vs: that head's 8-bit scales)."""
    n = kb.shape[0]
    ns = max(0, min(pos0 + n, num_sink) - pos0)
    K = np.empty(kb.shape)
    V = np.empty(vb.shape)
    K[:ns] = O.bf16_bits_to_f64(kb[:ns])
    V[:ns] = O.bf16_bits_to_f64(vb[:ns])
    if k_dtype == "bf16":
        K[ns:] = O.bf16_bits_to_f64(kb[ns:])
        V[ns:] = O.bf16_bits_to_f64(vb[ns:])
    elif k_dtype == "int4":
        K[ns:] = O.int4_decode_row(*O.int4_encode_row(kb[ns:]))
        V[ns:] = O.int4_decode_row(*O.int4_encode_row(vb[ns:]))
    elif k_dtype == "e4m3_tok":
        codes, sc = O.quantize_token_rows(kb[ns:])
        K[ns:] = O.e4m3_decode(codes) * sc.astype(np.float64)[:, None]
        V[ns:] = O.int8_decode(O.quantize_row(vb[ns:], vs, "int8").view(np.int8)) * float(vs)
    else:
        K[ns:] = O.e4m3_decode(O.quantize_row(kb[ns:], ks, "e4m3")) * float(ks)
        V[ns:] = O.int8_decode(O.quantize_row(vb[ns:], vs, "int8").view(np.int8)) * float(vs)
    return K, V


def _head_scales(w: Workload, h: int):
    ks = None if w.k_scales is None else np.float32(w.k_scales[h].item())
    vs = None if w.v_scales is None else np.float32(w.v_scales[h].item())
    return ks, vs


def _head_task(args):
    """Oracle rows [G][D] of the G query heads of one KV head of one sequence (pool worker)."""
    k_dtype, num_sink, ks, vs, kb, vb, pos0, q, scale, window = args
    K, V = _decode_head(k_dtype, num_sink, ks, vs, kb, vb, pos0)
    return O.decode_attention(q, K[:, None, :], V[:, None, :], scale, window=window)


def _seq_tasks(w: Workload, s: int, step: int, kb: np.ndarray, vb: np.ndarray, pos0: int):
    q = O.bf16_bits_to_f64(bf16_bits(w.q[step, s]))
    for h in range(w.H_kv):
        ks, vs = _head_scales(w, h)
        yield (w.k_dtype, w.num_sink, ks, vs, np.ascontiguousarray(kb[:, h]), np.ascontiguousarray(vb[:, h]), pos0,
               q[h * w.G:(h + 1) * w.G], w.scale, w.window)


def reference_seq(w: Workload, s: int, step: int, kb: np.ndarray, vb: np.ndarray, pos0: int = 0) -> np.ndarray:
    """Oracle output [H_q][D] of every query head of sequence s at `step`; kb/vb are the logical
    bf16 rows of positions pos0 .. ctx-1 (the window start or 0 up to the new token)."""
    return np.concatenate([_head_task(t) for t in _seq_tasks(w, s, step, kb, vb, pos0)])


def reference_all(w: Workload, step: int = 0, processes: int = 0) -> np.ndarray:
    """Oracle output [B][H_q][D] of every (sequence, query head) row of a decode step.  With
    processes > 1 the (sequence, KV head) pieces run in a pool of spawned processes (each piece is
    the same oracle call; only where it runs differs)."""
    out = np.zeros((w.B, w.H_q, w.D))
    if processes <= 1:
        for s in range(w.B):
            kb, vb, pos0 = logical_tokens(w, s, step)
            out[s] = reference_seq(w, s, step, kb, vb, pos0)
        return out
    import multiprocessing as mp

    def tasks():
        for s in range(w.B):
            kb, vb, pos0 = logical_tokens(w, s, step)
            yield from _seq_tasks(w, s, step, kb, vb, pos0)
    with mp.get_context("spawn").Pool(processes) as pool:
        for i, rows in enumerate(pool.imap(_head_task, tasks())):
            s, h = divmod(i, w.H_kv)
            out[s, h * w.G:(h + 1) * w.G] = rows
    return out


def reference_row(w: Workload, s: int, h: int, step: int, kb: np.ndarray, vb: np.ndarray) -> np.ndarray:
    """Oracle output of query head h of sequence s (kb/vb: logical bf16 bit rows from position 0)."""
    return reference_seq(w, s, step, kb, vb)[h]

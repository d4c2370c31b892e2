"""Chunked prefill over caches that are not plain bf16: 8-bit K/V with per-head scales or with
per-token K scales, INT4 with a scale and zero point per 32 dims, and bf16 with sink tokens kept
in their own buffer ("KV Cache 的显存账本：PagedAttention 与连续批处理" §七; untitled KV-cache
article at ldpk.cn/news/58971 §5.2 and §7).

A chunk that extends a long quantised context, or that follows a prefix-cache hit on a quantised
pool, attends over the stored codes: the GPU decodes every block (code times scale, sinks from the
sink buffer) and must stay within max-abs 2e-2 / mean-abs 2e-3 of the fp64 oracle, which decodes
the same codes exactly (PagedKVCache.gather) and runs its causal prefill_attention.  The chunk's
K/V go in through the library's bulk append first, so the stored codes are the library's own;
never-written slots and sink rows start as NaN (or codes that decode to NaN)."""

import numpy as np
import pytest
import torch

import oracle as O
from paged_kv_cache_table_gb300 import native as N
from paged_kv_cache_table_gb300.workloads import bf16_bits, make_prefill_workload

from harness import BF16_NAN, E4M3_NAN, INT4_FILL, INT8_OUTSIDE, TOK_FILL, assert_attention_close, to_f64

pytestmark = pytest.mark.gpu

KINDS = {"fp8": ("e4m3", "int8"), "fp8_token": ("e4m3_tok", "int8"), "int4": ("int4", "int4"), "bf16": ("bf16", "bf16")}


def _scales(w, num_sink):
    """Per-KV-head calibration scales from the absmax of the non-sink tokens (the input recipe of the
    8-bit workloads): K / 448, V / 127."""
    keep_f = torch.from_numpy(w.fill_pos >= num_sink)
    keep_n = torch.from_numpy(w.new_pos >= num_sink)
    k = torch.cat([w.fill_k[keep_f], w.new_k[keep_n]]).float().abs().amax(dim=(0, 2))
    v = torch.cat([w.fill_v[keep_f], w.new_v[keep_n]]).float().abs().amax(dim=(0, 2))
    return (k / 448.0).float(), (v / 127.0).float()


class QuantPrefill:
    def __init__(self, w, kind, num_sink=0, window=0):
        self.w, self.kind, self.num_sink, self.window = w, kind, num_sink, window
        kd, vd = KINDS[kind]
        n_slots = w.num_blocks * 16
        shape = (n_slots, w.H_kv, w.D)
        if kd == "bf16":
            self.k = torch.full(shape, BF16_NAN, dtype=torch.int16, device="cuda").view(torch.bfloat16)
            self.v = torch.full(shape, BF16_NAN, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        elif kd == "int4":
            nbytes = n_slots * w.H_kv * (w.D // 2 + w.D // 32 * 4)
            self.k = torch.full((nbytes,), INT4_FILL, dtype=torch.uint8, device="cuda")
            self.v = torch.full((nbytes,), INT4_FILL, dtype=torch.uint8, device="cuda")
        elif kd == "e4m3_tok":
            self.k = torch.full((n_slots * w.H_kv * (w.D + 4),), TOK_FILL, dtype=torch.uint8, device="cuda")
            self.v = torch.full(shape, INT8_OUTSIDE, dtype=torch.uint8, device="cuda")
        else:
            self.k = torch.full(shape, E4M3_NAN, dtype=torch.uint8, device="cuda")
            self.v = torch.full(shape, INT8_OUTSIDE, dtype=torch.uint8, device="cuda")
        self.ks = self.vs = None
        if kd in ("e4m3", "e4m3_tok"):
            ks, vs = _scales(w, num_sink)
            self.ks = None if kd == "e4m3_tok" else ks
            self.vs = vs
        self.k_scales = None if self.ks is None else self.ks.cuda()
        self.v_scales = None if self.vs is None else self.vs.cuda()
        self.k_sink = self.v_sink = None
        if num_sink:
            sshape = (w.B, num_sink, w.H_kv, w.D)
            self.k_sink = torch.full(sshape, BF16_NAN, dtype=torch.int16, device="cuda").view(torch.bfloat16)
            self.v_sink = torch.full(sshape, BF16_NAN, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        self.desc = N.make_desc(w.B, w.H_q, w.H_kv, w.D, w.num_blocks, w.max_blocks, kd, vd, self.k_scales,
                                self.v_scales, self.k_sink, self.v_sink, num_sink, sliding_window=window)
        self.tables = torch.from_numpy(w.tables).cuda()
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def append(self, which):
        w = self.w
        k, v, seq, pos = ((w.fill_k, w.fill_v, w.fill_seq, w.fill_pos) if which == "fill"
                          else (w.new_k, w.new_v, w.new_seq, w.new_pos))
        if len(seq):
            N.pa_kv_append_tokens(self.desc, self.k, self.v, k.cuda(), v.cuda(), len(seq), torch.from_numpy(seq).cuda(),
                                  torch.from_numpy(pos).cuda(), self.tables, self.err)

    def _out(self):
        w = self.w
        return torch.full((max(1, int(w.q_start()[-1])), w.H_q, w.D), float("nan"), dtype=torch.bfloat16,
                          device="cuda")

    def attend(self, ctx=None):
        w = self.w
        out = self._out()
        ctx = w.context_lens() if ctx is None else ctx
        N.pa_prefill_attention(self.desc, out, w.q.cuda(), self.k, self.v, self.tables,
                               torch.from_numpy(w.q_start()).cuda(),
                               torch.from_numpy(np.ascontiguousarray(ctx, dtype=np.int32)).cuda(), int(w.chunk.max()),
                               w.scale, self.err)
        return out

    def attend_ws(self, ctx=None, fill=0):
        """pa_prefill_attention_ws: every attended block decoded once into the workspace (filled
        with the byte `fill` first: its contents must not matter), then the bf16 tensor-core path."""
        w = self.w
        out = self._out()
        ctx = w.context_lens() if ctx is None else ctx
        max_ctx = int(w.max_blocks * 16)
        nbytes = N.pa_prefill_workspace_size(self.desc, max_ctx)
        ws = torch.full((max(nbytes, 1),), fill, dtype=torch.uint8, device="cuda") if nbytes else None
        N.pa_prefill_attention_ws(self.desc, out, w.q.cuda(), self.k, self.v, self.tables,
                                  torch.from_numpy(w.q_start()).cuda(),
                                  torch.from_numpy(np.ascontiguousarray(ctx, dtype=np.int32)).cuda(),
                                  int(w.chunk.max()), max_ctx, w.scale, ws, nbytes, self.err)
        return out, nbytes

    def step_ws(self):
        """pa_prefill_step_ws: the chunk's append and the workspace attention in one call."""
        w = self.w
        out = self._out()
        max_ctx = int(w.max_blocks * 16)
        nbytes = N.pa_prefill_workspace_size(self.desc, max_ctx)
        ws = torch.empty((max(nbytes, 1),), dtype=torch.uint8, device="cuda") if nbytes else None
        N.pa_prefill_step_ws(self.desc, out, w.q.cuda(), self.k, self.v, w.new_k.cuda(), w.new_v.cuda(),
                             len(w.new_seq), torch.from_numpy(w.new_seq).cuda(), torch.from_numpy(w.new_pos).cuda(),
                             self.tables, torch.from_numpy(w.q_start()).cuda(),
                             torch.from_numpy(w.context_lens()).cuda(), int(w.chunk.max()), max_ctx, w.scale, ws,
                             nbytes, self.err)
        return out

    def step(self):
        """pa_prefill_step: the chunk's append and the attention in one call."""
        w = self.w
        out = self._out()
        N.pa_prefill_step(self.desc, out, w.q.cuda(), self.k, self.v, w.new_k.cuda(), w.new_v.cuda(), len(w.new_seq),
                          torch.from_numpy(w.new_seq).cuda(), torch.from_numpy(w.new_pos).cuda(), self.tables,
                          torch.from_numpy(w.q_start()).cuda(), torch.from_numpy(w.context_lens()).cuda(),
                          int(w.chunk.max()), w.scale, self.err)
        return out

    def oracle(self):
        """The oracle's cache of the same kind, filled with the same tokens, gathered and decoded
        exactly, then causal prefill attention per sequence."""
        w = self.w
        kd, vd = KINDS[self.kind]
        ks = None if self.ks is None else self.ks.numpy().astype(np.float32)
        vs = None if self.vs is None else self.vs.numpy().astype(np.float32)
        cache = O.PagedKVCache(w.num_blocks, w.H_kv, w.D, k_dtype=kd, v_dtype=vd, k_scales=ks, v_scales=vs,
                               num_seqs=w.B, num_sink=self.num_sink)
        tables = w.tables.astype(np.int64)
        for k, v, seq, pos in ((w.fill_k, w.fill_v, w.fill_seq, w.fill_pos), (w.new_k, w.new_v, w.new_seq, w.new_pos)):
            kb, vb = bf16_bits(k), bf16_bits(v)
            for i in range(len(seq)):
                cache.append(int(seq[i]), tables[seq[i]], int(pos[i]), kb[i], vb[i])
        qv = O.bf16_bits_to_f64(bf16_bits(w.q))
        qs = w.q_start()
        out = np.zeros((int(qs[-1]), w.H_q, w.D))
        for s in range(w.B):
            ctx = int(w.context_lens()[s])
            K, V = cache.gather(s, tables[s], ctx)
            out[qs[s]:qs[s + 1]] = O.prefill_attention(qv[qs[s]:qs[s + 1]], K, V, w.scale, int(w.ctx_old[s]),
                                                       window=self.window)
        return out


def _check(g, out, what):
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0, what
    assert_attention_close(to_f64(out), g.oracle(), what)


@pytest.mark.parametrize("kind", ["fp8", "fp8_token", "int4"])
@pytest.mark.parametrize("H_q,H_kv", [(32, 8), (64, 8), (16, 4)])
def test_prefill_over_quantized_cache(kind, H_q, H_kv):
    w = make_prefill_workload(H_q=H_q, H_kv=H_kv, D=128, cached_list=[0, 17, 100, 300], chunk_list=[5, 16, 33, 70],
                              seed=31)
    g = QuantPrefill(w, kind)
    g.append("fill")
    g.append("new")
    _check(g, g.attend(), f"{kind} {H_q}/{H_kv}")


@pytest.mark.parametrize("kind", ["fp8", "fp8_token", "int4", "bf16"])
def test_prefill_with_sinks(kind):
    """4 sink positions kept in bf16: chunks that start inside the sink range, right after it, and
    far beyond it; a sequence shorter than the sinks."""
    w = make_prefill_workload(H_q=32, H_kv=8, D=128, cached_list=[0, 2, 4, 200, 1], chunk_list=[3, 9, 20, 40, 1],
                              seed=32)
    g = QuantPrefill(w, kind, num_sink=4)
    g.append("fill")
    g.append("new")
    _check(g, g.attend(), f"{kind} with sinks")


def test_prefill_bf16_sinks_head_dim_64():
    w = make_prefill_workload(H_q=8, H_kv=2, D=64, cached_list=[0, 6, 90], chunk_list=[12, 30, 7], seed=33)
    g = QuantPrefill(w, "bf16", num_sink=4)
    g.append("fill")
    g.append("new")
    _check(g, g.attend(), "bf16 sinks d 64")


@pytest.mark.parametrize("kind", ["fp8", "int4"])
def test_prefill_quantized_sliding_window(kind):
    w = make_prefill_workload(H_q=32, H_kv=8, D=128, cached_list=[0, 300, 60], chunk_list=[100, 50, 77], seed=34)
    g = QuantPrefill(w, kind, window=64)
    g.append("fill")
    g.append("new")
    _check(g, g.attend(), f"{kind} window 64")


@pytest.mark.parametrize("kind", ["fp8_token", "int4", "bf16"])
def test_prefill_step_equals_append_then_attention(kind):
    w = make_prefill_workload(H_q=32, H_kv=8, D=128, cached_list=[10, 150], chunk_list=[40, 9], seed=35)
    a, b = QuantPrefill(w, kind, num_sink=4), QuantPrefill(w, kind, num_sink=4)
    for g in (a, b):
        g.append("fill")
    a.append("new")
    out_a = a.attend()
    out_b = b.step()
    torch.cuda.synchronize()
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    assert torch.equal(a.k.view(torch.uint8) if a.k.dtype != torch.uint8 else a.k,
                       b.k.view(torch.uint8) if b.k.dtype != torch.uint8 else b.k)
    _check(b, out_b, f"{kind} prefill step")


def test_prefill_quantized_invalid_length_and_bad_block():
    w = make_prefill_workload(H_q=32, H_kv=8, D=128, cached_list=[20, 40, 30], chunk_list=[10, 10, 10], seed=36)
    g = QuantPrefill(w, "fp8")
    g.append("fill")
    g.append("new")
    ref = g.oracle()
    ctx = w.context_lens().copy()
    ctx[1] = 5  # fewer context tokens than queries
    out = to_f64(g.attend(ctx))
    torch.cuda.synchronize()
    assert int(g.err.item()) & N.PA_EFLAG_CTX_OVERFLOW
    assert np.all(out[10:20] == 0)
    keep = np.r_[0:10, 20:30]
    assert_attention_close(out[keep], ref[keep], "other sequences")
    g.err.zero_()
    g.tables[2, 1] = w.num_blocks + 5
    out = to_f64(g.attend())
    torch.cuda.synchronize()
    assert int(g.err.item()) & N.PA_EFLAG_BAD_BLOCK_ID
    assert np.all(out[20:30] == 0)
    assert_attention_close(out[:20], ref[:20], "sequences with valid tables")


def test_one_token_chunks_agree_with_the_decode_path():
    """A chunk of one token is a decode step: both paths over the same 8-bit cache with sinks
    match the oracle."""
    w = make_prefill_workload(H_q=32, H_kv=8, D=128, cached_list=[40, 3, 300], chunk_list=[1, 1, 1], seed=37)
    g = QuantPrefill(w, "fp8", num_sink=4)
    g.append("fill")
    g.append("new")
    ref = g.oracle()
    pre = g.attend()
    out = torch.empty((w.B, w.H_q, w.D), dtype=torch.bfloat16, device="cuda")
    ctx = torch.from_numpy(w.context_lens()).cuda()
    nbytes = N.pa_decode_workspace_size(g.desc, int(w.context_lens().max()), 0)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    N.pa_decode_attention(g.desc, out, w.q.cuda(), g.k, g.v, g.tables, ctx, int(w.context_lens().max()), w.scale, 0,
                          ws, nbytes, g.err)
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    assert_attention_close(to_f64(pre), ref, "prefill of one token")
    assert_attention_close(to_f64(out), ref, "decode")



# ---- pa_prefill_attention_ws: each attended block decoded once, then the tcgen05 kernel ----

@pytest.mark.parametrize("kind", ["fp8", "fp8_token", "int4"])
@pytest.mark.parametrize("H_q,H_kv", [(32, 8), (64, 8), (16, 4), (8, 8), (16, 8)])
def test_prefill_ws_over_quantized_cache(kind, H_q, H_kv):
    w = make_prefill_workload(H_q=H_q, H_kv=H_kv, D=128, cached_list=[0, 17, 100, 300], chunk_list=[5, 16, 33, 70],
                              seed=31)
    g = QuantPrefill(w, kind)
    g.append("fill")
    g.append("new")
    out, nbytes = g.attend_ws()
    assert nbytes > 0
    _check(g, out, f"ws {kind} {H_q}/{H_kv}")


@pytest.mark.parametrize("kind", ["fp8", "fp8_token", "int4", "bf16"])
def test_prefill_ws_with_sinks(kind):
    w = make_prefill_workload(H_q=32, H_kv=8, D=128, cached_list=[0, 2, 4, 200, 1], chunk_list=[3, 9, 20, 40, 1],
                              seed=32)
    g = QuantPrefill(w, kind, num_sink=4)
    g.append("fill")
    g.append("new")
    out, nbytes = g.attend_ws()
    assert nbytes > 0
    _check(g, out, f"ws {kind} with sinks")


@pytest.mark.parametrize("kind", ["fp8", "int4"])
def test_prefill_ws_sliding_window(kind):
    """Blocks before the first query's window are neither decoded nor read."""
    w = make_prefill_workload(H_q=32, H_kv=8, D=128, cached_list=[0, 300, 60], chunk_list=[100, 50, 77], seed=34)
    g = QuantPrefill(w, kind, window=64)
    g.append("fill")
    g.append("new")
    out, _ = g.attend_ws()
    _check(g, out, f"ws {kind} window 64")


@pytest.mark.parametrize("kind", ["fp8", "int4"])
def test_prefill_ws_long_chunks_many_tiles(kind):
    """Chunks of several 64-token items per sequence over contexts of many 128-key tiles, a
    workspace full of 0xFF bytes (NaN in bf16) against one of zeros: identical, and both match the
    oracle and the block-by-block path."""
    w = make_prefill_workload(H_q=32, H_kv=8, D=128, cached_list=[1500, 40, 700], chunk_list=[300, 130, 257],
                              seed=38)
    g = QuantPrefill(w, kind, num_sink=4)
    g.append("fill")
    g.append("new")
    a, _ = g.attend_ws(fill=0)
    b, _ = g.attend_ws(fill=0xFF)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    _check(g, a, f"ws {kind} long chunks")
    _check(g, g.attend(), f"block by block {kind} long chunks")


def test_prefill_ws_plain_shapes_need_no_workspace():
    """bf16 without sinks and head_dim 64 with sinks take the plain path: no workspace."""
    w = make_prefill_workload(H_q=32, H_kv=8, D=128, cached_list=[10, 90], chunk_list=[20, 33], seed=39)
    g = QuantPrefill(w, "bf16")
    g.append("fill")
    g.append("new")
    out, nbytes = g.attend_ws()
    assert nbytes == 0
    _check(g, out, "ws bf16 plain")
    w = make_prefill_workload(H_q=8, H_kv=2, D=64, cached_list=[0, 6, 90], chunk_list=[12, 30, 7], seed=33)
    g = QuantPrefill(w, "bf16", num_sink=4)
    g.append("fill")
    g.append("new")
    out, nbytes = g.attend_ws()
    assert nbytes == 0
    _check(g, out, "ws bf16 sinks d 64")


def test_prefill_ws_invalid_length_and_bad_block():
    w = make_prefill_workload(H_q=32, H_kv=8, D=128, cached_list=[20, 40, 30], chunk_list=[10, 10, 10], seed=36)
    g = QuantPrefill(w, "fp8")
    g.append("fill")
    g.append("new")
    ref = g.oracle()
    ctx = w.context_lens().copy()
    ctx[1] = 5  # fewer context tokens than queries
    out, _ = g.attend_ws(ctx)
    out = to_f64(out)
    torch.cuda.synchronize()
    assert int(g.err.item()) & N.PA_EFLAG_CTX_OVERFLOW
    assert np.all(out[10:20] == 0)
    keep = np.r_[0:10, 20:30]
    assert_attention_close(out[keep], ref[keep], "other sequences")
    g.err.zero_()
    g.tables[2, 1] = w.num_blocks + 5
    out, _ = g.attend_ws()
    out = to_f64(out)
    torch.cuda.synchronize()
    assert int(g.err.item()) & N.PA_EFLAG_BAD_BLOCK_ID
    assert np.all(out[20:30] == 0)
    assert_attention_close(out[:20], ref[:20], "sequences with valid tables")


@pytest.mark.parametrize("kind", ["fp8", "fp8_token", "int4", "bf16"])
def test_prefill_step_ws_equals_append_then_attention_ws(kind):
    w = make_prefill_workload(H_q=32, H_kv=8, D=128, cached_list=[10, 150, 600], chunk_list=[40, 9, 130], seed=35)
    a, b = QuantPrefill(w, kind, num_sink=4), QuantPrefill(w, kind, num_sink=4)
    for g in (a, b):
        g.append("fill")
    a.append("new")
    out_a, _ = a.attend_ws()
    out_b = b.step_ws()
    torch.cuda.synchronize()
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    assert torch.equal(a.k.view(torch.uint8) if a.k.dtype != torch.uint8 else a.k,
                       b.k.view(torch.uint8) if b.k.dtype != torch.uint8 else b.k)
    _check(b, out_b, f"{kind} prefill step, workspace path")

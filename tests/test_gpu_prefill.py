"""Chunked-prefill attention on the GPU vs the oracle's causal attention (prefill_attention).

The chunk's K/V are appended through the library's bulk append, its queries attend causally
over the cached prefix plus the chunk; outputs must be within max-abs 2e-2 / mean-abs 2e-3 of
the fp64 oracle.  Never-written slots hold NaN, so reading past a row's causal limit would show.
"""

import numpy as np
import pytest
import torch

import oracle as O
from paged_kv_cache_table_gb300 import native as N
from paged_kv_cache_table_gb300.workloads import bf16_bits, make_prefill_workload

from harness import BF16_NAN, assert_attention_close, to_f64

pytestmark = pytest.mark.gpu


class PrefillGpu:
    def __init__(self, w):
        self.w = w
        shape = (w.num_blocks * 16, w.H_kv, w.D)
        self.k = torch.full(shape, BF16_NAN, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        self.v = torch.full(shape, BF16_NAN, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        self.desc = N.make_desc(w.B, w.H_q, w.H_kv, w.D, w.num_blocks, w.max_blocks)
        self.tables = torch.from_numpy(w.tables).cuda()
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        for k, v, seq, pos in ((w.fill_k, w.fill_v, w.fill_seq, w.fill_pos), (w.new_k, w.new_v, w.new_seq, w.new_pos)):
            if len(seq):
                N.pa_kv_append_tokens(self.desc, self.k, self.v, k.cuda(), v.cuda(), len(seq),
                                      torch.from_numpy(seq).cuda(), torch.from_numpy(pos).cuda(), self.tables,
                                      self.err)

    def run(self, q_start=None, ctx=None, max_q=None):
        w = self.w
        q_start = w.q_start() if q_start is None else q_start
        ctx = w.context_lens() if ctx is None else ctx
        max_q = int(w.chunk.max()) if max_q is None else max_q
        out = torch.full((max(1, int(q_start[-1])), w.H_q, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
        N.pa_prefill_attention(self.desc, out, w.q.cuda(), self.k, self.v, self.tables,
                               torch.from_numpy(np.ascontiguousarray(q_start, dtype=np.int32)).cuda(),
                               torch.from_numpy(np.ascontiguousarray(ctx, dtype=np.int32)).cuda(), max_q, w.scale,
                               self.err)
        torch.cuda.synchronize()
        return to_f64(out)


def oracle_prefill(w, seqs=None):
    """Oracle rows for every query token (sequence-major), built from the logical token stream."""
    qv = O.bf16_bits_to_f64(bf16_bits(w.q))
    qs = w.q_start()
    out = np.zeros((int(qs[-1]), w.H_q, w.D))
    fk, fv = bf16_bits(w.fill_k), bf16_bits(w.fill_v)
    nk, nv = bf16_bits(w.new_k), bf16_bits(w.new_v)
    for s in (range(w.B) if seqs is None else seqs):
        ci = np.nonzero(w.fill_seq == s)[0]
        ci = ci[np.argsort(w.fill_pos[ci])]
        ni = np.arange(qs[s], qs[s + 1])
        K = O.bf16_bits_to_f64(np.concatenate([fk[ci], nk[ni]]))
        V = O.bf16_bits_to_f64(np.concatenate([fv[ci], nv[ni]]))
        out[qs[s]:qs[s + 1]] = O.prefill_attention(qv[qs[s]:qs[s + 1]], K, V, w.scale, int(w.ctx_old[s]))
    return out


@pytest.mark.parametrize("H_q,H_kv,D", [(8, 2, 64), (32, 8, 128), (64, 8, 128), (8, 8, 128), (12, 4, 128),
                                        (6, 1, 64), (16, 2, 64)])
def test_prefill_matches_oracle(H_q, H_kv, D):
    w = make_prefill_workload(H_q=H_q, H_kv=H_kv, D=D, cached_list=[0, 17, 100, 3], chunk_list=[5, 16, 33, 70])
    g = PrefillGpu(w)
    out = g.run()
    assert int(g.err.item()) == 0
    assert_attention_close(out, oracle_prefill(w), f"prefill {H_q}/{H_kv}/{D}")


def test_prefill_medium_random_lengths():
    w = make_prefill_workload(B=5, H_q=32, H_kv=8, D=128, cached_range=(0, 700), chunk=129, seed=7)
    g = PrefillGpu(w)
    out = g.run()
    assert int(g.err.item()) == 0
    assert_attention_close(out, oracle_prefill(w), "prefill medium")


def test_prefill_of_one_token_equals_decode():
    w = make_prefill_workload(H_q=32, H_kv=8, D=128, cached_list=[40, 16, 1, 300], chunk_list=[1, 1, 1, 1])
    g = PrefillGpu(w)
    pre = g.run()
    # the same rows through the decode path (queries are one token per sequence)
    out = torch.empty((w.B, w.H_q, w.D), dtype=torch.bfloat16, device="cuda")
    ctx = torch.from_numpy(w.context_lens()).cuda()
    nbytes = N.pa_decode_workspace_size(g.desc, int(w.context_lens().max()), 0)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    N.pa_decode_attention(g.desc, out, w.q.cuda(), g.k, g.v, g.tables, ctx, int(w.context_lens().max()), w.scale,
                          0, ws, nbytes, g.err)
    dec = to_f64(out)
    ref = oracle_prefill(w)
    assert_attention_close(pre, ref, "prefill 1")
    assert_attention_close(dec, ref, "decode")


def test_prefill_invalid_lengths_and_bad_blocks():
    w = make_prefill_workload(H_q=8, H_kv=2, D=64, cached_list=[20, 20, 20], chunk_list=[10, 10, 10])
    g = PrefillGpu(w)
    ref = oracle_prefill(w)
    ctx = w.context_lens().copy()
    ctx[1] = 5  # fewer context tokens than queries: invalid
    out = g.run(ctx=ctx)
    assert int(g.err.item()) & N.PA_EFLAG_CTX_OVERFLOW
    assert np.all(out[10:20] == 0)
    keep = np.r_[0:10, 20:30]
    assert_attention_close(out[keep], ref[keep], "other sequences")
    g.err.zero_()
    g.tables[2, 0] = w.num_blocks + 3
    out = g.run()
    assert int(g.err.item()) & N.PA_EFLAG_BAD_BLOCK_ID
    assert np.all(out[20:30] == 0)
    assert_attention_close(out[:20], ref[:20], "sequences with valid tables")


@pytest.mark.slow
def test_prefill_full_size_sampled():
    w = make_prefill_workload()  # 8 sequences, cached U[0, 3584], chunks of 512
    g = PrefillGpu(w)
    out = g.run()
    assert int(g.err.item()) == 0
    assert np.all(np.isfinite(out))
    seqs = [0, 3, 7]
    ref = oracle_prefill(w, seqs)
    qs = w.q_start()
    rows = np.concatenate([np.arange(qs[s], qs[s + 1]) for s in seqs])
    assert_attention_close(out[rows], ref[rows], "prefill full size")


# ---- the tcgen05 kernel (head_dim 128, G a power of two): work items, order and edge paths ----

def test_prefill_tc_invalid_lengths_and_bad_blocks():
    """G = 4, d 128: an invalid sequence is zeroed and flagged; a bad block id zeroes the rows of
    the query tiles whose keys include it and is flagged; other rows are unaffected."""
    w = make_prefill_workload(H_q=32, H_kv=8, D=128, cached_list=[20, 300, 20, 150], chunk_list=[40, 70, 10, 200])
    g = PrefillGpu(w)
    ref = oracle_prefill(w)
    qs = w.q_start()
    ctx = w.context_lens().copy()
    ctx[1] = 50  # fewer context tokens than queries: invalid
    out = g.run(ctx=ctx)
    assert int(g.err.item()) & N.PA_EFLAG_CTX_OVERFLOW
    assert np.all(out[qs[1]:qs[2]] == 0)
    keep = np.r_[qs[0]:qs[1], qs[2]:qs[4]]
    assert_attention_close(out[keep], ref[keep], "valid sequences next to an invalid one")
    g.err.zero_()
    g.tables[3, 0] = w.num_blocks + 3  # block 0 is read by every query tile of sequence 3
    out = g.run()
    assert int(g.err.item()) & N.PA_EFLAG_BAD_BLOCK_ID
    assert np.all(out[qs[3]:qs[4]] == 0)
    assert_attention_close(out[:qs[3]], ref[:qs[3]], "sequences with valid tables")


def test_prefill_tc_many_ragged_items():
    """40 sequences, G = 8 (32 query tokens per work item), chunks of 0..300 tokens over 0..500
    cached: the longest-first item list with ragged tiles, empty chunks and one-token chunks;
    every row against the oracle."""
    rng = np.random.default_rng(11)
    chunks = rng.integers(0, 301, 40)
    chunks[[3, 17]] = 0
    chunks[25] = 1
    cached = rng.integers(0, 501, 40)
    w = make_prefill_workload(H_q=32, H_kv=4, D=128, cached_list=cached.tolist(), chunk_list=chunks.tolist(), seed=11)
    g = PrefillGpu(w)
    out = g.run()
    assert int(g.err.item()) == 0
    assert_attention_close(out, oracle_prefill(w), "40 ragged sequences")


def test_prefill_tc_more_items_than_resident_ctas():
    """1300 sequences x 8 KV heads = 10400 work items: more than one CTA's list holds (64) for
    every resident CTA (one per SM), so the launch adds CTAs that start as others finish."""
    rng = np.random.default_rng(12)
    B = 1300
    w = make_prefill_workload(H_q=64, H_kv=8, D=128, cached_list=rng.integers(0, 61, B).tolist(),
                              chunk_list=rng.integers(1, 4, B).tolist(), seed=12)
    g = PrefillGpu(w)
    out = g.run()
    assert int(g.err.item()) == 0
    assert_attention_close(out, oracle_prefill(w), "1300 sequences")


def test_prefill_tc_over_4096_sequences():
    """4200 sequences: beyond the 4096 whose geometry the kernel ranks in shared memory, work
    items run in their plain order (last tiles first, sequences in order); every row checked."""
    rng = np.random.default_rng(13)
    B = 4200
    w = make_prefill_workload(H_q=32, H_kv=8, D=128, cached_list=rng.integers(0, 31, B).tolist(),
                              chunk_list=rng.integers(0, 3, B).tolist(), seed=13)
    g = PrefillGpu(w)
    out = g.run()
    assert int(g.err.item()) == 0
    assert_attention_close(out, oracle_prefill(w), "4200 sequences")

"""pa_decode_attention_shared: a prompt prefix shared by many sequences attended once for all.

Sequences forked from one cached prompt point their first blocks at the same physical blocks
("大模型推理KV Cache显存优化：从PagedAttention到AI内存系统演进" §3.1; §3.3: only whole blocks are
shared, the partly filled last block is copied at the fork).  The result must be the attention
of every sequence over its own logical token stream (untitled KV-cache article at
ldpk.cn/news/58971 §2.1), whichever sequences the caller lists: each case is compared with the
oracle, and with pa_decode_attention on the same state.  The list is a hint the library checks —
sequences whose context does not cover the prefix, whose table differs in a prefix block, that
are listed twice or not at all, or an out-of-range entry, must all still get their exact rows.
"""

import numpy as np
import pytest
import torch

from paged_kv_cache_table_gb300 import native as P
from paged_kv_cache_table_gb300.workloads import make_workload

from harness import GpuState, OracleState, assert_attention_close, to_f64

pytestmark = pytest.mark.gpu


def _forked(w):
    """Both states after the fork of the prefix's partial block, the private suffixes and one
    steady-state append; returns them and the context lengths of the step."""
    g, o = GpuState(w), OracleState(w)
    pos = w.positions(0)
    g.prepare(pos), o.prepare(pos)
    g.append(w.k_new[0], w.v_new[0], pos)
    o.append(w.k_new[0], w.v_new[0], pos)
    seqs, poss, rows = [], [], []
    off = 0
    for s in range(w.B):
        n = int(w.suffix_len[s])
        seqs += [s] * (n - 1)
        poss += list(range(w.prefix + 1, w.prefix + n))
        rows += list(range(off + 1, off + n))
        off += n
    idx = torch.tensor(rows, dtype=torch.long)
    for state in (g, o):
        for p in range(w.prefix + 1, w.prefix + int(w.suffix_len.max())):
            state.prepare(np.where(p < w.prefix + w.suffix_len, p, -1).astype(np.int32))
        state.bulk_append(w.suffix_k[idx], w.suffix_v[idx], np.array(seqs, np.int32), np.array(poss, np.int32))
    steady = (w.prefix + w.suffix_len).astype(np.int32)
    for state in (g, o):
        state.prepare(steady)
        state.append(w.k_new[0], w.v_new[0], steady)
    return g, o, steady + 1


def _set_table(g, o, s, b, block):
    g.tables[s, b] = block
    g.tables_dev.copy_(torch.from_numpy(g.tables))
    o.tables[s, b] = block


SHAPES = {
    "gqa4_d128": dict(),
    "gqa8_d128": dict(H_q=64, H_kv=8),
    "gqa4_d64": dict(H_q=8, H_kv=2, D=64),
    "mha_d128": dict(H_q=8, H_kv=8),
}


@pytest.mark.parametrize("shape", sorted(SHAPES))
@pytest.mark.parametrize("partition", [0, 32, 512])
def test_all_listed_matches_oracle_and_plain_decode(shape, partition):
    # prefix of 300 tokens: 18 whole shared blocks (three 128-key chunks, the last one ragged)
    w = make_workload("prefix_cow", B=12, prefix=300, suffix_range=(3, 90), steps=1, **SHAPES[shape])
    g, o, ctx = _forked(w)
    shared_len = (w.prefix // 16) * 16
    ref = o.attend(w.q[0], ctx)
    out = g.attend_shared(w.q[0], ctx, list(range(w.B)), shared_len, partition)
    assert_attention_close(to_f64(out), ref, f"{shape} p{partition} shared")
    plain = g.attend(w.q[0], ctx, partition)
    assert_attention_close(to_f64(out), to_f64(plain), f"{shape} p{partition} shared vs plain")
    assert g.err_bits() == 0


def test_subsets_duplicates_and_prefix_lengths():
    w = make_workload("prefix_cow", B=10, prefix=520, suffix_range=(1, 200), steps=1)
    g, o, ctx = _forked(w)
    ref = o.attend(w.q[0], ctx)
    lists = {
        "every other": [0, 2, 4, 6, 8],
        "one": [7],
        "duplicates": [3, 3, 1, 1, 9, 3],
        "reversed": list(range(w.B))[::-1],
    }
    for name, seqs in lists.items():
        for shared_len in (16, 256, 512):
            out = g.attend_shared(w.q[0], ctx, seqs, shared_len)
            assert_attention_close(to_f64(out), ref, f"{name} L{shared_len}")
    assert g.err_bits() == 0


def test_unqualified_members_are_attended_in_full():
    w = make_workload("prefix_cow", B=8, prefix=300, suffix_range=(20, 120), steps=1)
    g, o, ctx = _forked(w)
    shared_len = 288
    ctx = ctx.copy()
    ctx[2] = 100          # context shorter than the prefix: positions 0..99 only
    ctx[5] = shared_len   # context exactly the prefix: no block of its own past it
    # sequence 6's table points prefix block 4 at a private block of sequence 7 (other data):
    # taking the shared rows for it would be wrong
    _set_table(g, o, 6, 4, int(g.tables[7, w.prefix // 16 + 1]))
    ref = o.attend(w.q[0], ctx)
    out = g.attend_shared(w.q[0], ctx, list(range(w.B)), shared_len)
    assert_attention_close(to_f64(out), ref, "unqualified members")
    assert g.err_bits() == 0
    # the first listed sequence does not cover the prefix: nothing is shared, all rows exact
    out = g.attend_shared(w.q[0], ctx, [2, 0, 1, 3], shared_len)
    assert_attention_close(to_f64(out), ref, "short leader")
    assert g.err_bits() == 0


def test_out_of_range_entries_flag_bad_seq():
    w = make_workload("prefix_cow", B=6, prefix=200, suffix_range=(5, 60), steps=1)
    g, o, ctx = _forked(w)
    ref = o.attend(w.q[0], ctx)
    for seqs in ([w.B + 3, 0, 1], [0, -1, 2, w.B]):
        out = g.attend_shared(w.q[0], ctx, seqs, 192)
        assert_attention_close(to_f64(out), ref, f"list {seqs}")
        assert g.err_bits() == P.PA_EFLAG_BAD_SEQ
        g.err.zero_()


def test_bad_prefix_block_zeroes_rows_like_plain_decode():
    w = make_workload("prefix_cow", B=6, prefix=200, suffix_range=(5, 60), steps=1)
    g, o, ctx = _forked(w)
    for s in range(w.B):
        g.tables[s, 3] = w.num_blocks + 7
    g.tables_dev.copy_(torch.from_numpy(g.tables))
    out = g.attend_shared(w.q[0], ctx, list(range(w.B)), 192)
    assert g.err_bits() & P.PA_EFLAG_BAD_BLOCK_ID
    g.err.zero_()
    plain = g.attend(w.q[0], ctx)
    assert g.err_bits() & P.PA_EFLAG_BAD_BLOCK_ID
    assert torch.all(plain == 0) and torch.all(out == 0)


def test_result_does_not_depend_on_workspace_contents():
    w = make_workload("prefix_cow", B=9, prefix=400, suffix_range=(1, 300), steps=1)
    g, o, ctx = _forked(w)
    seqs = [0, 1, 2, 4, 5, 7, 8]
    base = g.attend_shared(w.q[0], ctx, seqs, 384, ws_fill=0)
    assert_attention_close(to_f64(base), o.attend(w.q[0], ctx), "ws zeros")
    for fill in (0xFF, 0x7F, 0x80):
        assert torch.equal(g.attend_shared(w.q[0], ctx, seqs, 384, ws_fill=fill), base), hex(fill)
    assert g.err_bits() == 0


def test_nothing_to_share_is_the_plain_decode():
    w = make_workload("prefix_cow", B=5, prefix=100, suffix_range=(5, 40), steps=1)
    g, o, ctx = _forked(w)
    plain = g.attend(w.q[0], ctx)
    assert torch.equal(g.attend_shared(w.q[0], ctx, list(range(w.B)), 0), plain)
    assert torch.equal(g.attend_shared(w.q[0], ctx, [], 96), plain)
    assert g.err_bits() == 0


def test_graph_replay_matches_eager_calls():
    """The shared call (flag clearing, prefix kernel, decode, merge) captured once in a CUDA graph
    and replayed with new queries in the captured buffer equals an eager call each time."""
    w = make_workload("prefix_cow", B=8, prefix=300, suffix_range=(10, 200), steps=1)
    g, o, ctx = _forked(w)
    shared_len = 288
    ctx_dev = torch.from_numpy(np.ascontiguousarray(ctx, dtype=np.int32)).to(g.dev)
    max_ctx = int(ctx.max())
    seqs = torch.arange(w.B, dtype=torch.int32, device=g.dev)
    nbytes = P.pa_decode_shared_workspace_size(g.desc, max_ctx, 0, shared_len)
    ws_graph = torch.empty(nbytes, dtype=torch.uint8, device=g.dev)
    ws_eager = torch.empty(nbytes, dtype=torch.uint8, device=g.dev)
    q_buf = w.q[0].to(g.dev)
    out_buf = torch.empty((w.B, w.H_q, w.D), dtype=torch.bfloat16, device=g.dev)
    out_eager = torch.empty_like(out_buf)

    def call(q, out, ws):
        P.pa_decode_attention_shared(g.desc, out, q, g.k, g.v, g.tables_dev, ctx_dev, max_ctx, w.scale, 0, seqs,
                                     w.B, shared_len, ws, nbytes, g.err)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call(q_buf, out_buf, ws_graph)  # warm-up outside the capture
        side.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            call(q_buf, out_buf, ws_graph)
    torch.cuda.synchronize()
    gen = torch.Generator().manual_seed(12)
    for r in range(3):
        q_new = (torch.randn((w.B, w.H_q, w.D), generator=gen) * 0.5).to(torch.bfloat16)
        q_buf.copy_(q_new.to(g.dev))
        graph.replay()
        torch.cuda.synchronize()
        call(q_buf, out_eager, ws_eager)
        torch.cuda.synchronize()
        assert torch.equal(out_buf, out_eager), f"replay {r}"
        if r == 2:
            assert_attention_close(to_f64(out_buf), o.attend(q_new, ctx), "replay vs oracle")
    assert g.err_bits() == 0

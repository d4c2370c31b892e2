"""GPU path vs the CPU oracle, element by element, through the C ABI.

Append, copy-on-write and block-table indexing must match bit for bit (whole pools, sink
buffers and tables are compared, including never-written slots that hold NaN).  Attention
outputs must be within max-abs 2e-2 and mean-abs 2e-3 of the fp64 oracle.
"""

import numpy as np
import pytest
import torch

from paged_kv_cache_table_gb300 import native as N
from paged_kv_cache_table_gb300.workloads import make_workload

from harness import (GpuState, OracleState, assert_attention_close, assert_pools_equal, to_f64)

pytestmark = pytest.mark.gpu

PARTITIONS = [0, 16, 48, 512, 1 << 20]


def _run_and_compare(w, partition=0, steps=None):
    g = GpuState(w)
    o = OracleState(w)
    for i in range(w.steps if steps is None else steps):
        out, gpairs = g.step(i, partition)
        ref, opairs = o.step(i)
        assert [tuple(p) for p in gpairs.tolist()] == [tuple(p) for p in opairs]
        assert_attention_close(to_f64(out), ref, f"{w.name} step {i} partition {partition}")
    assert g.err_bits() == 0
    assert_pools_equal(g, o)
    return g, o


@pytest.mark.parametrize("partition", PARTITIONS)
def test_tiny_paged_decode(partition):
    # 4 sequences with cached lengths {1, 17, 100, 256}, GQA-4, d 64, 64-block pool
    _run_and_compare(make_workload("tiny"), partition)


@pytest.mark.parametrize("partition", [0, 32, 512])
def test_8b_shape_reduced(partition):
    w = make_workload("8b", B=7, ctx_range=(1, 700), steps=3)
    _run_and_compare(w, partition)


@pytest.mark.parametrize("partition", [0, 64])
def test_70b_shape_gqa8_reduced(partition):
    w = make_workload("70b", B=3, ctx_fixed=527, steps=2)
    _run_and_compare(w, partition)


@pytest.mark.parametrize("H_q,H_kv,D", [(8, 8, 128), (8, 1, 128), (4, 4, 64), (16, 2, 64), (12, 4, 128),
                                        (32, 16, 64), (6, 2, 128)])
def test_head_layouts(H_q, H_kv, D):
    w = make_workload("8b", B=5, H_q=H_q, H_kv=H_kv, D=D, ctx_range=(1, 300), steps=2)
    _run_and_compare(w, 0)
    _run_and_compare(w, 32)


@pytest.mark.parametrize("partition", [0, 32, 512])
def test_quantized_cache_with_sinks_reduced(partition):
    w = make_workload("long_quant", B=3, ctx_fixed=611, steps=2)
    _run_and_compare(w, partition)


def test_quantized_short_contexts_inside_sink_range():
    # cached lengths 0..5 with 4 sinks: some sequences attend to sinks only
    w = make_workload("long_quant", B=6, ctx_list=[0, 1, 2, 3, 4, 5], steps=2)
    _run_and_compare(w, 0)
    _run_and_compare(w, 16)


def test_bf16_with_sinks():
    w = make_workload("8b", B=4, ctx_range=(1, 80), steps=2, num_sink=4)
    _run_and_compare(w, 0)


def test_prefix_sharing_fork_with_copy_on_write_then_steady_step():
    # prefix of 40 tokens ends inside its third block: every sequence forks there
    w = make_workload("prefix_cow", B=6, prefix=40, suffix_range=(5, 60), steps=1)
    g, o = GpuState(w), OracleState(w)
    pos = w.positions(0)  # 40 for everybody: the shared, partly filled block is written
    gp = g.prepare(pos)
    op = o.prepare(pos)
    assert len(gp) == w.B and [tuple(p) for p in gp.tolist()] == [tuple(p) for p in op]
    g.append(w.k_new[0], w.v_new[0], pos)
    o.append(w.k_new[0], w.v_new[0], pos)
    ctx = w.context_lens(0)
    for part in (0, 16, 512):
        assert_attention_close(to_f64(g.attend(w.q[0], ctx, part)), o.attend(w.q[0], ctx), f"fork p{part}")
    assert_pools_equal(g, o)
    # the shared source block was copied, never written: its refcount keeps the prefix owner
    src = int(gp[0][0])
    assert g.bm.refcount(src) == 1 and o.pool.refcount[src] == 1
    # private suffixes, then a steady-state step (no copy needed)
    seqs, poss, rows = [], [], []
    off = 0
    for s in range(w.B):
        n = int(w.suffix_len[s])
        seqs += [s] * (n - 1)
        poss += list(range(w.prefix + 1, w.prefix + n))
        rows += list(range(off + 1, off + n))
        off += n
    seqs = np.array(seqs, dtype=np.int32)
    poss = np.array(poss, dtype=np.int32)
    idx = torch.tensor(rows, dtype=torch.long)
    for state in (g, o):
        # tokens beyond the fork go to private blocks: make every slot writable first
        for p in range(w.prefix + 1, w.prefix + int(w.suffix_len.max())):
            step_pos = np.where(p < w.prefix + w.suffix_len, p, -1).astype(np.int32)
            assert len(state.prepare(step_pos)) == 0
        state.bulk_append(w.suffix_k[idx], w.suffix_v[idx], seqs, poss)
    steady = (w.prefix + w.suffix_len).astype(np.int32)
    for state in (g, o):
        assert len(state.prepare(steady)) == 0
        state.append(w.k_new[0], w.v_new[0], steady)
    ctx2 = steady + 1
    ref = o.attend(w.q[0], ctx2)
    for part in (0, 32):
        assert_attention_close(to_f64(g.attend(w.q[0], ctx2, part)), ref, f"steady p{part}")
    assert g.err_bits() == 0
    assert_pools_equal(g, o)


def test_empty_and_single_token_contexts():
    w = make_workload("8b", B=5, ctx_list=[0, 0, 1, 15, 16], steps=1, H_q=8, H_kv=2, D=128)
    g, o = GpuState(w), OracleState(w)
    pos = w.positions(0).copy()
    pos[0] = -1  # padding row: nothing appended, context 0
    ctx = w.context_lens(0).copy()
    ctx[0] = 0
    g.prepare(pos), o.prepare(pos)
    g.append(w.k_new[0], w.v_new[0], pos)
    o.append(w.k_new[0], w.v_new[0], pos)
    for part in (0, 16):
        out = to_f64(g.attend(w.q[0], ctx, part))
        ref = o.attend(w.q[0], ctx)
        assert np.all(out[0] == 0.0)
        assert_attention_close(out, ref, "edge")
        # a single cached token: the output is that token's V (rounded to bf16)
        v1 = o.cache.gather(1, o.tables[1], 1)[1]
        assert np.allclose(out[1], np.repeat(v1[0], w.G, axis=0), atol=1e-2)
    assert g.err_bits() == 0
    assert_pools_equal(g, o)


def test_bad_block_id_sets_flag_and_zeroes_only_that_row():
    w = make_workload("8b", B=4, ctx_list=[40, 40, 40, 40], steps=1, H_q=8, H_kv=2, D=128)
    g, o = GpuState(w), OracleState(w)
    pos = w.positions(0)
    g.prepare(pos), o.prepare(pos)
    g.append(w.k_new[0], w.v_new[0], pos)
    o.append(w.k_new[0], w.v_new[0], pos)
    ctx = w.context_lens(0)
    ref = o.attend(w.q[0], ctx)
    g.tables_dev[2, 1] = w.num_blocks + 5  # corrupt one entry of sequence 2
    for part in (0, 16):
        g.err.zero_()
        out = to_f64(g.attend(w.q[0], ctx, part))
        assert g.err_bits() & N.PA_EFLAG_BAD_BLOCK_ID
        assert np.all(out[2] == 0.0)
        keep = [0, 1, 3]
        assert_attention_close(out[keep], ref[keep], "other rows")


def test_context_overflow_sets_flag_and_zeroes_row():
    w = make_workload("8b", B=3, ctx_list=[20, 20, 20], steps=1, H_q=8, H_kv=2, D=64)
    g, o = GpuState(w), OracleState(w)
    pos = w.positions(0)
    g.prepare(pos), o.prepare(pos)
    g.append(w.k_new[0], w.v_new[0], pos)
    o.append(w.k_new[0], w.v_new[0], pos)
    ctx = w.context_lens(0).copy()
    ref = o.attend(w.q[0], ctx)
    bad_ctx = ctx.copy()
    bad_ctx[1] = w.max_blocks * 16 + 1  # longer than the table can address
    for part in (0, 16):
        g.err.zero_()
        out = to_f64(g.attend(w.q[0], bad_ctx, part, max_ctx=int(bad_ctx.max())))
        assert g.err_bits() & N.PA_EFLAG_CTX_OVERFLOW
        assert np.all(out[1] == 0.0)
        assert_attention_close(out[[0, 2]], ref[[0, 2]], "other rows")
    # an append beyond the table sets the flag and writes nothing
    g.err.zero_()
    before = g.pools()
    far = np.array([-1, w.max_blocks * 16, -1], dtype=np.int32)
    g.append(w.k_new[0], w.v_new[0], far)
    assert g.err_bits() & N.PA_EFLAG_CTX_OVERFLOW
    after = g.pools()
    assert np.array_equal(before[0], after[0]) and np.array_equal(before[1], after[1])


def test_bulk_append_rejects_bad_sequence_index():
    w = make_workload("tiny")
    g = GpuState(w, fill=False)
    seq = np.array([0, 9, -1], dtype=np.int32)
    pos = np.array([0, 0, 0], dtype=np.int32)
    g.bulk_append(w.fill_k[:3], w.fill_v[:3], seq, pos)
    assert g.err_bits() & N.PA_EFLAG_BAD_SEQ


def test_block_copy_skips_out_of_range_pairs():
    w = make_workload("tiny")
    g = GpuState(w)
    before = g.pools()
    pairs = torch.tensor([[0, w.num_blocks], [-1, 3]], dtype=torch.int32, device="cuda")
    N.pa_block_copy(g.desc, g.k, g.v, pairs, 2, g.err)
    assert g.err_bits() & N.PA_EFLAG_BAD_BLOCK_ID
    after = g.pools()
    assert np.array_equal(before[0], after[0]) and np.array_equal(before[1], after[1])


def test_host_errors_enqueue_nothing():
    w = make_workload("tiny")
    g = GpuState(w)
    ctx = torch.from_numpy(w.context_lens(0)).cuda()
    out = torch.zeros((w.B, w.H_q, w.D), dtype=torch.bfloat16, device="cuda")
    need = N.pa_decode_workspace_size(g.desc, 300, 0)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    with pytest.raises(N.PaError) as e:
        N.pa_decode_attention(g.desc, out, w.q[0].cuda(), g.k, g.v, g.tables_dev, ctx, 300, w.scale, 0, ws,
                              need - 1, g.err)
    assert e.value.status == N.PA_ERR_WORKSPACE_TOO_SMALL
    with pytest.raises(N.PaError) as e:
        N.pa_decode_attention(g.desc, out, w.q[0].cuda(), g.k, g.v, g.tables_dev, ctx, 300, w.scale, 24, ws,
                              need, g.err)
    assert e.value.status == N.PA_ERR_INVALID_ARG  # partition not a multiple of 16
    with pytest.raises(N.PaError) as e:
        N.pa_decode_attention(g.desc, out, 0, g.k, g.v, g.tables_dev, ctx, 300, w.scale, 0, ws, need, g.err)
    assert e.value.status == N.PA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(out == 0)

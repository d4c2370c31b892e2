"""Sliding-window decode and prefill on the GPU vs the oracle, through the C ABI.

Untitled KV-cache article at ldpk.cn/news/58971 §5.3: each query attends only the most recent W
positions and the cache keeps only those.  Every decode step here appends, attends with the
window, then releases the blocks behind the window (pa_bm_slide_window vs the oracle pool's
slide_window), so later steps reuse released blocks.  Released table entries are -1 and the
positions before the first window were never written (NaN), so a kernel that read outside the
window would set PA_EFLAG_BAD_BLOCK_ID or produce NaN.  Pools and tables must match the oracle
bit for bit; attention within max-abs 2e-2 / mean-abs 2e-3 of the fp64 oracle.
"""

import numpy as np
import pytest
import torch

import oracle as O
from paged_kv_cache_table_gb300 import native as N
from paged_kv_cache_table_gb300.workloads import bf16_bits, make_prefill_workload, make_workload

from harness import (BF16_NAN, GpuState, OracleState, assert_attention_close, assert_pools_equal, to_f64)
from test_gpu_prefill import PrefillGpu

pytestmark = pytest.mark.gpu


def _run_and_compare(w, partition=0):
    g = GpuState(w)
    o = OracleState(w)
    for i in range(w.steps):
        out, gpairs = g.step(i, partition)
        ref, opairs = o.step(i)
        assert [tuple(p) for p in gpairs.tolist()] == [tuple(p) for p in opairs]
        assert_attention_close(to_f64(out), ref, f"{w.name} window {w.window} step {i} partition {partition}")
        assert g.bm.num_free() == o.pool.num_free()
    assert g.err_bits() == 0
    assert_pools_equal(g, o)
    return g, o


@pytest.mark.parametrize("window", [1, 16, 40, 333])
@pytest.mark.parametrize("partition", [0, 32, 512])
def test_sliding_decode_8b_shape_reduced(window, partition):
    # 20 steps: windows cross block edges, blocks are released and handed out again
    w = make_workload("8b", B=7, ctx_range=(1, 700), steps=20, window=window)
    _run_and_compare(w, partition)


def test_sliding_decode_gqa8_and_d64():
    _run_and_compare(make_workload("70b", B=3, ctx_fixed=527, steps=4, window=100), 0)
    _run_and_compare(make_workload("8b", B=5, H_q=16, H_kv=2, D=64, ctx_range=(1, 300), steps=6, window=50), 0)
    _run_and_compare(make_workload("8b", B=5, H_q=16, H_kv=2, D=64, ctx_range=(1, 300), steps=6, window=50), 48)


@pytest.mark.parametrize("partition", [0, 32])
def test_sliding_decode_quantized_with_sinks(partition):
    # long contexts: the sinks fall outside the window
    _run_and_compare(make_workload("long_quant", B=3, ctx_fixed=611, steps=3, window=64), partition)
    # short contexts: sinks partly inside the window
    _run_and_compare(make_workload("long_quant", B=6, ctx_list=[0, 1, 2, 3, 4, 9], steps=4, window=3), partition)


def test_bf16_sinks_with_window():
    _run_and_compare(make_workload("8b", B=4, ctx_range=(1, 80), steps=5, num_sink=4, window=6), 0)


def test_window_covering_the_context_equals_full_attention_bitwise():
    base = make_workload("8b", B=6, ctx_range=(1, 400), steps=1)
    wide = make_workload("8b", B=6, ctx_range=(1, 400), steps=1, window=1 << 20)
    outs = []
    for w in (base, wide):
        g = GpuState(w)
        out, _ = g.step(0)
        assert g.err_bits() == 0
        outs.append(out.view(torch.int16).cpu().numpy())
    assert np.array_equal(outs[0], outs[1])


def _oracle_prefill_window(w, window):
    qv = O.bf16_bits_to_f64(bf16_bits(w.q))
    qs = w.q_start()
    out = np.zeros((int(qs[-1]), w.H_q, w.D))
    fk, fv = bf16_bits(w.fill_k), bf16_bits(w.fill_v)
    nk, nv = bf16_bits(w.new_k), bf16_bits(w.new_v)
    for s in range(w.B):
        ci = np.nonzero(w.fill_seq == s)[0]
        ci = ci[np.argsort(w.fill_pos[ci])]
        ni = np.arange(qs[s], qs[s + 1])
        K = O.bf16_bits_to_f64(np.concatenate([fk[ci], nk[ni]]))
        V = O.bf16_bits_to_f64(np.concatenate([fv[ci], nv[ni]]))
        out[qs[s]:qs[s + 1]] = O.prefill_attention(qv[qs[s]:qs[s + 1]], K, V, w.scale, int(w.ctx_old[s]), window)
    return out


def _windowed_prefill(w, window):
    """A PrefillGpu for workload w under window W, its pool as the previous step's release left it."""
    g = PrefillGpu(w)
    g.desc = N.make_desc(w.B, w.H_q, w.H_kv, w.D, w.num_blocks, w.max_blocks, sliding_window=window)
    # What the previous step's release left: blocks wholly before position ctx_old - W are gone
    # (-1), and the positions of the first kept block that no query of the chunk reads are
    # overwritten with NaN.
    nan_pos, nan_seq = [], []
    for s in range(w.B):
        first = int(w.ctx_old[s])
        gone = max(0, first - window) // 16
        g.tables[s, :gone] = -1
        lo = max(0, first - window + 1)  # window start of the chunk's first query
        for p in range(gone * 16, lo):
            nan_seq.append(s)
            nan_pos.append(p)
    if nan_seq:
        rows = torch.full((len(nan_seq), w.H_kv, w.D), BF16_NAN, dtype=torch.int16).view(torch.bfloat16).cuda()
        N.pa_kv_append_tokens(g.desc, g.k, g.v, rows, rows, len(nan_seq),
                              torch.tensor(nan_seq, dtype=torch.int32).cuda(),
                              torch.tensor(nan_pos, dtype=torch.int32).cuda(), g.tables, g.err)
    return g


@pytest.mark.parametrize("window", [1, 7, 16, 45, 200])
@pytest.mark.parametrize("H_q,H_kv,D", [(8, 2, 64), (32, 8, 128), (8, 8, 128)])
def test_sliding_prefill_matches_oracle(window, H_q, H_kv, D):
    w = make_prefill_workload(H_q=H_q, H_kv=H_kv, D=D, cached_list=[0, 17, 100, 300], chunk_list=[5, 16, 33, 70])
    g = _windowed_prefill(w, window)
    out = g.run()
    assert int(g.err.item()) == 0
    assert_attention_close(out, _oracle_prefill_window(w, window), f"prefill window {window}")


@pytest.mark.parametrize("window", [64, 200, 600])
@pytest.mark.parametrize("H_q,H_kv", [(32, 8), (64, 8), (16, 16)])
def test_sliding_prefill_long_chunks(window, H_q, H_kv):
    """Chunks spanning several tensor-core work items (d 128): later tiles start their keys
    inside the window, the first key tile partly before it."""
    w = make_prefill_workload(H_q=H_q, H_kv=H_kv, D=128, cached_list=[0, 500, 1000, 37],
                              chunk_list=[300, 257, 129, 411], seed=21)
    g = _windowed_prefill(w, window)
    out = g.run()
    assert int(g.err.item()) == 0
    assert_attention_close(out, _oracle_prefill_window(w, window), f"prefill window {window}, long chunks")

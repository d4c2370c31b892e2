"""INT4 KV cache on the GPU vs the oracle, through the C ABI.

Untitled KV-cache article at ldpk.cn/news/58971 §5.2: int4 codes with a scale and a zero point
(per 32 dims of every token's head row here).  Appended codes and group parameters must match
the oracle's encoder bit for bit (whole pools, read by the documented PA_INT4 byte layout, with
never-written slots holding all-ones codes and NaN-scale parameters), copy-on-write must carry
the parameters, and attention must be within max-abs 2e-2 / mean-abs 2e-3 of the fp64 oracle
over the decoded values.
"""

import numpy as np
import pytest

from paged_kv_cache_table_gb300 import native as N
from paged_kv_cache_table_gb300.workloads import make_workload

from harness import GpuState, OracleState, assert_attention_close, assert_pools_equal, to_f64

pytestmark = pytest.mark.gpu


def _run_and_compare(w, partition=0):
    g = GpuState(w)
    o = OracleState(w)
    for i in range(w.steps):
        out, gpairs = g.step(i, partition)
        ref, opairs = o.step(i)
        assert [tuple(p) for p in gpairs.tolist()] == [tuple(p) for p in opairs]
        assert_attention_close(to_f64(out), ref, f"{w.name} step {i} partition {partition}")
    assert g.err_bits() == 0
    assert_pools_equal(g, o)
    return g, o


@pytest.mark.parametrize("partition", [0, 16, 48, 512, 1 << 20])
def test_int4_8b_shape_reduced(partition):
    _run_and_compare(make_workload("int4_8b", B=7, ctx_range=(1, 700), steps=3), partition)


@pytest.mark.parametrize("H_q,H_kv", [(8, 2), (64, 8), (16, 16), (12, 6), (4, 4), (32, 4)])
def test_int4_head_layouts(H_q, H_kv):
    w = make_workload("int4_8b", B=5, H_q=H_q, H_kv=H_kv, ctx_range=(1, 300), steps=2)
    _run_and_compare(w, 0)
    _run_and_compare(w, 32)


def test_int4_sinks_and_short_contexts():
    _run_and_compare(make_workload("int4_8b", B=6, ctx_list=[0, 1, 2, 3, 4, 37], steps=3, num_sink=4), 0)
    _run_and_compare(make_workload("int4_8b", B=4, ctx_range=(1, 100), steps=2, num_sink=4), 32)


def test_int4_sliding_window():
    _run_and_compare(make_workload("int4_8b", B=6, ctx_range=(1, 500), steps=12, window=40), 0)


def test_int4_copy_on_write_carries_parameters():
    # prefix of 40 tokens ends inside its third block: every sequence copies it at the fork
    w = make_workload("prefix_cow", B=3, prefix=40, suffix_range=(1, 30), steps=2, kv="int4")
    g = GpuState(w)
    o = OracleState(w)
    lens = w.suffix_len.astype(np.int64)
    for p in range(w.prefix, w.prefix + int(lens.max())):
        pos = np.where(p < w.prefix + lens, p, -1).astype(np.int32)
        gp = g.prepare(pos)
        op = o.prepare(pos)
        assert [tuple(x) for x in gp.tolist()] == [tuple(x) for x in op]
        seq = np.nonzero(pos >= 0)[0]
        idx = np.array([int(lens[:s].sum()) + (p - w.prefix) for s in seq])
        g.bulk_append(w.suffix_k[idx], w.suffix_v[idx], seq, pos[seq])
        o.bulk_append(w.suffix_k[idx], w.suffix_v[idx], seq, pos[seq])
    w.ctx_old = (w.prefix + lens).astype(np.int32)
    for i in range(w.steps):
        out, _ = g.step(i)
        ref, _ = o.step(i)
        assert_attention_close(to_f64(out), ref, f"int4 prefix step {i}")
    assert g.err_bits() == 0
    assert_pools_equal(g, o)



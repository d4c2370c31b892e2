"""Per-token K scales on the GPU (PA_FP8_E4M3_TOKEN K, INT8 V) against the oracle's "e4m3_tok"
cache, through the C ABI.

Untitled KV-cache article at ldpk.cn/news/58971 §5.2: K develops outlier channels, so a scale per
tensor or per head fails on long contexts; here every token's K head row carries its own scale.
The append must write the same codes and the same fp32 scale bits as the oracle (whole pools are
compared, never-written slots included), copy-on-write must carry the scales with the block, and
attention must stay within max-abs 2e-2 / mean-abs 2e-3 of the fp64 oracle in every split mode,
with sinks, under a sliding window and through pa_decode_step.  The kernels never read a slot or a
scale outside the attended positions: the pools start filled with NaN codes and huge scales."""

import numpy as np
import pytest
import torch

from paged_kv_cache_table_gb300 import native as N
from paged_kv_cache_table_gb300.workloads import make_workload

from harness import GpuState, OracleState, assert_attention_close, assert_pools_equal, to_f64

pytestmark = pytest.mark.gpu


def _run(w, partition, steps=None, fused=False):
    g, o = GpuState(w), OracleState(w)
    for i in range(w.steps if steps is None else steps):
        if fused:
            pos = w.positions(i)
            gp = g.prepare(pos)
            out = g.decode_step(w.k_new[i], w.v_new[i], w.q[i], pos, w.context_lens(i), partition)
            if w.window:
                g.slide(w.context_lens(i))
        else:
            out, gp = g.step(i, partition)
        ref, op = o.step(i)
        assert [tuple(p) for p in gp.tolist()] == [tuple(p) for p in op]
        assert_attention_close(to_f64(out), ref, f"{w.name} step {i} partition {partition}")
    assert g.err_bits() == 0
    assert_pools_equal(g, o)
    return g, o


@pytest.mark.parametrize("partition", [0, 16, 48, 512])
def test_token_scales_match_oracle(partition):
    w = make_workload("long_quant_tok", B=6, ctx_range=(1, 700), steps=3)
    _run(w, partition)


def test_token_scales_through_the_decode_step_call():
    w = make_workload("long_quant_tok", B=5, ctx_range=(3, 500), steps=3)
    _run(w, 0, fused=True)


def test_token_scales_short_contexts_inside_sink_range():
    w = make_workload("long_quant_tok", B=6, ctx_list=[0, 1, 2, 3, 4, 5], steps=2)
    _run(w, 0)
    _run(w, 16)


def test_token_scales_with_outlier_tokens():
    """Rows with one channel 10^4 times larger than the rest: each token keeps its own range."""
    w = make_workload("long_quant_tok", B=3, ctx_fixed=300, steps=2)
    w.fill_k[::5, :, 7] = 400.0
    w.k_new[:, :, :, 7] = -300.0
    _run(w, 0)


@pytest.mark.parametrize("H_q,H_kv", [(16, 4), (48, 12), (64, 16)])
def test_token_scales_head_layouts(H_q, H_kv):
    w = make_workload("long_quant_tok", B=4, H_q=H_q, H_kv=H_kv, ctx_range=(1, 300), steps=2)
    _run(w, 0)
    _run(w, 32)


def test_token_scales_sliding_window():
    w = make_workload("long_quant_tok", B=4, ctx_range=(60, 400), window=50, steps=3)
    _run(w, 0)
    _run(w, 16, fused=True)


def test_token_scales_copy_on_write_fork():
    """A shared prefix ending inside a block: every sequence copies that block (codes and
    scales) before writing its first private token.  (No sinks: the shared prefix is written
    once, through the first sequence, and sink rows are per sequence.)"""
    w = make_workload("prefix_cow", B=5, prefix=40, suffix_range=(5, 30), quant=True, kv="e4m3_tok", steps=1)
    assert w.k_dtype == "e4m3_tok"
    g, o = GpuState(w), OracleState(w)
    pos = w.positions(0)
    gp, op = g.prepare(pos), o.prepare(pos)
    assert len(gp) == w.B and [tuple(p) for p in gp.tolist()] == [tuple(p) for p in op]
    g.append(w.k_new[0], w.v_new[0], pos)
    o.append(w.k_new[0], w.v_new[0], pos)
    ctx = w.context_lens(0)
    for part in (0, 16):
        assert_attention_close(to_f64(g.attend(w.q[0], ctx, part)), o.attend(w.q[0], ctx), f"fork p{part}")
    assert g.err_bits() == 0
    assert_pools_equal(g, o)


def test_token_scale_shapes_rejected_on_the_host():
    w = make_workload("long_quant_tok", B=2, ctx_fixed=20, H_q=12, H_kv=6, steps=1)
    k = torch.zeros(w.num_blocks * 16 * w.H_kv * 132, dtype=torch.uint8, device="cuda")
    v = torch.zeros(w.num_blocks * 16 * w.H_kv * 128, dtype=torch.uint8, device="cuda")
    vs = w.v_scales.cuda()
    desc = N.make_desc(w.B, w.H_q, w.H_kv, w.D, w.num_blocks, w.max_blocks, "e4m3_tok", "int8", None, vs)
    assert N.pa_decode_workspace_size(desc, 64, 0) == 0  # 6 KV heads: scales rows not 16-byte multiples
    with pytest.raises(N.PaError) as e:
        N.pa_kv_append(desc, k, v, w.k_new[0].cuda(), w.v_new[0].cuda(), torch.zeros((2, w.max_blocks),
                       dtype=torch.int32, device="cuda"), torch.zeros(2, dtype=torch.int32, device="cuda"))
    assert e.value.status == N.PA_ERR_UNSUPPORTED

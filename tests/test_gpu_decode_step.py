"""pa_decode_step against pa_kv_append followed by pa_decode_attention.

The step call overlaps the append with the attention's streaming of every block that the append
does not write, and waits for the append only before the blocks holding the appended positions.
Its results must be the ones of the two calls made one after the other: every output bit and every
byte of the pools (codes, group parameters, sink rows), step after step, for every cache kind,
both split modes, sinks, sliding windows and copy-on-write forks.  The separate calls are pinned to
the oracle by the other GPU tests, so bit equality with them is the parity bar here.
"""

import numpy as np
import pytest
import torch

import paged_kv_cache_table_gb300 as P
from paged_kv_cache_table_gb300.workloads import make_workload

from harness import GpuState

pytestmark = pytest.mark.gpu


def _step_fused(g: GpuState, i: int, partition: int):
    w = g.w
    pos = np.ascontiguousarray(w.positions(i), dtype=np.int32)
    pairs = g.prepare(pos)
    ctx = np.ascontiguousarray(w.context_lens(i), dtype=np.int32)
    max_ctx = int(ctx.max())
    out = torch.full((w.B, w.H_q, w.D), float("nan"), dtype=torch.bfloat16, device=g.dev)
    nbytes = P.pa_decode_workspace_size(g.desc, max_ctx, partition)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=g.dev)
    P.pa_decode_step(g.desc, out, w.q[i].to(g.dev), g.k, g.v, w.k_new[i].to(g.dev), w.v_new[i].to(g.dev),
                     g.tables_dev, torch.from_numpy(pos).to(g.dev), torch.from_numpy(ctx).to(g.dev), max_ctx,
                     w.scale, partition, ws, nbytes, g.err)
    if w.window:
        g.slide(w.context_lens(i))
    return out, pairs


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy()


def _compare(w, partition=0):
    sep, fused = GpuState(w), GpuState(w)
    for i in range(len(w.q)):
        o1, p1 = sep.step(i, partition)
        o2, p2 = _step_fused(fused, i, partition)
        assert np.array_equal(np.asarray(p1), np.asarray(p2))
        assert np.array_equal(_bits(o1), _bits(o2)), f"step {i}: outputs differ"
        for a, b in zip(sep.pools(), fused.pools()):
            if a is not None:
                assert np.array_equal(a, b), f"step {i}: pools differ"
        assert sep.err_bits() == fused.err_bits() == 0


@pytest.mark.parametrize("partition", [0, 512])
def test_step_equals_append_then_attention_bf16(partition):
    _compare(make_workload("8b", B=7, ctx_range=(1, 700), steps=3), partition)


def test_step_tiny_d64():
    _compare(make_workload("tiny"))


@pytest.mark.parametrize("partition", [0, 512])
def test_step_8bit_with_sinks(partition):
    _compare(make_workload("long_quant", B=3, ctx_fixed=611, steps=2), partition)


def test_step_8bit_contexts_inside_the_sink_range():
    # the appended positions are sink positions: the step also writes the bf16 sink rows
    _compare(make_workload("long_quant", B=6, ctx_list=[0, 1, 2, 3, 4, 5], steps=3))


def test_step_int4():
    _compare(make_workload("int4_8b", B=5, ctx_range=(1, 900), steps=3))


def test_step_int4_with_sinks():
    _compare(make_workload("int4_8b", B=6, ctx_list=[0, 1, 2, 3, 4, 37], steps=3, num_sink=4))


@pytest.mark.parametrize("partition", [0, 48])
def test_step_sliding_window(partition):
    _compare(make_workload("8b", B=5, H_q=16, H_kv=2, D=64, ctx_range=(1, 300), steps=6, window=50), partition)


def test_step_prefix_fork_with_copy_on_write():
    _compare(make_workload("prefix_cow", B=6, prefix=40, suffix_range=(5, 60), steps=2))


def test_step_empty_and_single_token_contexts():
    _compare(make_workload("8b", B=5, ctx_list=[0, 0, 1, 15, 16], steps=2, H_q=8, H_kv=2, D=128))


def test_step_host_errors_enqueue_nothing():
    w = make_workload("tiny")
    g = GpuState(w)
    before = g.pools()
    pos = torch.from_numpy(np.ascontiguousarray(w.positions(0), dtype=np.int32)).cuda()
    ctx = torch.from_numpy(np.ascontiguousarray(w.context_lens(0), dtype=np.int32)).cuda()
    out = torch.empty((w.B, w.H_q, w.D), dtype=torch.bfloat16, device="cuda")
    nbytes = P.pa_decode_workspace_size(g.desc, int(w.context_lens(0).max()), 0)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    kn, vn, q = w.k_new[0].cuda(), w.v_new[0].cuda(), w.q[0].cuda()
    bad = [
        dict(workspace_bytes=nbytes - 1),          # workspace too small
        dict(q=None),                              # missing attention input
        dict(ws_off=8),                            # misaligned workspace
        dict(scale=float("nan")),                  # non-finite scale
    ]
    for b in bad:
        ws_arg = ws.data_ptr() + b.get("ws_off", 0)
        with pytest.raises(P.PaError):
            P.pa_decode_step(g.desc, out, b.get("q", q), g.k, g.v, kn, vn, g.tables_dev, pos, ctx,
                             int(w.context_lens(0).max()), b.get("scale", w.scale), 0, ws_arg,
                             b.get("workspace_bytes", nbytes), g.err)
    torch.cuda.synchronize()
    for a, c in zip(before, g.pools()):
        if a is not None:
            assert np.array_equal(a, c), "a rejected step must not have appended"

"""The balanced split's partial rows, their prefix sums and the merge through the workspace.

A sequence whose blocks fall to several CTAs leaves one partial row per CTA in the caller's
workspace, which the library never clears: results must not depend on what the workspace held
before (zeros, all ones, random bytes, the rows of an earlier call with other context lengths),
and a call captured once in a CUDA graph must, on every replay with new queries, equal an eager
call.  Each case is checked bit for bit against an eager call on a fresh workspace, and against
the oracle, including sequences split over dozens of CTAs (several rounds of eight partials per
merged row) and empty contexts (zero rows).
"""

import numpy as np
import pytest
import torch

from paged_kv_cache_table_gb300 import native as P
from paged_kv_cache_table_gb300.workloads import make_workload

from harness import GpuState, OracleState, assert_attention_close, to_f64

pytestmark = pytest.mark.gpu


def _setup(w):
    g, o = GpuState(w), OracleState(w)
    pos = w.positions(0)
    g.prepare(pos), o.prepare(pos)
    g.append(w.k_new[0], w.v_new[0], pos)
    o.append(w.k_new[0], w.v_new[0], pos)
    return g, o


def _attend(g, q, ctx_dev, max_ctx, ws, out=None):
    w = g.w
    if out is None:
        out = torch.full((w.B, w.H_q, w.D), float("nan"), dtype=torch.bfloat16, device=g.dev)
    P.pa_decode_attention(g.desc, out, q, g.k, g.v, g.tables_dev, ctx_dev, max_ctx, w.scale, 0, ws,
                          ws.numel(), g.err)
    return out


CASES = {
    # many short sequences: most split over two or three CTAs
    "short": dict(B=24, ctx_range=(1, 700)),
    # two long sequences: each split over about 76 CTAs
    "long": dict(B=2, ctx_fixed=9000),
    # a long one among short ones and empty ones
    "mixed": dict(B=6, ctx_list=[0, 5000, 1, 300, 0, 17]),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_result_does_not_depend_on_workspace_contents(case):
    w = make_workload("8b", steps=1, **CASES[case])
    g, o = _setup(w)
    ctx = w.context_lens(0).copy()
    if case == "mixed":
        ctx[[0, 4]] = 0
    ref = o.attend(w.q[0], ctx)
    q = w.q[0].to(g.dev)
    ctx_dev = torch.from_numpy(np.ascontiguousarray(ctx, dtype=np.int32)).to(g.dev)
    max_ctx = int(ctx.max())
    nbytes = P.pa_decode_workspace_size(g.desc, max_ctx, 0)
    ws0 = torch.zeros(nbytes, dtype=torch.uint8, device=g.dev)
    base = _attend(g, q, ctx_dev, max_ctx, ws0)
    assert_attention_close(to_f64(base), ref, f"{case} vs oracle")
    if case == "mixed":
        assert np.all(to_f64(base)[[0, 4]] == 0.0)
    gen = torch.Generator(device="cpu").manual_seed(5)
    fills = {
        "ones": torch.full((nbytes,), 0xFF, dtype=torch.uint8),
        "random": torch.randint(0, 256, (nbytes,), generator=gen, dtype=torch.uint8),
    }
    for name, fill in fills.items():
        ws = fill.to(g.dev)
        out = _attend(g, q, ctx_dev, max_ctx, ws)
        assert torch.equal(out, base), name
        # the same workspace again, holding the rows of the call just made
        out = _attend(g, q, ctx_dev, max_ctx, ws)
        assert torch.equal(out, base), name + " reused"
    # an earlier call with other context lengths (other splits) on the same workspace
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=g.dev)
    other = np.maximum(ctx // 3, 0).astype(np.int32)
    _attend(g, q, torch.from_numpy(other).to(g.dev), max_ctx, ws)
    assert torch.equal(_attend(g, q, ctx_dev, max_ctx, ws), base)
    assert g.err_bits() == 0


def test_graph_replay_matches_eager_calls():
    """One call captured in a CUDA graph, replayed with new queries in the captured buffer, must
    equal an eager call each time."""
    w = make_workload("8b", steps=1, B=12, ctx_range=(200, 3000))
    g, o = _setup(w)
    ctx = w.context_lens(0)
    ctx_dev = torch.from_numpy(np.ascontiguousarray(ctx, dtype=np.int32)).to(g.dev)
    max_ctx = int(ctx.max())
    nbytes = P.pa_decode_workspace_size(g.desc, max_ctx, 0)
    ws_graph = torch.empty(nbytes, dtype=torch.uint8, device=g.dev)
    ws_eager = torch.empty(nbytes, dtype=torch.uint8, device=g.dev)
    q_buf = w.q[0].to(g.dev)
    out_buf = torch.empty((w.B, w.H_q, w.D), dtype=torch.bfloat16, device=g.dev)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _attend(g, q_buf, ctx_dev, max_ctx, ws_graph, out_buf)  # warm-up outside the capture
        side.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            _attend(g, q_buf, ctx_dev, max_ctx, ws_graph, out_buf)
    torch.cuda.synchronize()
    gen = torch.Generator().manual_seed(11)
    for r in range(4):
        q_new = (torch.randn((w.B, w.H_q, w.D), generator=gen) * 0.5).to(torch.bfloat16)
        q_buf.copy_(q_new.to(g.dev))
        graph.replay()
        torch.cuda.synchronize()
        eager = _attend(g, q_buf, ctx_dev, max_ctx, ws_eager)
        torch.cuda.synchronize()
        assert torch.equal(out_buf, eager), f"replay {r}"
        if r == 3:
            assert_attention_close(to_f64(out_buf), o.attend(q_new, ctx), "replay vs oracle")
    assert g.err_bits() == 0

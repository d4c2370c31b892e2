"""The allocation-free decode entry point, for callers that cannot allocate device memory when
they call into the library (a plugin inside a framework that owns all device memory, a
latency-critical path where cudaMalloc/cudaFree could synchronise the device, a caller that
cannot recover from an out-of-memory failure mid-step).  It must give the same output as the
workspace entry point on consecutive calls, and reject problems too large for its static
scratch.  This file is collected last on purpose: it also runs after the other GPU tests."""

import numpy as np
import pytest
import torch

from paged_kv_cache_table_gb300 import native as N
from paged_kv_cache_table_gb300.workloads import make_workload

from harness import ATOL_MAX, ATOL_MEAN, GpuState, to_f64

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 8 << 20


def _noalloc(g, q, ctx, partition):
    w = g.w
    out = torch.full((w.B, w.H_q, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    N.pa_decode_attention_noalloc(g.desc, out, q.cuda(), g.k, g.v, g.tables_dev,
                                  torch.from_numpy(ctx).cuda(), int(ctx.max()), w.scale, partition, g.err)
    return out


@pytest.mark.parametrize("partition", [0, 512])
def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row(partition):
    w = make_workload("8b", B=9, ctx_range=(1, 900), steps=2)
    g = GpuState(w)
    for i in range(2):  # two consecutive calls: the second sees the first one's leftovers
        pos = w.positions(i)
        g.prepare(pos)
        g.append(w.k_new[i], w.v_new[i], pos)
        ctx = w.context_lens(i)
        ref = to_f64(g.attend(w.q[i], ctx, partition))
        got = to_f64(_noalloc(g, w.q[i], ctx, partition))
        assert np.all(np.isfinite(got))
        err = np.abs(got - ref)
        assert err.max() <= ATOL_MAX and err.mean() <= ATOL_MEAN, (i, err.max(), err.mean())
    assert g.err_bits() == 0


def test_noalloc_quantized_cache_matches():
    w = make_workload("long_quant", B=3, ctx_fixed=300, steps=2)
    g = GpuState(w)
    for i in range(2):
        pos = w.positions(i)
        g.prepare(pos)
        g.append(w.k_new[i], w.v_new[i], pos)
        ctx = w.context_lens(i)
        ref = to_f64(g.attend(w.q[i], ctx, 0))
        got = to_f64(_noalloc(g, w.q[i], ctx, 0))
        err = np.abs(got - ref)
        assert err.max() <= ATOL_MAX and err.mean() <= ATOL_MEAN, (i, err.max(), err.mean())
    assert g.err_bits() == 0


def test_noalloc_rejects_problems_beyond_its_static_scratch():
    w = make_workload("tiny")
    g = GpuState(w)
    big_ctx = 1 << 20  # fixed 16-token partitions over a long context need far more than 8 MiB
    assert N.pa_decode_workspace_size(g.desc, big_ctx, 16) > STATIC_SCRATCH_BYTES
    out = torch.zeros((w.B, w.H_q, w.D), dtype=torch.bfloat16, device="cuda")
    ctx = torch.from_numpy(w.context_lens(0)).cuda()
    with pytest.raises(N.PaError) as e:
        N.pa_decode_attention_noalloc(g.desc, out, w.q[0].cuda(), g.k, g.v, g.tables_dev, ctx, big_ctx,
                                      w.scale, 16, g.err)
    assert e.value.status == N.PA_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert torch.all(out == 0)

"""The allocation-free decode entry point, for callers that cannot allocate device memory when
they call into the library (a plugin inside a framework that owns all device memory, a
latency-critical path where cudaMalloc/cudaFree could synchronise the device, a caller that
cannot recover from an out-of-memory failure mid-step).

It runs the same kernels with the same plan as the workspace entry point, so its output must be
bit-identical to it, on consecutive calls, even after a call of another shape has left its
headers and partials all over the shared scratch array; and it must match the oracle, at the
benchmark's full 8b and 70b shapes too.  Problems too large for the static scratch are rejected.
This file is collected last on purpose: it also runs after the other GPU tests."""

import numpy as np
import pytest
import torch

from paged_kv_cache_table_gb300 import native as N
from paged_kv_cache_table_gb300.workloads import make_workload

from harness import GpuState, OracleState, assert_attention_close, reference_all, to_f64

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 8 << 20


def _dirty_the_scratch():
    """One allocation-free call of a different problem (9 sequences, 16-token partitions): nearly
    all of the 8 MiB array is left holding that call's headers and partials."""
    w = make_workload("8b", B=9, ctx_range=(700, 800), steps=1, seed=99)
    g = GpuState(w)
    assert N.pa_decode_workspace_size(g.desc, int(w.context_lens(0).max()), 16) > 7 << 20
    pos = w.positions(0)
    g.prepare(pos)
    g.append(w.k_new[0], w.v_new[0], pos)
    g.attend_noalloc(w.q[0], w.context_lens(0), 16)
    torch.cuda.synchronize()
    assert g.err_bits() == 0


@pytest.mark.parametrize("partition", [0, 512])
def test_noalloc_equals_workspace_entry_point_and_oracle_on_two_calls_in_a_row(partition):
    _dirty_the_scratch()
    w = make_workload("8b", B=9, ctx_range=(1, 900), steps=2)
    g, ora = GpuState(w), OracleState(w)
    for i in range(2):  # two consecutive calls: the second sees the first one's leftovers
        pos = w.positions(i)
        g.prepare(pos)
        g.append(w.k_new[i], w.v_new[i], pos)
        ref, _ = ora.step(i)
        ctx = w.context_lens(i)
        got = g.attend_noalloc(w.q[i], ctx, partition)
        ws = g.attend(w.q[i], ctx, partition)
        assert torch.equal(got.view(torch.int16), ws.view(torch.int16)), f"call {i}: differs from the workspace call"
        assert_attention_close(to_f64(got), ref, f"no-alloc call {i}, partition {partition}")
    assert g.err_bits() == 0


@pytest.mark.slow
@pytest.mark.parametrize("name", ["8b", "70b"])
def test_noalloc_full_size_against_oracle(name):
    """The benchmark's shapes in its launch configuration (balanced split), every row."""
    w = make_workload(name, steps=1)
    ref = reference_all(w, 0)
    _dirty_the_scratch()
    g = GpuState(w)
    ctx = w.context_lens(0)
    assert N.pa_decode_workspace_size(g.desc, int(ctx.max()), 0) <= STATIC_SCRATCH_BYTES
    pos = w.positions(0)
    g.prepare(pos)
    g.append(w.k_new[0], w.v_new[0], pos)
    for call in range(2):
        got = g.attend_noalloc(w.q[0], ctx, 0)
        assert_attention_close(to_f64(got), ref, f"{name} no-alloc, call {call}")
    assert g.err_bits() == 0


def test_noalloc_quantized_cache_matches():
    _dirty_the_scratch()
    w = make_workload("long_quant", B=3, ctx_fixed=300, steps=2)
    g, ora = GpuState(w), OracleState(w)
    for i in range(2):
        pos = w.positions(i)
        g.prepare(pos)
        g.append(w.k_new[i], w.v_new[i], pos)
        ref, _ = ora.step(i)
        ctx = w.context_lens(i)
        got = g.attend_noalloc(w.q[i], ctx, 0)
        assert torch.equal(got.view(torch.int16), g.attend(w.q[i], ctx, 0).view(torch.int16))
        assert_attention_close(to_f64(got), ref, f"8-bit no-alloc call {i}")
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

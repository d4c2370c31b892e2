"""Host-side checks of the test harness itself (no GPU): the full-size reference attends exactly
the positions a decode step attends."""

import numpy as np

import oracle as O
from paged_kv_cache_table_gb300.workloads import make_workload

from harness import OracleState, logical_tokens, reference_all


def test_logical_tokens_cover_the_attended_positions():
    """From position 0 (or the sliding window's start) to the new token: ctx rows in all."""
    cases = [make_workload("tiny", steps=1),
             make_workload("swa", B=3, ctx_range=(5000, 6000), steps=1)]
    for w in cases:
        ctx = w.context_lens(0)
        for s in range(w.B):
            kb, vb, pos0 = logical_tokens(w, s, 0)
            assert pos0 == O.window_start(int(ctx[s]), w.window)
            assert kb.shape[0] == int(ctx[s]) - pos0 == vb.shape[0]


def test_reference_all_equals_the_oracle_pool():
    """The per-sequence reference (logical stream, no pool) gives exactly what the oracle's own
    paged pool gives after the same step, for bf16, 8-bit with sinks and INT4 caches."""
    for w in (make_workload("tiny", steps=1),
              make_workload("long_quant", B=2, ctx_fixed=70, steps=1),
              make_workload("long_quant_tok", B=2, ctx_fixed=70, steps=1),
              make_workload("int4_8b", B=3, ctx_range=(1, 90), H_q=8, H_kv=2, steps=1)):
        ora = OracleState(w)
        out, _ = ora.step(0)
        assert np.array_equal(reference_all(w, 0), out), w.name

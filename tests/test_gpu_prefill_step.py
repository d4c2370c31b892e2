"""pa_prefill_step against pa_kv_append_tokens followed by pa_prefill_attention.

The step call lets the attention kernel's set-up and query copies run while the chunk's append
does, and holds back only its K/V copies.  Its results must be the ones of the two calls made one
after the other: every output bit and every byte of the pools, on both attention kernels (the
tensor-core one for head_dim 128, the warp-MMA one otherwise), under a sliding window, and for
consecutive chunks of the same sequences.  The separate calls are pinned to the oracle by the
other prefill tests, so bit equality with them is the parity bar here.
"""

import numpy as np
import pytest
import torch

from paged_kv_cache_table_gb300 import native as N
from paged_kv_cache_table_gb300.workloads import make_prefill_workload

from harness import BF16_NAN

pytestmark = pytest.mark.gpu


class Pools:
    """Pools holding a workload's cached tokens (not yet its chunk), unused slots NaN."""

    def __init__(self, w, window=0):
        self.w = w
        shape = (w.num_blocks * 16, w.H_kv, w.D)
        self.k = torch.full(shape, BF16_NAN, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        self.v = torch.full(shape, BF16_NAN, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        self.desc = N.make_desc(w.B, w.H_q, w.H_kv, w.D, w.num_blocks, w.max_blocks, sliding_window=window)
        self.tables = torch.from_numpy(w.tables).cuda()
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        if len(w.fill_seq):
            N.pa_kv_append_tokens(self.desc, self.k, self.v, w.fill_k.cuda(), w.fill_v.cuda(), len(w.fill_seq),
                                  torch.from_numpy(w.fill_seq).cuda(), torch.from_numpy(w.fill_pos).cuda(),
                                  self.tables, self.err)

    def bits(self):
        torch.cuda.synchronize()
        return self.k.view(torch.int16).cpu().numpy(), self.v.view(torch.int16).cpu().numpy()


def _chunk_args(w, rows):
    """Device arguments of the chunk rows `rows` (indices into the workload's new tokens)."""
    seq = w.new_seq[rows]
    pos = w.new_pos[rows]
    # the chunk's queries are its tokens: per sequence, the rows in order
    B = w.B
    counts = np.bincount(seq, minlength=B)
    q_start = np.zeros(B + 1, dtype=np.int32)
    q_start[1:] = np.cumsum(counts)
    ctx = np.array([int(pos[seq == s].max()) + 1 if counts[s] else int(w.ctx_old[s]) for s in range(B)],
                   dtype=np.int32)
    return dict(k_new=w.new_k[rows].cuda(), v_new=w.new_v[rows].cuda(), n=len(rows),
                seq=torch.from_numpy(np.ascontiguousarray(seq, dtype=np.int32)).cuda(),
                pos=torch.from_numpy(np.ascontiguousarray(pos, dtype=np.int32)).cuda(),
                q=w.q[rows].cuda(), q_start=torch.from_numpy(q_start).cuda(),
                ctx=torch.from_numpy(ctx).cuda(), max_q=max(1, int(counts.max())), T=len(rows))


def _out(w, T):
    return torch.full((max(1, T), w.H_q, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")


def _separate(p, a):
    w = p.w
    out = _out(w, a["T"])
    N.pa_kv_append_tokens(p.desc, p.k, p.v, a["k_new"], a["v_new"], a["n"], a["seq"], a["pos"], p.tables, p.err)
    N.pa_prefill_attention(p.desc, out, a["q"], p.k, p.v, p.tables, a["q_start"], a["ctx"], a["max_q"], w.scale,
                           p.err)
    return out


def _fused(p, a):
    w = p.w
    out = _out(w, a["T"])
    N.pa_prefill_step(p.desc, out, a["q"], p.k, p.v, a["k_new"], a["v_new"], a["n"], a["seq"], a["pos"], p.tables,
                      a["q_start"], a["ctx"], a["max_q"], w.scale, p.err)
    return out


def _compare(w, chunks, window=0):
    """Run the chunks (lists of new-token rows, each a whole suffix step of its sequences) both ways."""
    sep, fus = Pools(w, window), Pools(w, window)
    for rows in chunks:
        a = _chunk_args(w, np.asarray(rows))
        o1, o2 = _separate(sep, a), _fused(fus, a)
        torch.cuda.synchronize()
        assert np.array_equal(o1.view(torch.int16).cpu().numpy(), o2.view(torch.int16).cpu().numpy())
        for x, y in zip(sep.bits(), fus.bits()):
            assert np.array_equal(x, y)
        assert int(sep.err.item()) == int(fus.err.item()) == 0


def _split_chunk(w, parts):
    """The workload's chunk of every sequence cut into `parts` consecutive steps."""
    qs = w.q_start()
    steps = [[] for _ in range(parts)]
    for s in range(w.B):
        idx = np.arange(qs[s], qs[s + 1])
        for i, piece in enumerate(np.array_split(idx, parts)):
            steps[i].extend(piece.tolist())
    return [sorted(st, key=lambda r: (w.new_seq[r], w.new_pos[r])) for st in steps]


@pytest.mark.parametrize("H_q,H_kv,D", [(32, 8, 128), (64, 8, 128), (8, 8, 128), (8, 2, 64), (12, 4, 128)])
def test_step_equals_append_then_attention(H_q, H_kv, D):
    w = make_prefill_workload(H_q=H_q, H_kv=H_kv, D=D, cached_list=[0, 17, 300, 3, 1000],
                              chunk_list=[5, 130, 33, 260, 1], seed=31)
    _compare(w, _split_chunk(w, 1))


def test_step_bench_chunk():
    w = make_prefill_workload()  # 8 sequences x 512-token chunks over cached contexts
    _compare(w, _split_chunk(w, 1))


@pytest.mark.parametrize("D", [128, 64])
def test_step_two_chunks_in_a_row(D):
    w = make_prefill_workload(H_q=16, H_kv=4, D=D, cached_list=[0, 40, 700], chunk_list=[300, 64, 257], seed=32)
    _compare(w, _split_chunk(w, 2))


@pytest.mark.parametrize("window", [16, 200])
def test_step_sliding_window(window):
    w = make_prefill_workload(H_q=32, H_kv=8, D=128, cached_list=[0, 500, 37], chunk_list=[300, 257, 129],
                              seed=33)
    _compare(w, _split_chunk(w, 1), window=window)


def test_step_host_errors_enqueue_nothing():
    w = make_prefill_workload(H_q=8, H_kv=2, D=128, cached_list=[3, 40], chunk_list=[20, 7], seed=34)
    p = Pools(w)
    before = p.bits()
    a = _chunk_args(w, np.arange(len(w.new_seq)))
    out = _out(w, a["T"])
    bad = [
        dict(scale=float("nan")),             # non-finite scale
        dict(max_q=-1),                       # negative query bound
        dict(q=None),                         # missing attention input
        dict(out_off=8),                      # misaligned output
        dict(k_new=None),                     # missing append input
    ]
    for b in bad:
        o = out.data_ptr() + b.get("out_off", 0)
        with pytest.raises(N.PaError):
            N.pa_prefill_step(p.desc, o, b.get("q", a["q"]), p.k, p.v, b.get("k_new", a["k_new"]), a["v_new"], a["n"],
                              a["seq"], a["pos"], p.tables, a["q_start"], a["ctx"], b.get("max_q", a["max_q"]),
                              b.get("scale", w.scale), p.err)
    for x, y in zip(before, p.bits()):
        assert np.array_equal(x, y), "a rejected step must not have appended"

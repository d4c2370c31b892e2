"""Pins of the oracle's sliding-window attention and block-granular window freeing.

Untitled KV-cache article at ldpk.cn/news/58971 §5.3: under sliding-window attention every
position attends only the most recent W tokens, and the cache keeps only those W positions'
K and V (O(W) memory instead of O(S)).  Reading: the query at position p sees positions
max(0, p - W + 1) .. p (its own included); blocks go back to the pool once all their positions
lie before the window of the sequence's latest query.

Pins: torch SDPA with an explicit band mask in fp64 (a library routine, not the oracle's own
formula), closed forms (W = 1 gives the query's own V; W >= ctx gives full attention), a paged
decode loop that frees blocks as it slides compared with an unpaged cache of the same tokens,
the exact block count held at every length, shared blocks surviving until every holder slid
past them, and planted mistakes.
"""

import numpy as np
import pytest
import torch

import oracle as O


def _banded_sdpa(q_all, K, V, scale, window):
    """Every position's query over the whole sequence, through torch SDPA with a band mask."""
    n, H_q, d = q_all.shape
    G = H_q // K.shape[1]
    i = torch.arange(n)[:, None]
    j = torch.arange(n)[None, :]
    allowed = (j <= i) & (j > i - window) if window > 0 else (j <= i)
    qt = torch.from_numpy(q_all).permute(1, 0, 2).unsqueeze(0)
    kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(G, dim=0).unsqueeze(0)
    vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(G, dim=0).unsqueeze(0)
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=allowed, scale=scale)
    return out[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("window", [1, 2, 15, 16, 17, 33, 200])
def test_windowed_prefill_and_decode_match_banded_sdpa(window):
    rng = np.random.default_rng(40 + window)
    ctx, H_q, H_kv, d = 70, 8, 2, 16
    q_all = rng.standard_normal((ctx, H_q, d))
    K = rng.standard_normal((ctx, H_kv, d))
    V = rng.standard_normal((ctx, H_kv, d))
    ref = _banded_sdpa(q_all, K, V, 0.25, window)
    for first in (0, 29, 69):
        got = O.prefill_attention(q_all[first:], K, V, 0.25, first, window)
        assert np.allclose(got, ref[first:], rtol=0, atol=1e-12)
    for c in (1, 16, 17, 40, 70):  # decode: the last token of a c-token sequence
        got = O.decode_attention(q_all[c - 1], K[:c], V[:c], 0.25, window)
        assert np.allclose(got, ref[c - 1], rtol=0, atol=1e-12)


def test_window_closed_forms():
    rng = np.random.default_rng(50)
    K = rng.standard_normal((37, 2, 8))
    V = rng.standard_normal((37, 2, 8))
    q = rng.standard_normal((4, 8))
    # W = 1: the query sees only its own token
    assert np.array_equal(O.decode_attention(q, K, V, 0.5, 1), V[36, [0, 0, 1, 1]])
    # W >= ctx: no token falls outside, identical to full attention
    full = O.decode_attention(q, K, V, 0.5)
    assert np.array_equal(O.decode_attention(q, K, V, 0.5, 37), full)
    assert np.array_equal(O.decode_attention(q, K, V, 0.5, 1000), full)
    assert O.window_start(37, 0) == 0 and O.window_start(37, 10) == 27 and O.window_start(5, 10) == 0


def _held_blocks(row):
    return int((np.asarray(row) >= 0).sum())


@pytest.mark.parametrize("window,num_sink", [(1, 0), (16, 0), (23, 0), (40, 4), (5, 4)])
def test_sliding_decode_loop_frees_blocks_and_matches_unpaged(window, num_sink):
    """Decode 150 tokens one at a time: append (after making the slot writable), attend with
    the window, then release the blocks the window left behind.  Every step equals windowed
    attention over an unpaged cache of the same tokens; the sequence never holds more blocks
    than the window's positions span, and released blocks are handed out again."""
    rng = np.random.default_rng(60 + window)
    H_q, H, d, steps = 4, 2, 8, 150
    pool = O.BlockPool(64)
    cache = O.PagedKVCache(64, H, d, num_seqs=1, num_sink=num_sink)
    dense = O.ContiguousKVCache(1, H, steps, d)
    row = np.full(16, -1)
    kb = O.f32_to_bf16_bits(rng.standard_normal((steps, H, d)).astype(np.float32))
    vb = O.f32_to_bf16_bits(rng.standard_normal((steps, H, d)).astype(np.float32))
    q = rng.standard_normal((steps, H_q, d))
    seen, allocs, max_held = set(), 0, 0
    for pos in range(steps):
        if pos >= num_sink:
            act = pool.prepare_append(row, pos)
            if act[0] == "alloc":
                seen.add(act[1])
                allocs += 1
        cache.append(0, row, pos, kb[pos], vb[pos])
        dense.append(0, O.bf16_bits_to_f64(kb[pos]), O.bf16_bits_to_f64(vb[pos]))
        ctx = pos + 1
        a = O.window_start(ctx, window)
        K, V = cache.gather(0, row, ctx, a)
        Kd, Vd = dense.view(0)
        assert np.array_equal(K, Kd[a:]) and np.array_equal(V, Vd[a:])
        assert np.array_equal(O.decode_attention(q[pos], K, V, 0.3),
                              O.decode_attention(q[pos], Kd, Vd, 0.3, window))
        pool.slide_window(row, ctx, window)
        # exactly the blocks that hold positions a .. ctx - 1 stay (sinks hold no paged block)
        lo_blk = max(a, num_sink) // 16 if ctx > num_sink else 0
        expect = (ctx - 1) // 16 - lo_blk + 1 if ctx > num_sink else 0
        assert _held_blocks(row) == expect
        assert expect <= -(-(window - 1) // 16) + 1
        assert pool.num_free() + _held_blocks(row) == 64
        max_held = max(max_held, _held_blocks(row))
    # O(W) memory: every logical block was allocated once, but released blocks were handed
    # out again (lowest free first), so few distinct physical blocks were ever used
    assert allocs == (steps - 1) // 16 + 1 - num_sink // 16
    assert len(seen) <= max_held + 1 < allocs


def test_shared_block_survives_until_every_holder_slides_past():
    pool = O.BlockPool(16)
    owner = np.full(8, -1)
    for p in range(48):
        pool.prepare_append(owner, p)
    other = pool.fork(owner, 3)
    assert pool.refcount[owner[0]] == 2
    # the owner slides past blocks 0 and 1: they keep the fork's reference
    assert pool.slide_window(owner, 48, 16) == 0
    assert owner[0] == -1 and owner[1] == -1 and owner[2] >= 0
    assert pool.refcount[other[0]] == 1 and pool.refcount[other[1]] == 1
    # the fork slides too: now they go back to the pool
    assert pool.slide_window(other, 48, 16) == 2
    assert other[2] == owner[2] and pool.refcount[owner[2]] == 2
    # no window or a window covering the context frees nothing
    row = pool.fork(other, 3)
    assert pool.slide_window(row, 48, 0) == 0 and pool.slide_window(row, 48, 48) == 0


def test_planted_window_mistakes_are_caught():
    rng = np.random.default_rng(70)
    q_all = rng.standard_normal((30, 4, 8))
    K = rng.standard_normal((30, 2, 8))
    V = rng.standard_normal((30, 2, 8))
    ref = _banded_sdpa(q_all, K, V, 0.5, 7)

    def one_too_many(q, K, V, scale, window):  # the window holds W + 1 tokens
        return O.decode_attention(q, K, V, scale, window + 1)

    assert np.allclose(O.decode_attention(q_all[29], K, V, 0.5, 7), ref[29], atol=1e-12)
    assert not np.allclose(one_too_many(q_all[29], K, V, 0.5, 7), ref[29], atol=1e-6)

    # releasing one block too early loses a position the window still needs
    pool = O.BlockPool(8)
    row = np.full(4, -1)
    for p in range(40):
        pool.prepare_append(row, p)
    early = row.copy()
    for lb in range((40 - 20) // 16 + 1):
        early[lb] = -1
    with pytest.raises((IndexError, ValueError)):
        O.PagedKVCache(8, 2, 8, num_seqs=1).gather(0, early, 40, O.window_start(40, 20))
    pool.slide_window(row, 40, 20)
    O.PagedKVCache(8, 2, 8, num_seqs=1).gather(0, row, 40, O.window_start(40, 20))

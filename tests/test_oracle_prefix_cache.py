"""Pins of the oracle's prefix cache (block_hashes, PrefixCache).

"大模型推理KV Cache显存优化：从PagedAttention到AI内存系统演进", prefix-cache section: a cached
block is identified by its parent's hash, its own tokens and extra inputs; only full blocks are
cached; a cache salt separates tenants; a hit needs identical tokens; low-value entries are
evicted.  §7.2: lookup by hash, and shared blocks must not be modified.

Pins: brute force (the number of blocks a request reuses equals the longest common prefix, in
whole blocks, with the cached request), isolation by salt and extra key, the chain property of
the digests, refcount conservation in the pool, LRU order with leaf-first ties, capacity, reuse
giving bit-identical K/V and attention against recomputing, and planted mistakes (a hash that
drops the parent, a cache that keeps partial blocks).
"""

import hashlib

import numpy as np
import pytest

import oracle as O


def _lcp_blocks(a, b):
    n = 0
    for x, y in zip(a, b):
        if x != y:
            break
        n += 1
    return n // 16


def test_digests_cover_full_blocks_and_form_a_chain():
    rng = np.random.default_rng(1)
    toks = rng.integers(0, 50000, 200)
    h = O.block_hashes(toks)
    assert len(h) == 200 // 16 and all(len(x) == 32 for x in h)
    for n in (0, 15, 16, 17, 100, 199):
        assert O.block_hashes(toks[:n]) == h[:n // 16]
    assert len(set(h)) == len(h)
    # one changed token in block 5 changes digests 5.. and nothing before
    t2 = toks.copy()
    t2[5 * 16 + 7] += 1
    h2 = O.block_hashes(t2)
    assert h2[:5] == h[:5] and all(a != b for a, b in zip(h2[5:], h[5:]))
    # the same block contents under different parents differ (identity covers the prefix)
    rep = np.tile(toks[:16], 3)
    hr = O.block_hashes(rep)
    assert len(set(hr)) == 3


def test_salt_and_extra_key_change_every_digest():
    toks = np.arange(64)
    base = O.block_hashes(toks)
    for kw in (dict(salt=1), dict(salt=2 ** 63), dict(extra_key=7)):
        other = O.block_hashes(toks, **kw)
        assert all(a != b for a, b in zip(base, other))
    assert O.block_hashes(toks, salt=5) == O.block_hashes(toks, salt=5)


def test_digest_is_sha256_of_the_documented_bytes():
    # the first block's digest from hashlib, with the byte layout spelled out independently
    toks = list(range(100, 116))
    root = hashlib.sha256((3).to_bytes(8, "little")).digest()
    body = b"".join(t.to_bytes(4, "little", signed=True) for t in toks) + (9).to_bytes(8, "little")
    assert O.block_hashes(toks, salt=3, extra_key=9)[0] == hashlib.sha256(root + body).digest()


def _serve(pool, cache, kv, seq, toks, salt=0, extra=0, k_bits=None, v_bits=None):
    """One request: reuse the cached prefix, write the rest of its tokens, register its full
    blocks.  Returns (table row, blocks reused)."""
    row = np.full(64, -1, dtype=np.int64)
    hashes = O.block_hashes(toks, salt, extra)
    hit = cache.match(hashes, (len(toks) - 1) // 16, row)
    for p in range(hit * 16, len(toks)):
        act = pool.prepare_append(row, p)
        assert act[0] != "copy"  # reused blocks are full: nothing writes into them
        if kv is not None:
            kv.append(seq, row, p, k_bits[p], v_bits[p])
    cache.insert(hashes, row, len(toks) // 16)
    return row, hit


def test_reuse_equals_longest_common_prefix_in_blocks():
    rng = np.random.default_rng(2)
    pool = O.BlockPool(2000)
    cache = O.PrefixCache(pool)
    system = list(rng.integers(0, 1000, 100))       # shared system prompt (6 blocks + 4 tokens)
    docs = [list(rng.integers(0, 1000, 40)) for _ in range(3)]
    served = []
    for i in range(40):
        d = docs[rng.integers(0, 3)] if rng.random() < 0.7 else []
        q = list(rng.integers(0, 1000, int(rng.integers(1, 60))))
        toks = system + d + q if rng.random() < 0.8 else q + system
        best = max([_lcp_blocks(toks, s) for s in served] + [0])
        _, hit = _serve(pool, cache, None, 0, toks)
        assert hit == min(best, (len(toks) - 1) // 16), i
        served.append(toks)


def test_salt_and_extra_key_isolate_tenants():
    pool = O.BlockPool(100)
    cache = O.PrefixCache(pool)
    toks = list(range(80))
    _serve(pool, cache, None, 0, toks, salt=11)
    assert _serve(pool, cache, None, 0, toks, salt=12)[1] == 0
    assert _serve(pool, cache, None, 0, toks, salt=11, extra=1)[1] == 0
    assert _serve(pool, cache, None, 0, toks, salt=11)[1] == (80 - 1) // 16


def test_refcounts_release_and_lru_eviction_leaf_first():
    pool = O.BlockPool(40)
    cache = O.PrefixCache(pool)
    a = list(range(48))            # 3 full blocks
    b = list(range(1000, 1033))    # 2 full blocks + 1 token
    ra, _ = _serve(pool, cache, None, 0, a)
    rb, _ = _serve(pool, cache, None, 0, b)
    assert len(cache) == 5
    for blk in ra[:3]:
        assert pool.refcount[blk] == 2  # the request and the cache
    # a second request on a's prefix shares its first two blocks (cap: one token recomputed)
    rc, hit = _serve(pool, cache, None, 0, a)
    assert hit == 2 and list(rc[:2]) == list(ra[:2]) and pool.refcount[ra[0]] == 3
    # nothing is evictable while every block is held by a request
    assert cache.evict(10) == 0
    a_blocks = [int(x) for x in ra[:3]]
    pool.release(ra, 64)
    pool.release(rc, 64)
    # b's entries are older but still held by request b; a's three entries were all refreshed by
    # the second request's registration (same time), so they go leaf first
    order = []
    while True:
        before = set(cache.blocks().tolist())
        if cache.evict(1) == 0:
            break
        order.append((before - set(cache.blocks().tolist())).pop())
    assert order == a_blocks[::-1]
    assert len(cache) == 2  # b's blocks: still held by request b
    pool.release(rb, 64)
    assert cache.evict(10) == 2 and len(cache) == 0
    assert pool.num_free() == 40


def test_capacity_evicts_idle_entries_to_make_room():
    pool = O.BlockPool(64)
    cache = O.PrefixCache(pool, capacity=4)
    r1, _ = _serve(pool, cache, None, 0, list(range(64)))  # 4 blocks: fills the cache
    pool.release(r1, 64)
    r2, _ = _serve(pool, cache, None, 0, list(range(500, 532)))  # 2 more: evicts r1's leaf side
    assert len(cache) == 4
    assert _serve(pool, cache, None, 0, list(range(64)) + [1])[1] == 2
    # with every entry held, registration stops instead of evicting
    held = O.PrefixCache(O.BlockPool(16), capacity=1)
    row = np.full(8, -1)
    for p in range(32):
        held.pool.prepare_append(row, p)
    assert held.insert(O.block_hashes(range(32)), row, 2) == 1


def test_reused_prefix_gives_identical_kv_and_attention():
    rng = np.random.default_rng(3)
    H, d, nb = 2, 8, 64
    pool = O.BlockPool(nb)
    cache = O.PrefixCache(pool)
    kv = O.PagedKVCache(nb, H, d, num_seqs=2)
    shared = list(rng.integers(0, 999, 70))
    toks = [shared + list(rng.integers(0, 999, 9)), shared + list(rng.integers(0, 999, 30))]
    # K/V of a token depend on the whole prefix in a real model; here the shared tokens get one
    # set of rows and the private ones their own, which is what reuse must preserve
    kb = O.f32_to_bf16_bits(rng.standard_normal((110, H, d)).astype(np.float32))
    vb = O.f32_to_bf16_bits(rng.standard_normal((110, H, d)).astype(np.float32))
    rows, hits = [], []
    for s in range(2):
        r, h = _serve(pool, cache, kv, s, toks[s], k_bits=kb, v_bits=vb)
        rows.append(r)
        hits.append(h)
    assert hits == [0, 4]
    dense = O.PagedKVCache(nb, H, d, num_seqs=1)
    q = rng.standard_normal((4, d))
    for p in range(len(toks[1])):
        dense.append(0, np.arange(8), p, kb[p], vb[p])
    K1, V1 = kv.gather(1, rows[1], len(toks[1]))
    K2, V2 = dense.gather(0, np.arange(8), len(toks[1]))
    assert np.array_equal(K1, K2) and np.array_equal(V1, V2)
    assert np.array_equal(O.decode_attention(q, K1, V1, 0.3), O.decode_attention(q, K2, V2, 0.3))
    assert list(rows[1][:4]) == list(rows[0][:4])


def test_planted_prefix_cache_mistakes_are_caught():
    def parentless(tokens, salt=0, extra_key=0):  # drops h_{i-1}: identical blocks collide
        t = [int(x) for x in tokens]
        return [hashlib.sha256(np.array(t[i * 16:(i + 1) * 16], dtype="<i4").tobytes()).digest()
                for i in range(len(t) // 16)]

    a = list(range(32))
    b = [7] * 16 + list(range(16, 32))  # block 1 equal, block 0 different
    assert _lcp_blocks(a, b) == 0
    pool = O.BlockPool(16)
    good = O.PrefixCache(pool)
    row = np.full(4, -1)
    for p in range(32):
        pool.prepare_append(row, p)
    good.insert(O.block_hashes(a), row, 2)
    assert good.match(O.block_hashes(b)[1:], 1, np.full(4, -1)) == 0
    assert set(parentless(a)) & set(parentless(b))  # the planted hash would reuse a's block 1
    # a cache that also registered the partial tail would hand out a block the owner still fills
    assert len(O.block_hashes(list(range(40)))) == 2

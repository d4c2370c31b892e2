"""The library's host prefix cache (pa_pc_*) against the oracle's, on the CPU.

The digests must equal the oracle's SHA-256 chain (hashlib) byte for byte, including negative
token ids, large salts and extra keys; a random serving simulation (shared system prompts,
documents, tenants with different salts, requests finishing, capacity and explicit eviction)
must make the same hits, tables, refcounts and evictions in both; concurrent callers must leave
the cache and the pool consistent.
"""

import threading

import numpy as np
import pytest

import oracle as O
from paged_kv_cache_table_gb300 import build as B
from paged_kv_cache_table_gb300 import native as N


@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()


@pytest.mark.parametrize("n,salt,extra", [(0, 0, 0), (15, 0, 0), (16, 0, 0), (17, 3, 0), (200, 2 ** 64 - 1, 5),
                                          (1000, 12345678901234, 2 ** 63)])
def test_digests_match_the_oracle_chain(n, salt, extra):
    rng = np.random.default_rng(n)
    toks = rng.integers(-2 ** 31, 2 ** 31, n, dtype=np.int64).astype(np.int32)
    got = N.block_hashes(toks, salt, extra)
    ref = O.block_hashes(toks.tolist(), salt, extra)
    assert got.shape == (n // 16, 32)
    assert [bytes(r) for r in got] == ref


def _dig(hashes):
    return np.frombuffer(b"".join(hashes), dtype=np.uint8).reshape(len(hashes), 32) if hashes else \
        np.zeros((0, 32), dtype=np.uint8)


@pytest.mark.parametrize("capacity", [0, 30])
def test_serving_simulation_matches_oracle(capacity):
    rng = np.random.default_rng(7 + capacity)
    NB, M = 600, 40
    bm, pool = N.BlockManager(NB), O.BlockPool(NB)
    pc, opc = N.PrefixCache(bm, capacity), O.PrefixCache(pool, capacity)
    systems = [list(rng.integers(0, 1000, int(rng.integers(20, 120)))) for _ in range(3)]
    docs = [list(rng.integers(0, 1000, 48)) for _ in range(4)]
    live = []  # (row, orow)
    hits_total = 0
    for step in range(300):
        toks = list(systems[rng.integers(0, 3)])
        if rng.random() < 0.6:
            toks += docs[rng.integers(0, 4)]
        toks += list(rng.integers(0, 1000, int(rng.integers(1, 50))))
        salt = int(rng.integers(0, 2))
        hashes = O.block_hashes(toks, salt)
        digests = N.block_hashes(np.array(toks, dtype=np.int32), salt)
        cap = (len(toks) - 1) // 16
        row = np.full(M, -1, dtype=np.int32)
        orow = np.full(M, -1, dtype=np.int64)
        hit = pc.match(digests, cap, row)
        ohit = opc.match(hashes, cap, orow)
        assert hit == ohit
        hits_total += hit
        for p in range(hit * 16, len(toks)):
            bm.prepare_step(row[None, :], np.array([p], dtype=np.int32))
            assert pool.prepare_append(orow, p)[0] != "copy"
        assert np.array_equal(row, orow)
        assert pc.insert(digests, row, len(toks) // 16) == opc.insert(hashes, orow, len(toks) // 16)
        live.append((row, orow))
        # requests finish in random order
        while live and rng.random() < 0.45:
            r, o = live.pop(int(rng.integers(0, len(live))))
            assert bm.release(r, M) == pool.release(o, M)
        if step % 25 == 24:
            k = int(rng.integers(1, 20))
            assert pc.evict(k) == opc.evict(k)
        assert len(pc) == len(opc)
        assert bm.num_free() == pool.num_free()
    assert hits_total > 100
    for b in range(NB):
        assert bm.refcount(b) == pool.refcount[b]
    for r, o in live:
        bm.release(r, M)
        pool.release(o, M)
    assert pc.clear() == opc.clear()
    assert bm.num_free() == NB and pool.num_free() == NB


def test_bad_arguments_and_foreign_blocks():
    bm = N.BlockManager(8)
    pc = N.PrefixCache(bm)
    d = N.block_hashes(np.arange(32, dtype=np.int32))
    with pytest.raises(N.PaError):
        pc.insert(d, np.array([5, 6], dtype=np.int32), 2)  # never allocated
    row = np.full(4, -1, dtype=np.int32)
    assert pc.match(d, 2, row) == 0 and len(pc) == 0
    assert N.lib().pa_pc_create(None, 0) is None
    assert N.lib().pa_pc_evict(None, 1) == -1 and N.lib().pa_pc_size(None) == -1


def test_concurrent_callers_keep_cache_and_pool_consistent():
    NB, M = 4000, 16
    bm = N.BlockManager(NB)
    pc = N.PrefixCache(bm, 200)
    prefix = np.arange(160, dtype=np.int32)
    errors = []

    def worker(seed):
        rng = np.random.default_rng(seed)
        try:
            for _ in range(150):
                toks = np.concatenate([prefix[:int(rng.integers(16, 160))],
                                       rng.integers(0, 50, int(rng.integers(1, 40))).astype(np.int32)])
                d = N.block_hashes(toks)
                row = np.full(M, -1, dtype=np.int32)
                hit = pc.match(d, (len(toks) - 1) // 16, row)
                for p in range(hit * 16, len(toks)):
                    bm.prepare_step(row[None, :], np.array([p], dtype=np.int32))
                pc.insert(d, row, len(toks) // 16)
                bm.release(row, M)
                if rng.random() < 0.2:
                    pc.evict(3)
        except Exception as e:  # pragma: no cover - reported below
            errors.append(e)

    ts = [threading.Thread(target=worker, args=(s,)) for s in range(6)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errors
    # every held block is a cache entry holding exactly its own reference
    assert len(pc) <= 200
    held = [b for b in range(NB) if bm.refcount(b) > 0]
    assert len(held) == len(pc) and all(bm.refcount(b) == 1 for b in held)
    assert pc.clear() == len(held) and bm.num_free() == NB

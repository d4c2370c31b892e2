"""Prefix cache end to end on the GPU: requests reuse cached prefix blocks, prefill only their
own suffix over the shared blocks, register their full blocks and decode, all through the C ABI,
beside the oracle doing the same with its own pool and cache.

Hits, tables and refcounts must agree exactly; prefill and decode outputs within max-abs 2e-2 /
mean-abs 2e-3 of the fp64 oracle; every cached block's bytes must be unchanged at the end (shared
blocks are never written).  A token's K/V rows here are a fixed function of the block digest it
belongs to (full blocks) or of the request (tail), which is what reuse has to preserve.
"""

import hashlib

import numpy as np
import pytest
import torch

import oracle as O
from paged_kv_cache_table_gb300 import native as N

from harness import BF16_NAN, assert_attention_close, to_f64

pytestmark = pytest.mark.gpu

H_q, H_kv, D, NB, M = 16, 4, 128, 400, 48
SCALE = 1.0 / np.sqrt(D)


def _rows(seed_bytes, n):
    g = torch.Generator().manual_seed(int.from_bytes(hashlib.sha256(seed_bytes).digest()[:8], "little") >> 1)
    k = torch.randn((n, H_kv, D), generator=g).to(torch.bfloat16)
    v = torch.randn((n, H_kv, D), generator=g).to(torch.bfloat16)
    return k, v


def _kv_of_request(toks, digests, rid):
    """K/V rows of every position: full blocks from their digest, the tail from the request."""
    ks, vs = [], []
    for i in range(len(digests)):
        k, v = _rows(bytes(digests[i]), 16)
        ks.append(k)
        vs.append(v)
    tail = len(toks) - 16 * len(digests)
    if tail:
        k, v = _rows(b"tail" + rid.to_bytes(4, "little"), tail)
        ks.append(k)
        vs.append(v)
    return torch.cat(ks), torch.cat(vs)


def _bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def test_requests_reuse_cached_prefixes_through_prefill_and_decode():
    rng = np.random.default_rng(5)
    dev = "cuda"
    kc = torch.full((NB * 16, H_kv, D), BF16_NAN, dtype=torch.int16, device=dev).view(torch.bfloat16)
    vc = torch.full((NB * 16, H_kv, D), BF16_NAN, dtype=torch.int16, device=dev).view(torch.bfloat16)
    desc = N.make_desc(1, H_q, H_kv, D, NB, M)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    bm, pool = N.BlockManager(NB), O.BlockPool(NB)
    pc, opc = N.PrefixCache(bm), O.PrefixCache(pool)
    system = list(rng.integers(0, 500, 150))
    docs = [list(rng.integers(0, 500, 64)) for _ in range(2)]
    cached_bytes = {}  # block -> (K bits, V bits) when registered
    hits = []
    live = []
    for rid in range(8):
        toks = system + (docs[rid % 2] if rid % 3 else []) + list(rng.integers(0, 500, int(rng.integers(5, 40))))
        n = len(toks)
        digests = N.block_hashes(np.array(toks, dtype=np.int32))
        hashes = O.block_hashes(toks)
        assert [bytes(d) for d in digests] == hashes
        row = np.full(M, -1, dtype=np.int32)
        orow = np.full(M, -1, dtype=np.int64)
        hit = pc.match(digests, (n - 1) // 16, row)
        assert hit == opc.match(hashes, (n - 1) // 16, orow)
        hits.append(hit)
        first = hit * 16
        for p in range(first, n):
            bm.prepare_step(row[None, :], np.array([p], dtype=np.int32))
            assert pool.prepare_append(orow, p)[0] != "copy"
        assert np.array_equal(row, orow)
        K, V = _kv_of_request(toks, digests, rid)
        tab = torch.from_numpy(row[None, :].copy()).to(dev)
        m = n - first
        N.pa_kv_append_tokens(desc, kc, vc, K[first:].to(dev), V[first:].to(dev), m,
                              torch.zeros(m, dtype=torch.int32, device=dev),
                              torch.arange(first, n, dtype=torch.int32, device=dev), tab, err)
        # prefill of the suffix over the shared blocks
        q = torch.randn((m, H_q, D), generator=torch.Generator().manual_seed(rid)).to(torch.bfloat16)
        out = torch.empty((m, H_q, D), dtype=torch.bfloat16, device=dev)
        N.pa_prefill_attention(desc, out, q.to(dev), kc, vc, tab, torch.tensor([0, m], dtype=torch.int32, device=dev),
                               torch.tensor([n], dtype=torch.int32, device=dev), m, SCALE, err)
        torch.cuda.synchronize()
        Kf = O.bf16_bits_to_f64(_bits(K))
        Vf = O.bf16_bits_to_f64(_bits(V))
        ref = O.prefill_attention(O.bf16_bits_to_f64(_bits(q)), Kf, Vf, SCALE, first)
        assert_attention_close(to_f64(out), ref, f"request {rid} prefill")
        # register its full blocks, then one decode step
        pc.insert(digests, row, n // 16)
        opc.insert(hashes, orow, n // 16)
        for i in range(n // 16):
            b = int(row[i])
            if b not in cached_bytes:
                cached_bytes[b] = (_bits(K[16 * i:16 * i + 16]).copy(), _bits(V[16 * i:16 * i + 16]).copy())
        bm.prepare_step(row[None, :], np.array([n], dtype=np.int32))
        pool.prepare_append(orow, n)
        tab.copy_(torch.from_numpy(row[None, :].copy()))
        kn, vn = _rows(b"dec" + rid.to_bytes(4, "little"), 1)
        N.pa_kv_append(desc, kc, vc, kn.to(dev), vn.to(dev), tab, torch.tensor([n], dtype=torch.int32, device=dev), err)
        qd = torch.randn((1, H_q, D), generator=torch.Generator().manual_seed(100 + rid)).to(torch.bfloat16)
        od = torch.empty((1, H_q, D), dtype=torch.bfloat16, device=dev)
        nbytes = N.pa_decode_workspace_size(desc, n + 1, 0)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        N.pa_decode_attention(desc, od, qd.to(dev), kc, vc, tab, torch.tensor([n + 1], dtype=torch.int32, device=dev),
                              n + 1, SCALE, 0, ws, nbytes, err)
        torch.cuda.synchronize()
        Kd = np.concatenate([Kf, O.bf16_bits_to_f64(_bits(kn))])
        Vd = np.concatenate([Vf, O.bf16_bits_to_f64(_bits(vn))])
        refd = O.decode_attention(O.bf16_bits_to_f64(_bits(qd))[0], Kd, Vd, SCALE)
        assert_attention_close(to_f64(od)[0], refd, f"request {rid} decode")
        live.append((row, orow))
        if rid % 2 == 1:  # some requests finish; their cached blocks stay with the cache
            r, o = live.pop(0)
            assert bm.release(r, M) == pool.release(o, M)
        assert bm.num_free() == pool.num_free()
    assert int(err.item()) == 0
    assert sum(h > 0 for h in hits) >= 5 and max(hits) >= 9
    # cached blocks were never written after registration
    kb = kc.view(torch.int16).cpu().numpy().view(np.uint16)
    vb = vc.view(torch.int16).cpu().numpy().view(np.uint16)
    for b, (k0, v0) in cached_bytes.items():
        assert np.array_equal(kb[16 * b:16 * b + 16], k0) and np.array_equal(vb[16 * b:16 * b + 16], v0)
    for b in range(NB):
        assert bm.refcount(b) == pool.refcount[b]

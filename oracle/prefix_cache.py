"""Oracle of the prefix cache: full-block hash chain, lookup, registration and eviction.

TEST INFRASTRUCTURE, NOT PRODUCT CODE (see the package docstring).

"大模型推理KV Cache显存优化：从PagedAttention到AI内存系统演进" (AI内存系统), the section on prefix
caching: PagedAttention decides where a KV block lives, the prefix cache decides whether a block
was computed before.  Requests that start with the same system prompt, few-shot examples or
document reuse the cached prefix blocks and compute only what follows.  A cached block is
identified by its parent block's hash, its own tokens and extra inputs (LoRA, multimodal), only
full blocks are cached, and a cache salt keeps tenants from reusing (and probing) each other's
entries.  A hit needs identical tokens; hot prefixes hold capacity and low-value entries are
evicted in the end.  AI内存系统 §7.2: matching must go through a hash or a prefix tree, never a
linear scan of the prefix library, and shared blocks must never be modified (copy-on-write).

Readings (the page fixes none of these details):
  * digest = SHA-256 (FIPS 180-4), taken here from Python's hashlib;
    h_root = SHA-256(salt as 8 bytes little-endian);
    h_i = SHA-256(h_{i-1} || the 16 token ids of block i as 4-byte little-endian int32 ||
    extra_key as 8 bytes little-endian), so a block's identity covers its whole prefix;
  * the lookup returns the longest run of leading blocks whose digests are cached, capped by the
    caller (an engine caps it at (n_tokens - 1) // 16 so that at least one prompt token is still
    computed to produce the next-token logits);
  * the cache holds one reference of its own on every registered block, so a block outlives the
    request that wrote it; a digest already cached keeps its first block (later duplicates stay
    private to their request);
  * eviction frees least-recently-used entries whose block no sequence holds (refcount 1, the
    cache's own); among entries used at the same time the deeper block goes first, so chains
    shrink from the leaf; every match and registration refreshes the entries it touches.
"""

from __future__ import annotations

import hashlib
import struct

import numpy as np

from .paged_kv import BLOCK_SIZE, BlockPool

__all__ = ["block_hashes", "PrefixCache"]


def block_hashes(tokens, salt: int = 0, extra_key: int = 0, block_size: int = BLOCK_SIZE):
    """Digests (32-byte strings) of every full block of a token sequence (partial tail: none)."""
    toks = [int(t) for t in tokens]
    h = hashlib.sha256(struct.pack("<Q", salt & 0xFFFFFFFFFFFFFFFF)).digest()
    out = []
    for i in range(len(toks) // block_size):
        blk = toks[i * block_size:(i + 1) * block_size]
        h = hashlib.sha256(h + struct.pack(f"<{block_size}i", *blk) +
                           struct.pack("<Q", extra_key & 0xFFFFFFFFFFFFFFFF)).digest()
        out.append(h)
    return out


class PrefixCache:
    """digest -> physical block, with the cache's own reference on each block of the pool."""

    def __init__(self, pool: BlockPool, capacity: int = 0):
        self.pool = pool
        self.capacity = int(capacity)  # 0 = bounded only by the pool
        self.entries = {}              # digest -> [block, last_use, depth]
        self.clock = 0

    def __len__(self):
        return len(self.entries)

    def match(self, hashes, max_blocks: int, table_row) -> int:
        """Write the physical blocks of the longest cached leading run (at most max_blocks) into
        table_row[0:n], take one reference on each for the request, and return n."""
        self.clock += 1
        n = 0
        for h in hashes[:max(0, max_blocks)]:
            e = self.entries.get(h)
            if e is None:
                break
            e[1] = self.clock
            table_row[n] = e[0]
            self.pool.incref(e[0])
            n += 1
        return n

    def insert(self, hashes, table_row, n_blocks: int) -> int:
        """Register blocks 0..n_blocks-1 of a request (their K/V written) under their digests.
        New entries take the cache's reference; digests already cached are refreshed only.
        Returns the number of new entries (capacity full: the LRU evictable entry makes room,
        and registration stops when none can)."""
        self.clock += 1
        added = 0
        for i in range(min(n_blocks, len(hashes))):
            h = hashes[i]
            e = self.entries.get(h)
            if e is not None:
                e[1] = self.clock
                continue
            if self.capacity and len(self.entries) >= self.capacity and self.evict(1) == 0:
                break
            blk = int(table_row[i])
            if self.pool.incref(blk) < 0:
                raise ValueError(f"block {blk} is not allocated")
            self.entries[h] = [blk, self.clock, i]
            added += 1
        return added

    def evict(self, n: int) -> int:
        """Free up to n LRU entries whose block only the cache holds; returns how many."""
        idle = [(e[1], -e[2], h) for h, e in self.entries.items() if self.pool.refcount[e[0]] == 1]
        idle.sort()
        freed = 0
        for _, _, h in idle[:max(0, n)]:
            blk = self.entries.pop(h)[0]
            self.pool.decref(blk)
            freed += 1
        return freed

    def clear(self) -> int:
        """Drop every entry's reference (blocks still held by sequences stay allocated)."""
        n = len(self.entries)
        for blk, _, _ in self.entries.values():
            self.pool.decref(blk)
        self.entries.clear()
        return n

    def blocks(self):
        return np.array(sorted(e[0] for e in self.entries.values()), dtype=np.int64)

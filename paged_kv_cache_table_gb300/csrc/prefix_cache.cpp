// Prefix cache: which physical blocks already hold the K/V of a token prefix.
//
// "大模型推理KV Cache显存优化：从PagedAttention到AI内存系统演进", prefix-cache section: PagedAttention
// decides where a block lives, the prefix cache whether it was computed before.  A cached block is
// identified by its parent block's hash, its own tokens and extra inputs (LoRA, multimodal); only
// full blocks are cached; a cache salt keeps tenants apart; a hit needs identical tokens; low-value
// entries are evicted.  Same page §7.2: matching goes through a hash, never a linear scan of the
// prefix library, and shared blocks are never modified (the pool's copy-on-write handles writes).
//
// Identity of block i of a request: h_i = SHA-256(h_{i-1} || its 16 token ids as little-endian
// int32 || extra_key as little-endian uint64), h_{-1} = SHA-256(salt as little-endian uint64).
// SHA-256 follows FIPS 180-4; its round constants are derived at first use from their definition
// (the fractional parts of the cube and square roots of the first primes) with integer roots.
//
// The cache takes one reference of its own on every block it registers (so a block outlives its
// request), keeps digest -> block in a hash map, and orders entries by (last use, depth) so that
// eviction takes the least recently used block that no sequence holds, leaf first.

#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <tuple>
#include <unordered_map>

#include "block_pool.h"
#include "pa.h"

namespace {

// ---------------------------------------------------------------------------------------------
// SHA-256 (FIPS 180-4)
// ---------------------------------------------------------------------------------------------
struct Sha256Consts {
  uint32_t k[64];
  uint32_t h0[8];
};

// floor(x^(1/n)) for n = 2, 3 by bisection on 128-bit integers (exact).
uint64_t int_root(unsigned __int128 x, int n) {
  uint64_t lo = 0, hi = uint64_t(1) << 42;  // every root taken here is below 2^36
  while (lo < hi) {
    const uint64_t mid = lo + (hi - lo + 1) / 2;
    unsigned __int128 p = mid;
    for (int i = 1; i < n; ++i) p *= mid;
    if (p <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

const Sha256Consts& sha256_consts() {
  static Sha256Consts c;
  static std::once_flag once;
  std::call_once(once, [] {
    int primes[64], n = 0;
    for (int v = 2; n < 64; ++v) {
      bool prime = true;
      for (int i = 0; i < n && primes[i] * primes[i] <= v; ++i)
        if (v % primes[i] == 0) prime = false;
      if (prime) primes[n++] = v;
    }
    // first 32 bits of the fractional part of p^(1/3): floor(p^(1/3) * 2^32) mod 2^32
    for (int i = 0; i < 64; ++i)
      c.k[i] = static_cast<uint32_t>(int_root(static_cast<unsigned __int128>(primes[i]) << 96, 3));
    for (int i = 0; i < 8; ++i)
      c.h0[i] = static_cast<uint32_t>(int_root(static_cast<unsigned __int128>(primes[i]) << 64, 2));
  });
  return c;
}

inline uint32_t rotr(uint32_t x, int n) { return (x >> n) | (x << (32 - n)); }

// One round of FIPS 180-4 §6.2.2 step 3 with the working variables renamed instead of shifted:
// the caller rotates the argument order, so only d and h change (d += T1, h = T1 + T2).
inline void sha256_round(uint32_t a, uint32_t b, uint32_t c, uint32_t& d, uint32_t e, uint32_t f, uint32_t g,
                         uint32_t& h, uint32_t kw) {
  const uint32_t t1 = h + (rotr(e, 6) ^ rotr(e, 11) ^ rotr(e, 25)) + ((e & f) ^ (~e & g)) + kw;
  const uint32_t t2 = (rotr(a, 2) ^ rotr(a, 13) ^ rotr(a, 22)) + ((a & b) ^ (a & c) ^ (b & c));
  d += t1;
  h = t1 + t2;
}

void sha256_block(uint32_t st[8], const uint8_t* blk, const uint32_t* k) {
  uint32_t w[64];
  for (int t = 0; t < 16; ++t)
    w[t] = (uint32_t(blk[4 * t]) << 24) | (uint32_t(blk[4 * t + 1]) << 16) | (uint32_t(blk[4 * t + 2]) << 8) |
           uint32_t(blk[4 * t + 3]);
  for (int t = 16; t < 64; ++t) {
    const uint32_t s0 = rotr(w[t - 15], 7) ^ rotr(w[t - 15], 18) ^ (w[t - 15] >> 3);
    const uint32_t s1 = rotr(w[t - 2], 17) ^ rotr(w[t - 2], 19) ^ (w[t - 2] >> 10);
    w[t] = s1 + w[t - 7] + s0 + w[t - 16];
  }
  uint32_t a = st[0], b = st[1], c = st[2], d = st[3], e = st[4], f = st[5], g = st[6], h = st[7];
  for (int t = 0; t < 64; t += 8) {  // eight rounds bring the names back to their places
    sha256_round(a, b, c, d, e, f, g, h, k[t] + w[t]);
    sha256_round(h, a, b, c, d, e, f, g, k[t + 1] + w[t + 1]);
    sha256_round(g, h, a, b, c, d, e, f, k[t + 2] + w[t + 2]);
    sha256_round(f, g, h, a, b, c, d, e, k[t + 3] + w[t + 3]);
    sha256_round(e, f, g, h, a, b, c, d, k[t + 4] + w[t + 4]);
    sha256_round(d, e, f, g, h, a, b, c, k[t + 5] + w[t + 5]);
    sha256_round(c, d, e, f, g, h, a, b, k[t + 6] + w[t + 6]);
    sha256_round(b, c, d, e, f, g, h, a, k[t + 7] + w[t + 7]);
  }
  st[0] += a; st[1] += b; st[2] += c; st[3] += d;
  st[4] += e; st[5] += f; st[6] += g; st[7] += h;
}

// Digest of a message of at most 119 bytes (two 64-byte blocks after padding).
void sha256_short(const uint8_t* msg, size_t len, uint8_t out[32]) {
  const Sha256Consts& c = sha256_consts();
  uint8_t buf[128];
  std::memset(buf, 0, sizeof(buf));
  std::memcpy(buf, msg, len);
  buf[len] = 0x80;
  const size_t total = len + 1 + 8 <= 64 ? 64 : 128;
  const uint64_t bits = static_cast<uint64_t>(len) * 8;
  for (int i = 0; i < 8; ++i) buf[total - 1 - i] = static_cast<uint8_t>(bits >> (8 * i));
  uint32_t st[8];
  std::memcpy(st, c.h0, sizeof(st));
  for (size_t off = 0; off < total; off += 64) sha256_block(st, buf + off, c.k);
  for (int i = 0; i < 8; ++i)
    for (int j = 0; j < 4; ++j) out[4 * i + j] = static_cast<uint8_t>(st[i] >> (24 - 8 * j));
}

void put_le(uint8_t* dst, uint64_t v, int bytes) {
  for (int i = 0; i < bytes; ++i) dst[i] = static_cast<uint8_t>(v >> (8 * i));
}

// ---------------------------------------------------------------------------------------------
// The cache
// ---------------------------------------------------------------------------------------------
struct Digest {
  uint8_t b[PA_PC_DIGEST_BYTES];
  bool operator==(const Digest& o) const { return std::memcmp(b, o.b, sizeof(b)) == 0; }
};

struct DigestHash {
  size_t operator()(const Digest& d) const {
    uint64_t x;
    std::memcpy(&x, d.b, sizeof(x));  // a SHA-256 prefix is already uniformly spread
    return static_cast<size_t>(x);
  }
};

// (last use, -depth, touch number): oldest first, deeper first; the touch number keeps keys
// unique even when a caller passes digests that are not one chain
using LruKey = std::tuple<uint64_t, int, uint64_t>;

struct Entry {
  int block;
  int depth;
  LruKey key;
};

}  // namespace

struct pa_pc {
  pa_bm* bm = nullptr;
  int capacity = 0;
  uint64_t clock = 0;
  uint64_t touches = 0;
  std::unordered_map<Digest, Entry, DigestHash> map;
  std::map<LruKey, Digest> lru;
  mutable std::mutex mu;

  LruKey next_key(int depth) { return LruKey{clock, -depth, ++touches}; }

  void touch(const Digest& d, Entry& e) {
    lru.erase(e.key);
    e.key = next_key(e.depth);
    lru.emplace(e.key, d);
  }

  // caller holds mu; takes the pool's lock itself
  int evict_locked(int n) {
    int freed = 0;
    std::lock_guard<std::mutex> g(bm->mu);
    for (auto it = lru.begin(); it != lru.end() && freed < n;) {
      auto e = map.find(it->second);
      const int b = e->second.block;
      if (bm->refcount[b] != 1) {  // some sequence still holds it
        ++it;
        continue;
      }
      bm->refcount[b] = 0;
      bm->release_locked(b);
      map.erase(e);
      it = lru.erase(it);
      ++freed;
    }
    return freed;
  }
};

extern "C" {

int pa_pc_block_hashes(const int32_t* tokens, int n_tokens, uint64_t salt, uint64_t extra_key,
                       uint8_t* digests) {
  if (n_tokens < 0 || (n_tokens > 0 && !tokens)) return -1;
  const int n_blocks = n_tokens / PA_BLOCK_SIZE;
  if (n_blocks > 0 && !digests) return -1;
  uint8_t prev[PA_PC_DIGEST_BYTES];
  uint8_t salt_le[8];
  put_le(salt_le, salt, 8);
  sha256_short(salt_le, 8, prev);
  uint8_t msg[PA_PC_DIGEST_BYTES + 4 * PA_BLOCK_SIZE + 8];
  for (int i = 0; i < n_blocks; ++i) {
    std::memcpy(msg, prev, PA_PC_DIGEST_BYTES);
    for (int t = 0; t < PA_BLOCK_SIZE; ++t)
      put_le(msg + PA_PC_DIGEST_BYTES + 4 * t, static_cast<uint32_t>(tokens[i * PA_BLOCK_SIZE + t]), 4);
    put_le(msg + PA_PC_DIGEST_BYTES + 4 * PA_BLOCK_SIZE, extra_key, 8);
    sha256_short(msg, sizeof(msg), digests + static_cast<size_t>(i) * PA_PC_DIGEST_BYTES);
    std::memcpy(prev, digests + static_cast<size_t>(i) * PA_PC_DIGEST_BYTES, PA_PC_DIGEST_BYTES);
  }
  return n_blocks;
}

pa_pc* pa_pc_create(pa_bm* bm, int capacity) {
  if (!bm || capacity < 0) return nullptr;
  pa_pc* pc = new (std::nothrow) pa_pc();
  if (!pc) return nullptr;
  pc->bm = bm;
  pc->capacity = capacity;
  return pc;
}

int pa_pc_clear(pa_pc* pc) {
  if (!pc) return -1;
  std::lock_guard<std::mutex> g(pc->mu);
  std::lock_guard<std::mutex> gb(pc->bm->mu);
  const int n = static_cast<int>(pc->map.size());
  for (auto& kv : pc->map) {
    const int b = kv.second.block;
    if (pc->bm->valid_allocated(b) && --pc->bm->refcount[b] == 0) pc->bm->release_locked(b);
  }
  pc->map.clear();
  pc->lru.clear();
  return n;
}

void pa_pc_destroy(pa_pc* pc) {
  if (!pc) return;
  pa_pc_clear(pc);
  delete pc;
}

int pa_pc_size(const pa_pc* pc) {
  if (!pc) return -1;
  std::lock_guard<std::mutex> g(pc->mu);
  return static_cast<int>(pc->map.size());
}

int pa_pc_match(pa_pc* pc, const uint8_t* digests, int n_blocks, int32_t* table_row) {
  if (!pc || n_blocks < 0 || (n_blocks > 0 && (!digests || !table_row))) return -1;
  std::lock_guard<std::mutex> g(pc->mu);
  ++pc->clock;
  std::lock_guard<std::mutex> gb(pc->bm->mu);
  int n = 0;
  for (; n < n_blocks; ++n) {
    Digest d;
    std::memcpy(d.b, digests + static_cast<size_t>(n) * PA_PC_DIGEST_BYTES, PA_PC_DIGEST_BYTES);
    auto it = pc->map.find(d);
    if (it == pc->map.end()) break;
    pc->touch(it->first, it->second);
    table_row[n] = it->second.block;
    ++pc->bm->refcount[it->second.block];
  }
  return n;
}

int pa_pc_insert(pa_pc* pc, const uint8_t* digests, const int32_t* table_row, int n_blocks) {
  if (!pc || n_blocks < 0 || (n_blocks > 0 && (!digests || !table_row))) return -1;
  std::lock_guard<std::mutex> g(pc->mu);
  ++pc->clock;
  int added = 0;
  for (int i = 0; i < n_blocks; ++i) {
    Digest d;
    std::memcpy(d.b, digests + static_cast<size_t>(i) * PA_PC_DIGEST_BYTES, PA_PC_DIGEST_BYTES);
    auto it = pc->map.find(d);
    if (it != pc->map.end()) {
      pc->touch(it->first, it->second);
      continue;
    }
    if (pc->capacity > 0 && static_cast<int>(pc->map.size()) >= pc->capacity && pc->evict_locked(1) == 0)
      break;
    const int b = table_row[i];
    {
      std::lock_guard<std::mutex> gb(pc->bm->mu);
      if (!pc->bm->valid_allocated(b)) return -1;  // entries registered so far stay
      ++pc->bm->refcount[b];
    }
    Entry e{b, i, pc->next_key(i)};
    auto ins = pc->map.emplace(d, e);
    pc->lru.emplace(e.key, ins.first->first);
    ++added;
  }
  return added;
}

int pa_pc_evict(pa_pc* pc, int n) {
  if (!pc || n < 0) return -1;
  std::lock_guard<std::mutex> g(pc->mu);
  return pc->evict_locked(n);
}

}  // extern "C"

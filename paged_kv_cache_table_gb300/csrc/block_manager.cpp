// Host block manager: physical block pool, free list, reference counts and the
// copy-on-write decision of a decode step.
//
// "KV Cache 的显存账本：PagedAttention 与连续批处理" §四: the cache is cut into equal
// blocks, any free block can serve any sequence, and requests with a common prefix point at
// the same physical blocks until they diverge.  "大模型推理KV Cache显存优化：从PagedAttention
// 到AI内存系统演进" §3.2: each block carries a reference count that must change atomically,
// a block is recycled only when its count reaches zero, and a sequence that writes into a
// shared block copies it first; §2.3: blocks go back to the pool on every exit path.
//
// Untitled KV-cache article at ldpk.cn/news/58971 §5.3: under a sliding window only the most
// recent W positions' K and V are kept; pa_bm_slide_window hands back, block by block, what
// falls behind the window.
//
// One mutex guards the pool, so concurrent callers never corrupt a count.  The free list
// is a min-heap: allocation returns the lowest-numbered free block (a deterministic policy
// that makes table contents reproducible).

#include <algorithm>
#include <new>

#include "block_pool.h"
#include "pa.h"

extern "C" {

pa_bm* pa_bm_create(int num_blocks, int block_size) {
  if (num_blocks <= 0 || block_size <= 0) return nullptr;
  pa_bm* bm = new (std::nothrow) pa_bm();
  if (!bm) return nullptr;
  try {
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->refcount.assign(num_blocks, 0);
    bm->is_free.assign(num_blocks, 1);
    bm->free_heap.resize(num_blocks);
    bm->nfree = num_blocks;
    for (int i = 0; i < num_blocks; ++i) bm->free_heap[i] = i;  // sorted == valid min-heap
  } catch (...) {
    delete bm;
    return nullptr;
  }
  return bm;
}

void pa_bm_destroy(pa_bm* bm) { delete bm; }

int pa_bm_alloc(pa_bm* bm) {
  if (!bm) return -1;
  std::lock_guard<std::mutex> g(bm->mu);
  return bm->alloc_locked();
}

int pa_bm_claim(pa_bm* bm, int blk) {
  if (!bm) return -1;
  std::lock_guard<std::mutex> g(bm->mu);
  if (blk < 0 || blk >= bm->num_blocks || !bm->is_free[blk]) return -1;
  bm->is_free[blk] = 0;  // its heap entry becomes stale and is skipped by alloc
  bm->refcount[blk] = 1;
  --bm->nfree;
  return 0;
}

int pa_bm_incref(pa_bm* bm, int blk) {
  if (!bm) return -1;
  std::lock_guard<std::mutex> g(bm->mu);
  if (!bm->valid_allocated(blk)) return -1;
  return ++bm->refcount[blk];
}

int pa_bm_decref(pa_bm* bm, int blk) {
  if (!bm) return -1;
  std::lock_guard<std::mutex> g(bm->mu);
  if (!bm->valid_allocated(blk)) return -1;
  int r = --bm->refcount[blk];
  if (r == 0) bm->release_locked(blk);
  return r;
}

int pa_bm_refcount(const pa_bm* bm, int blk) {
  if (!bm || blk < 0 || blk >= bm->num_blocks) return -1;
  std::lock_guard<std::mutex> g(bm->mu);
  return bm->refcount[blk];
}

int pa_bm_num_free(const pa_bm* bm) {
  if (!bm) return -1;
  std::lock_guard<std::mutex> g(bm->mu);
  return bm->nfree;
}

pa_status pa_bm_fork(pa_bm* bm, const int32_t* src_row, int32_t* dst_row, int n_blocks) {
  if (!bm || (n_blocks > 0 && (!src_row || !dst_row)) || n_blocks < 0) return PA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(bm->mu);
  for (int i = 0; i < n_blocks; ++i)
    if (!bm->valid_allocated(src_row[i])) return PA_ERR_INVALID_ARG;  // nothing changed yet
  for (int i = 0; i < n_blocks; ++i) {
    dst_row[i] = src_row[i];
    ++bm->refcount[src_row[i]];
  }
  return PA_OK;
}

int pa_bm_release(pa_bm* bm, int32_t* row, int n_blocks) {
  if (!bm || n_blocks < 0 || (n_blocks > 0 && !row)) return -1;
  std::lock_guard<std::mutex> g(bm->mu);
  int freed = 0;
  for (int i = 0; i < n_blocks; ++i) {
    int b = row[i];
    if (b < 0) continue;
    if (bm->valid_allocated(b)) {
      if (--bm->refcount[b] == 0) {
        bm->release_locked(b);
        ++freed;
      }
    }
    row[i] = -1;
  }
  return freed;
}

pa_status pa_bm_prepare_step(pa_bm* bm, int32_t* block_tables, int num_seqs,
                             int max_blocks_per_seq, const int32_t* positions,
                             int32_t* cow_pairs, int* n_pairs, int* n_changed) {
  if (n_pairs) *n_pairs = 0;
  if (n_changed) *n_changed = 0;
  if (!bm || !block_tables || !positions || !cow_pairs || !n_pairs || num_seqs < 0 ||
      max_blocks_per_seq <= 0)
    return PA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(bm->mu);
  int pairs = 0, changed = 0;
  pa_status st = PA_OK;
  for (int s = 0; s < num_seqs; ++s) {
    const int pos = positions[s];
    if (pos < 0) continue;
    const int lb = pos / bm->block_size;
    if (lb >= max_blocks_per_seq) {
      st = PA_ERR_INVALID_ARG;
      break;
    }
    int32_t* entry = block_tables + (size_t)s * max_blocks_per_seq + lb;
    const int pb = *entry;
    if (pb < 0) {
      const int nb = bm->alloc_locked();
      if (nb < 0) {
        st = PA_ERR_OUT_OF_BLOCKS;
        break;
      }
      *entry = nb;
      ++changed;
    } else if (pb < bm->num_blocks && bm->refcount[pb] > 1) {
      const int nb = bm->alloc_locked();
      if (nb < 0) {
        st = PA_ERR_OUT_OF_BLOCKS;
        break;
      }
      --bm->refcount[pb];  // still > 0: the other holders keep it
      *entry = nb;
      cow_pairs[2 * pairs] = pb;
      cow_pairs[2 * pairs + 1] = nb;
      ++pairs;
      ++changed;
    } else if (pb >= bm->num_blocks || bm->refcount[pb] == 0) {
      st = PA_ERR_INVALID_ARG;  // table names a block the pool does not hold
      break;
    }
  }
  *n_pairs = pairs;
  if (n_changed) *n_changed = changed;
  return st;
}

int pa_bm_slide_window(pa_bm* bm, int32_t* block_tables, int num_seqs, int max_blocks_per_seq,
                       const int32_t* context_lens, int window, int* n_freed) {
  if (n_freed) *n_freed = 0;
  if (!bm || !block_tables || !context_lens || num_seqs < 0 || max_blocks_per_seq <= 0 || window < 0)
    return -1;
  if (window == 0) return 0;
  std::lock_guard<std::mutex> g(bm->mu);
  int released = 0, freed = 0;
  for (int s = 0; s < num_seqs; ++s) {
    const int c = context_lens[s];
    if (c <= window) continue;
    const int n = std::min((c - window) / bm->block_size, max_blocks_per_seq);
    int32_t* row = block_tables + (size_t)s * max_blocks_per_seq;
    for (int lb = 0; lb < n; ++lb) {
      const int b = row[lb];
      if (b < 0) continue;
      if (!bm->valid_allocated(b)) {
        if (n_freed) *n_freed = freed;
        return -1;
      }
      if (--bm->refcount[b] == 0) {
        bm->release_locked(b);
        ++freed;
      }
      row[lb] = -1;
      ++released;
    }
  }
  if (n_freed) *n_freed = freed;
  return released;
}

}  // extern "C"

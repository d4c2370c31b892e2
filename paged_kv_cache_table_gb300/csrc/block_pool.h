// The host block pool behind pa_bm_* (block_manager.cpp), shared with the prefix cache
// (prefix_cache.cpp), which takes and drops references on the same pool under its lock.
#ifndef PA_BLOCK_POOL_H_
#define PA_BLOCK_POOL_H_

#include <algorithm>
#include <functional>
#include <mutex>
#include <vector>

struct pa_bm {
  int num_blocks = 0;
  int block_size = 0;
  std::vector<int> refcount;
  std::vector<int> free_heap;  // min-heap of free block ids
  std::vector<char> is_free;   // lazy deletion for claim()
  int nfree = 0;
  mutable std::mutex mu;

  int alloc_locked() {
    while (!free_heap.empty()) {
      std::pop_heap(free_heap.begin(), free_heap.end(), std::greater<int>());
      int b = free_heap.back();
      free_heap.pop_back();
      if (!is_free[b]) continue;  // claimed earlier: stale heap entry
      is_free[b] = 0;
      refcount[b] = 1;
      --nfree;
      return b;
    }
    return -1;
  }
  void release_locked(int b) {
    is_free[b] = 1;
    ++nfree;
    free_heap.push_back(b);
    std::push_heap(free_heap.begin(), free_heap.end(), std::greater<int>());
  }
  bool valid_allocated(int b) const { return b >= 0 && b < num_blocks && refcount[b] > 0; }
};

#endif  // PA_BLOCK_POOL_H_

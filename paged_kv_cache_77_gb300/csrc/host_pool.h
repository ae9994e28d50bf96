// BlockPool internals shared by the host generator and the request-level allocator.
//
// "KV Cache 管理设计文档" §2.4: a FIFO queue of free ids; the first id popped is the
// null block, never handed out. Each id also carries a reference count so that
// forked requests can share full blocks ("KV Cache 笔记", fork_blocks): 0 = free (or
// the null block), a popped id starts at 1, and it returns to the queue tail when
// its count drops back to 0.
#pragma once

#include <cstdint>
#include <deque>
#include <unordered_map>
#include <vector>

struct pkv_pool {
  int64_t num_blocks = 0;
  int32_t null_block = 0;
  std::deque<int32_t> queue;  // free ids, FIFO
  std::vector<int32_t> ref;   // reference count per id
};

namespace pkv {

// Pop n ids (the caller has checked that n are free); each gets one reference.
inline void pool_take(pkv_pool* p, int64_t n, int32_t* out) {
  for (int64_t i = 0; i < n; ++i) {
    const int32_t id = p->queue.front();
    p->queue.pop_front();
    p->ref[id] = 1;
    out[i] = id;
  }
}

// True if releasing ids[n] (one reference each) is valid: every id in range, not
// the null block, and listed at most as often as it is referenced.
inline bool pool_release_ok(const pkv_pool* p, const int32_t* ids, int64_t n) {
  std::unordered_map<int32_t, int32_t> count;
  for (int64_t i = 0; i < n; ++i) {
    const int32_t id = ids[i];
    if (id < 0 || id >= p->num_blocks || id == p->null_block) return false;
    if (++count[id] > p->ref[id]) return false;
  }
  return true;
}

// Drop one reference per id (validated by pool_release_ok); ids that reach zero go
// to the queue tail in the listed order and, if `released` is given, to it too.
inline void pool_release(pkv_pool* p, const int32_t* ids, int64_t n,
                         std::vector<int32_t>* released) {
  for (int64_t i = 0; i < n; ++i) {
    const int32_t id = ids[i];
    if (--p->ref[id] == 0) {
      p->queue.push_back(id);
      if (released) released->push_back(id);
    }
  }
}

}  // namespace pkv

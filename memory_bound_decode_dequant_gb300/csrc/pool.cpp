// pool.cpp -- host bookkeeping of the paged KV cache.
//
// "Mini Inference Engine", "The KV cache, paged like virtual memory": the cache is cut
// into fixed-size blocks handed out by integer id from a preallocated pool; each id
// carries a count of the sequences holding it, and running out is reported as a
// status, not thrown.  "Prefix sharing and copy-on-write": sequences may hold the same
// block; before one of them writes into a block that others also hold, it moves to a
// private copy, and the shared block must stay alive until that copy has been made.
//
// The block contents live on the GPU; this object only tracks ids and counts.  Every
// public call takes the pool's lock, so the pool may be shared between host threads.
#include <mutex>
#include <new>
#include <vector>

#include "../../include/mie.h"

namespace mie {
mie_status fail(mie_status s, const char *fmt, ...);
}

struct mie_pool {
  // holders[id] = number of sequences holding block id (0: free)
  std::vector<int> holders;
  // ids with no holder; the most recently freed id is handed out first, and a fresh
  // pool hands out 0, 1, 2, ...
  std::vector<int32_t> spare;
  std::mutex mu;

  explicit mie_pool(int n) : holders((size_t)n, 0) {
    spare.reserve((size_t)n);
    for (int id = n - 1; id >= 0; --id) spare.push_back(id);
  }
  int size() const { return (int)holders.size(); }
  bool held(int32_t id) const { return id >= 0 && id < size() && holders[(size_t)id] > 0; }

  // Hands out a block with one holder; false when none is spare.
  bool take(int32_t *id) {
    if (spare.empty()) return false;
    *id = spare.back();
    spare.pop_back();
    holders[(size_t)*id] = 1;
    return true;
  }
  // Drops one holder of a held block; the last one frees it.
  void release(int32_t id) {
    if (--holders[(size_t)id] == 0) spare.push_back(id);
  }
};

extern "C" mie_status mie_pool_create(int n_blocks, mie_pool **out) {
  if (!out) return mie::fail(MIE_E_ARG, "mie_pool_create: null out");
  *out = nullptr;
  if (n_blocks < 1) return mie::fail(MIE_E_SHAPE, "mie_pool_create: n_blocks = %d", n_blocks);
  mie_pool *p = new (std::nothrow) mie_pool(n_blocks);
  if (!p) return mie::fail(MIE_E_OOM, "mie_pool_create: out of host memory");
  *out = p;
  return MIE_OK;
}

extern "C" void mie_pool_destroy(mie_pool *p) { delete p; }

extern "C" mie_status mie_pool_alloc(mie_pool *p, int32_t *id) {
  if (!p || !id) return mie::fail(MIE_E_ARG, "mie_pool_alloc: null pointer");
  std::lock_guard<std::mutex> g(p->mu);
  if (!p->take(id)) {
    *id = -1;
    return mie::fail(MIE_E_OOM, "KV block pool exhausted (%d blocks)", p->size());
  }
  return MIE_OK;
}

extern "C" mie_status mie_pool_incref(mie_pool *p, int32_t id) {
  if (!p) return mie::fail(MIE_E_ARG, "mie_pool_incref: null pool");
  std::lock_guard<std::mutex> g(p->mu);
  if (!p->held(id)) return mie::fail(MIE_E_ARG, "mie_pool_incref: block %d is not live", id);
  ++p->holders[(size_t)id];
  return MIE_OK;
}

extern "C" mie_status mie_pool_decref(mie_pool *p, int32_t id) {
  if (!p) return mie::fail(MIE_E_ARG, "mie_pool_decref: null pool");
  std::lock_guard<std::mutex> g(p->mu);
  if (!p->held(id)) return mie::fail(MIE_E_ARG, "mie_pool_decref: block %d is not live", id);
  p->release(id);
  return MIE_OK;
}

extern "C" int mie_pool_refcount(const mie_pool *p, int32_t id) {
  if (!p || id < 0 || id >= p->size()) return -1;
  std::lock_guard<std::mutex> g(const_cast<mie_pool *>(p)->mu);
  return p->holders[(size_t)id];
}

extern "C" int mie_pool_free_count(const mie_pool *p) {
  if (!p) return -1;
  std::lock_guard<std::mutex> g(const_cast<mie_pool *>(p)->mu);
  return (int)p->spare.size();
}

// A write at logical position pos needs a block that the sequence holds alone.  When
// the table's block has other holders too, the sequence moves to a fresh block: the
// table entry changes now, but the sequence keeps its hold on the shared block, which
// it gives up (mie_pool_decref(copy_src)) only after the copy of the contents is
// queued.  Until then no other caller can free the shared block and hand it out again.
extern "C" mie_status mie_pool_writable(mie_pool *p, int32_t *table, int pos, int block_size, int32_t *block,
                                        int32_t *copy_src, int32_t *copy_dst) {
  if (!p || !table || !block || !copy_src || !copy_dst) return mie::fail(MIE_E_ARG, "mie_pool_writable: null pointer");
  if (pos < 0 || block_size < 1) return mie::fail(MIE_E_ARG, "mie_pool_writable: pos %d, block size %d", pos, block_size);
  *copy_src = *copy_dst = *block = -1;
  int32_t &entry = table[pos / block_size];
  std::lock_guard<std::mutex> g(p->mu);
  if (!p->held(entry)) return mie::fail(MIE_E_ARG, "mie_pool_writable: block %d is not live", entry);
  if (p->holders[(size_t)entry] > 1) {
    int32_t fresh = -1;
    if (!p->take(&fresh))
      return mie::fail(MIE_E_OOM, "KV block pool exhausted (%d blocks) on copy-on-write", p->size());
    *copy_src = entry;
    *copy_dst = fresh;
    entry = fresh;
  }
  *block = entry;
  return MIE_OK;
}

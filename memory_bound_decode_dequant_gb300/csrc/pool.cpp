// pool.cpp -- host bookkeeping of the paged KV cache.
//
// "Mini Inference Engine", "The KV cache, paged like virtual memory": the cache is cut
// into fixed-size blocks handed out from a preallocated pool by integer id, with a
// refcount per id and a LIFO free list; running out is a sentinel, not an exception.
// "Prefix sharing and copy-on-write": a shared block is split on its first write by
// allocate -> copy -> decref -> swap, so the source stays alive during the copy.
// The block contents live on the GPU; this object only tracks ids and counts.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "../../include/mie.h"

namespace mie {
mie_status fail(mie_status s, const char *fmt, ...);
}

struct mie_pool {
  std::vector<int> refcount;
  std::vector<int32_t> free_list;  // LIFO: back() is handed out next
  std::mutex mu;
};

extern "C" mie_status mie_pool_create(int n_blocks, mie_pool **out) {
  if (!out) return mie::fail(MIE_E_ARG, "mie_pool_create: null out");
  *out = nullptr;
  if (n_blocks < 1) return mie::fail(MIE_E_SHAPE, "mie_pool_create: n_blocks = %d", n_blocks);
  mie_pool *p = new (std::nothrow) mie_pool;
  if (!p) return mie::fail(MIE_E_OOM, "mie_pool_create: out of host memory");
  p->refcount.assign((size_t)n_blocks, 0);
  p->free_list.reserve((size_t)n_blocks);
  for (int i = n_blocks - 1; i >= 0; --i) p->free_list.push_back(i);  // hands out 0, 1, 2, ...
  *out = p;
  return MIE_OK;
}

extern "C" void mie_pool_destroy(mie_pool *p) { delete p; }

static bool live(const mie_pool *p, int32_t id) {
  return id >= 0 && (size_t)id < p->refcount.size() && p->refcount[(size_t)id] > 0;
}

static mie_status alloc_locked(mie_pool *p, int32_t *id) {
  if (p->free_list.empty()) {
    *id = -1;
    return mie::fail(MIE_E_OOM, "KV block pool exhausted (%zu blocks)", p->refcount.size());
  }
  *id = p->free_list.back();
  p->free_list.pop_back();
  p->refcount[(size_t)*id] = 1;
  return MIE_OK;
}

static mie_status decref_locked(mie_pool *p, int32_t id) {
  if (!live(p, id)) return mie::fail(MIE_E_ARG, "mie_pool_decref: block %d is not live", id);
  if (--p->refcount[(size_t)id] == 0) p->free_list.push_back(id);
  return MIE_OK;
}

extern "C" mie_status mie_pool_alloc(mie_pool *p, int32_t *id) {
  if (!p || !id) return mie::fail(MIE_E_ARG, "mie_pool_alloc: null pointer");
  std::lock_guard<std::mutex> g(p->mu);
  return alloc_locked(p, id);
}

extern "C" mie_status mie_pool_incref(mie_pool *p, int32_t id) {
  if (!p) return mie::fail(MIE_E_ARG, "mie_pool_incref: null pool");
  std::lock_guard<std::mutex> g(p->mu);
  if (!live(p, id)) return mie::fail(MIE_E_ARG, "mie_pool_incref: block %d is not live", id);
  ++p->refcount[(size_t)id];
  return MIE_OK;
}

extern "C" mie_status mie_pool_decref(mie_pool *p, int32_t id) {
  if (!p) return mie::fail(MIE_E_ARG, "mie_pool_decref: null pool");
  std::lock_guard<std::mutex> g(p->mu);
  return decref_locked(p, id);
}

extern "C" int mie_pool_refcount(const mie_pool *p, int32_t id) {
  if (!p || id < 0 || (size_t)id >= p->refcount.size()) return -1;
  std::lock_guard<std::mutex> g(const_cast<mie_pool *>(p)->mu);
  return p->refcount[(size_t)id];
}

extern "C" int mie_pool_free_count(const mie_pool *p) {
  if (!p) return -1;
  std::lock_guard<std::mutex> g(const_cast<mie_pool *>(p)->mu);
  return (int)p->free_list.size();
}

extern "C" mie_status mie_pool_writable(mie_pool *p, int32_t *table, int pos, int block_size, int32_t *block,
                                        int32_t *copy_src, int32_t *copy_dst) {
  if (!p || !table || !block || !copy_src || !copy_dst) return mie::fail(MIE_E_ARG, "mie_pool_writable: null pointer");
  if (pos < 0 || block_size < 1) return mie::fail(MIE_E_ARG, "mie_pool_writable: pos %d, block size %d", pos, block_size);
  std::lock_guard<std::mutex> g(p->mu);
  *copy_src = *copy_dst = -1;
  const int32_t old = table[pos / block_size];
  if (!live(p, old)) {
    *block = -1;
    return mie::fail(MIE_E_ARG, "mie_pool_writable: block %d is not live", old);
  }
  if (p->refcount[(size_t)old] == 1) {
    *block = old;
    return MIE_OK;
  }
  int32_t nw = -1;
  const mie_status s = alloc_locked(p, &nw);
  if (s != MIE_OK) {
    *block = -1;
    return s;
  }
  // The caller copies old -> nw before writing; the source keeps its other holders.
  *copy_src = old;
  *copy_dst = nw;
  decref_locked(p, old);
  table[pos / block_size] = nw;
  *block = nw;
  return MIE_OK;
}

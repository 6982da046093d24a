// Host-side document cache manager: which documents' K/V pages are resident in the paged pool.
//
// [NOTE] 研究背景与动机 (核心矛盾) and 关键设计 (Deferred Positional Encoding): with a
// position-free cache one physical copy of a document serves every position it is placed at,
// so a fixed page budget holds more distinct documents than a position-aware cache, which
// needs one copy per (document, position) variant.  Both policies are implemented here behind
// one interface so an engine can use the first and a simulator can compare the two:
//   - position_agnostic: key = document id;
//   - position-aware:    key = (document id, position index).
// Pages come from a fixed pool [0, num_pages).  Eviction is least-recently-used among entries
// that no running batch holds (pinned entries are never evicted).  Pure host code, no CUDA.
#include <cstdint>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "lazykv.h"

namespace lazykv {
int fail(int code, const char* fmt, ...);
}

struct lazy_doc_cache {
  struct Entry {
    std::vector<int32_t> pages;
    int pins = 0;
    std::list<uint64_t>::iterator lru;  // position in `order` (front = most recent)
  };
  int num_pages = 0;
  bool position_aware = false;
  std::vector<int32_t> free_pages;
  std::unordered_map<uint64_t, Entry> entries;
  std::list<uint64_t> order;
  long long hits = 0, misses = 0, evictions = 0;

  uint64_t key(int doc, int pos) const {
    return position_aware ? (uint64_t(uint32_t(doc)) << 32) | uint32_t(pos) : uint64_t(uint32_t(doc));
  }
  void touch(Entry& e, uint64_t k) {
    order.erase(e.lru);
    order.push_front(k);
    e.lru = order.begin();
  }
  // Evict unpinned entries from the LRU end until `need` pages are free; false if impossible.
  bool make_room(int need) {
    auto it = order.end();
    while (int(free_pages.size()) < need && it != order.begin()) {
      --it;
      auto e = entries.find(*it);
      if (e->second.pins > 0) continue;
      for (int32_t p : e->second.pages) free_pages.push_back(p);
      auto dead = it;
      ++it;  // `it` stays valid: erase only invalidates `dead`
      entries.erase(e);
      order.erase(dead);
      ++evictions;
    }
    return int(free_pages.size()) >= need;
  }
};

extern "C" lazy_doc_cache* lazy_doc_cache_create(int num_pages, int position_aware) {
  if (num_pages <= 0 || num_pages > (1 << 24)) {
    lazykv::fail(LAZY_EINVAL, "doc cache: num_pages %d outside [1, 2^24]", num_pages);
    return nullptr;
  }
  lazy_doc_cache* c = new (std::nothrow) lazy_doc_cache();
  if (!c) {
    lazykv::fail(LAZY_EINVAL, "doc cache: out of host memory");
    return nullptr;
  }
  c->num_pages = num_pages;
  c->position_aware = position_aware != 0;
  c->free_pages.reserve(num_pages);
  for (int p = num_pages - 1; p >= 0; --p) c->free_pages.push_back(p);  // hand out low ids first
  return c;
}

extern "C" void lazy_doc_cache_destroy(lazy_doc_cache* c) { delete c; }

extern "C" int lazy_doc_cache_lookup(lazy_doc_cache* c, int doc, int pos, int32_t* pages_out, int max_pages) {
  if (!c || doc < 0 || pos < 0) return lazykv::fail(LAZY_EINVAL, "doc cache: bad handle or ids");
  const uint64_t k = c->key(doc, pos);
  auto it = c->entries.find(k);
  if (it == c->entries.end()) return 0;
  const int n = int(it->second.pages.size());
  if (pages_out) {
    if (max_pages < n) return lazykv::fail(LAZY_EINVAL, "doc cache: pages_out holds %d, need %d", max_pages, n);
    for (int i = 0; i < n; ++i) pages_out[i] = it->second.pages[i];
  }
  return n;
}

extern "C" int lazy_doc_cache_acquire(lazy_doc_cache* c, int doc, int pos, int n_pages, int32_t* pages_out,
                                      int* hit) {
  if (!c || doc < 0 || pos < 0 || n_pages <= 0 || !pages_out || !hit)
    return lazykv::fail(LAZY_EINVAL, "doc cache: bad arguments");
  const uint64_t k = c->key(doc, pos);
  auto it = c->entries.find(k);
  if (it != c->entries.end()) {
    lazy_doc_cache::Entry& e = it->second;
    if (int(e.pages.size()) != n_pages)
      return lazykv::fail(LAZY_EINVAL, "doc cache: document %d cached with %d pages, asked for %d", doc,
                          int(e.pages.size()), n_pages);
    ++e.pins;
    c->touch(e, k);
    for (int i = 0; i < n_pages; ++i) pages_out[i] = e.pages[i];
    *hit = 1;
    ++c->hits;
    return LAZY_OK;
  }
  if (n_pages > c->num_pages) return lazykv::fail(LAZY_ERANGE, "doc cache: %d pages exceed the pool", n_pages);
  if (!c->make_room(n_pages))
    return lazykv::fail(LAZY_ERANGE, "doc cache: no room for %d pages (pinned entries hold the pool)", n_pages);
  lazy_doc_cache::Entry e;
  e.pages.resize(n_pages);
  for (int i = 0; i < n_pages; ++i) {
    e.pages[i] = c->free_pages.back();
    c->free_pages.pop_back();
    pages_out[i] = e.pages[i];
  }
  e.pins = 1;
  c->order.push_front(k);
  e.lru = c->order.begin();
  c->entries.emplace(k, std::move(e));
  *hit = 0;
  ++c->misses;
  return LAZY_OK;
}

extern "C" int lazy_doc_cache_release(lazy_doc_cache* c, int doc, int pos) {
  if (!c) return lazykv::fail(LAZY_EINVAL, "doc cache: bad handle");
  auto it = c->entries.find(c->key(doc, pos));
  if (it == c->entries.end() || it->second.pins <= 0)
    return lazykv::fail(LAZY_EINVAL, "doc cache: document %d (position %d) is not held", doc, pos);
  --it->second.pins;
  return LAZY_OK;
}

extern "C" int lazy_doc_cache_stats(const lazy_doc_cache* c, long long* hits, long long* misses,
                                    long long* evictions, int* entries, int* free_pages) {
  if (!c) return lazykv::fail(LAZY_EINVAL, "doc cache: bad handle");
  if (hits) *hits = c->hits;
  if (misses) *misses = c->misses;
  if (evictions) *evictions = c->evictions;
  if (entries) *entries = int(c->entries.size());
  if (free_pages) *free_pages = int(c->free_pages.size());
  return LAZY_OK;
}

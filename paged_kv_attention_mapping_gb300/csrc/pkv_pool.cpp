// Host-side page pool: free list, reference counts and the prefix cache.
//
// Helios README, "Paged attention": a fixed pool of pages; new tokens take
// pages from the free list; a page returns to the pool when the last request
// or prefix-cache entry that holds it lets go. Helios blog, "Prefix caching":
// complete page-size prompt blocks are keyed by a hash chained with the
// previous block's hash; a new request finds the longest matching chain and
// shares those physical pages; partial blocks are never stored; cached blocks
// live on with a sliding TTL and eviction takes unused blocks that no later
// block depends on (leaves) first.
//
// Definitions fixed here (the pages leave them open):
//  * allocation hands out the lowest free page id first;
//  * chain hash h_i = mix(h_{i-1}, tokens of block i), h_{-1} = a fixed seed,
//    mix = splitmix64 finalisation folded over the tokens; entries also keep
//    their tokens, and a lookup only matches when the tokens are equal;
//  * an entry is evictable when the cache is the page's only holder and no
//    cached block has it as parent; eviction order is oldest last use first,
//    ties by lower page id; expired entries (now - last_use > ttl) go first.
#include <stdint.h>

#include <map>
#include <new>
#include <set>
#include <unordered_map>
#include <vector>

#include "pagedkv.h"

namespace {

constexpr uint64_t CHAIN_SEED = 0x70616765645f6b76ull;  // "paged_kv"

uint64_t mix64(uint64_t x) {
  x += 0x9e3779b97f4a7c15ull;
  x = (x ^ (x >> 30)) * 0xbf58476d1ce4e5b9ull;
  x = (x ^ (x >> 27)) * 0x94d049bb133111ebull;
  return x ^ (x >> 31);
}

uint64_t chain_hash(uint64_t prev, const int32_t* tok, int32_t n) {
  uint64_t h = mix64(prev ^ 0xa0761d6478bd642full);
  for (int32_t i = 0; i < n; ++i) h = mix64(h ^ (uint64_t)(uint32_t)tok[i]);
  return h;
}

struct Entry {
  uint64_t parent = 0;
  bool has_parent = false;
  int32_t page = -1;
  int32_t children = 0;
  double last_use = 0.0;
  std::vector<int32_t> tokens;
};

}  // namespace

struct pkv_pool {
  int32_t num_pages = 0, page_size = 0;
  std::vector<int32_t> ref;
  std::set<int32_t> free_pages;
  std::unordered_map<uint64_t, Entry> cache;

  void drop(int32_t p) {
    if (--ref[p] == 0) free_pages.insert(p);
  }

  bool evictable(const Entry& e) const { return e.children == 0 && ref[e.page] == 1; }

  // oldest evictable entry (optionally only expired ones); false when none
  bool pick(double now, double ttl, bool expired_only, uint64_t* key) const {
    bool found = false;
    double best_t = 0.0;
    int32_t best_p = 0;
    for (const auto& kv : cache) {
      const Entry& e = kv.second;
      if (!evictable(e)) continue;
      if (expired_only && !(now - e.last_use > ttl)) continue;
      if (!found || e.last_use < best_t || (e.last_use == best_t && e.page < best_p)) {
        found = true;
        best_t = e.last_use;
        best_p = e.page;
        *key = kv.first;
      }
    }
    return found;
  }

  void evict(uint64_t key) {
    Entry e = cache[key];
    cache.erase(key);
    if (e.has_parent) {
      auto it = cache.find(e.parent);
      if (it != cache.end()) it->second.children -= 1;
    }
    drop(e.page);
  }
};

extern "C" int pkv_pool_create(int32_t num_pages, int32_t page_size, pkv_pool** out) {
  if (!out) return PKV_E_NULL;
  if (num_pages < 1 || page_size < 1) return PKV_E_SHAPE;
  pkv_pool* p = new (std::nothrow) pkv_pool();
  if (!p) return PKV_E_CAPACITY;
  p->num_pages = num_pages;
  p->page_size = page_size;
  p->ref.assign(num_pages, 0);
  for (int32_t i = 0; i < num_pages; ++i) p->free_pages.insert(i);
  *out = p;
  return PKV_OK;
}

extern "C" void pkv_pool_destroy(pkv_pool* p) { delete p; }

extern "C" int pkv_pool_free_count(const pkv_pool* p) { return p ? (int)p->free_pages.size() : PKV_E_NULL; }

extern "C" int pkv_pool_refcount(const pkv_pool* p, int32_t page) {
  if (!p) return PKV_E_NULL;
  if (page < 0 || page >= p->num_pages) return PKV_E_PAGES;
  return p->ref[page];
}

extern "C" int pkv_pool_alloc(pkv_pool* p, int32_t n, int32_t* pages) {
  if (!p || (n > 0 && !pages)) return PKV_E_NULL;
  if (n < 0) return PKV_E_SHAPE;
  if ((size_t)n > p->free_pages.size()) return PKV_E_CAPACITY;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t pg = *p->free_pages.begin();
    p->free_pages.erase(p->free_pages.begin());
    p->ref[pg] = 1;
    pages[i] = pg;
  }
  return PKV_OK;
}

extern "C" int pkv_pool_retain(pkv_pool* p, const int32_t* pages, int32_t n) {
  if (!p || (n > 0 && !pages)) return PKV_E_NULL;
  for (int32_t i = 0; i < n; ++i)
    if (pages[i] < 0 || pages[i] >= p->num_pages || p->ref[pages[i]] == 0) return PKV_E_PAGES;
  for (int32_t i = 0; i < n; ++i) p->ref[pages[i]] += 1;
  return PKV_OK;
}

extern "C" int pkv_pool_release(pkv_pool* p, const int32_t* pages, int32_t n) {
  if (!p || (n > 0 && !pages)) return PKV_E_NULL;
  // check first, so a bad list changes nothing (a page may appear several times)
  std::map<int32_t, int32_t> count;
  for (int32_t i = 0; i < n; ++i) {
    if (pages[i] < 0 || pages[i] >= p->num_pages) return PKV_E_PAGES;
    if (++count[pages[i]] > p->ref[pages[i]]) return PKV_E_PAGES;
  }
  for (int32_t i = 0; i < n; ++i) p->drop(pages[i]);
  return PKV_OK;
}

extern "C" int pkv_prefix_lookup(pkv_pool* p, const int32_t* tokens, int32_t n_tokens, double now, int32_t* pages,
                                 int32_t max_pages) {
  if (!p || (n_tokens > 0 && !tokens) || (max_pages > 0 && !pages)) return PKV_E_NULL;
  if (n_tokens < 0 || max_pages < 0) return PKV_E_SHAPE;
  const int32_t P = p->page_size;
  uint64_t h = CHAIN_SEED;
  int32_t n = 0;
  for (int32_t b = 0; b < n_tokens / P && n < max_pages; ++b) {
    const uint64_t hb = chain_hash(h, tokens + (int64_t)b * P, P);
    auto it = p->cache.find(hb);
    if (it == p->cache.end()) break;
    Entry& e = it->second;
    bool same = (int32_t)e.tokens.size() == P && (b == 0 ? !e.has_parent : (e.has_parent && e.parent == h));
    for (int32_t i = 0; same && i < P; ++i) same = e.tokens[i] == tokens[(int64_t)b * P + i];
    if (!same) break;
    e.last_use = now;
    p->ref[e.page] += 1;  // the caller now holds the page too
    pages[n++] = e.page;
    h = hb;
  }
  return n;
}

extern "C" int pkv_prefix_insert(pkv_pool* p, const int32_t* tokens, int32_t n_tokens, const int32_t* pages,
                                 int32_t n_pages, double now) {
  if (!p || (n_tokens > 0 && !tokens) || (n_pages > 0 && !pages)) return PKV_E_NULL;
  if (n_tokens < 0 || n_pages < 0) return PKV_E_SHAPE;
  const int32_t P = p->page_size;
  const int32_t blocks = n_tokens / P;  // partial last blocks are not stored
  if (blocks > n_pages) return PKV_E_PAGES;
  for (int32_t b = 0; b < blocks; ++b)
    if (pages[b] < 0 || pages[b] >= p->num_pages || p->ref[pages[b]] == 0) return PKV_E_PAGES;
  uint64_t h = CHAIN_SEED;
  int32_t added = 0;
  for (int32_t b = 0; b < blocks; ++b) {
    const uint64_t hb = chain_hash(h, tokens + (int64_t)b * P, P);
    auto it = p->cache.find(hb);
    if (it != p->cache.end()) {
      it->second.last_use = now;  // already cached (possibly on another page): keep that one
    } else {
      Entry e;
      e.parent = h;
      e.has_parent = b > 0;
      e.page = pages[b];
      e.last_use = now;
      e.tokens.assign(tokens + (int64_t)b * P, tokens + (int64_t)(b + 1) * P);
      p->ref[e.page] += 1;  // the cache holds the page
      if (b > 0) {
        auto par = p->cache.find(h);
        if (par != p->cache.end()) par->second.children += 1;
      }
      p->cache.emplace(hb, std::move(e));
      ++added;
    }
    h = hb;
  }
  return added;
}

extern "C" int pkv_prefix_evict(pkv_pool* p, double now, double ttl, int32_t want_free) {
  if (!p) return PKV_E_NULL;
  int32_t freed = 0;
  uint64_t key = 0;
  while (p->pick(now, ttl, true, &key)) {
    p->evict(key);
    ++freed;
  }
  while ((int32_t)p->free_pages.size() < want_free && p->pick(now, ttl, false, &key)) {
    p->evict(key);
    ++freed;
  }
  return freed;
}

extern "C" int pkv_prefix_size(const pkv_pool* p) { return p ? (int)p->cache.size() : PKV_E_NULL; }

"""Reference model of the host page pool and prefix cache — TEST INFRASTRUCTURE.

Plain Python, written from the serving pages' description: a fixed pool of
page ids handed out from a free list, a page freed when the last holder (a
request or the prefix cache) lets go (Helios README, "Paged attention"), and a
cache of complete page-size prompt blocks where a block is identified by the
whole prompt up to and including it, a request reusing the longest cached
chain, partial blocks never stored, a sliding TTL, and eviction of unused
blocks that no later block depends on (Helios blog, "Prefix caching").

Where the pages leave it open this model fixes: the lowest free id is handed
out first; eviction takes the oldest last use first (ties: lower page id),
expired entries before any others. Blocks are compared by their full token
prefix, so this model needs no hash at all.
"""
from __future__ import annotations


class PoolError(ValueError):
    pass


class PagePoolModel:
    def __init__(self, num_pages: int, page_size: int):
        if num_pages < 1 or page_size < 1:
            raise PoolError("sizes")
        self.P = page_size
        self.ref = [0] * num_pages
        self.entries = {}   # prefix tuple -> dict(page, last_use)

    # -- pages
    def free_count(self):
        return sum(1 for r in self.ref if r == 0)

    def alloc(self, n):
        free = [p for p, r in enumerate(self.ref) if r == 0]
        if n > len(free):
            raise PoolError("capacity")
        out = free[:n]
        for p in out:
            self.ref[p] = 1
        return out

    def retain(self, pages):
        for p in pages:
            if not 0 <= p < len(self.ref) or self.ref[p] == 0:
                raise PoolError("page")
        for p in pages:
            self.ref[p] += 1

    def release(self, pages):
        need = {}
        for p in pages:
            if not 0 <= p < len(self.ref):
                raise PoolError("page")
            need[p] = need.get(p, 0) + 1
            if need[p] > self.ref[p]:
                raise PoolError("page")
        for p in pages:
            self.ref[p] -= 1

    # -- prefix cache
    def _blocks(self, tokens):
        return [tuple(tokens[:(b + 1) * self.P]) for b in range(len(tokens) // self.P)]

    def lookup(self, tokens, now, max_pages=1 << 30):
        out = []
        for key in self._blocks(tokens)[:max_pages]:
            e = self.entries.get(key)
            if e is None:
                break
            e["last_use"] = now
            self.ref[e["page"]] += 1
            out.append(e["page"])
        return out

    def insert(self, tokens, pages, now):
        keys = self._blocks(tokens)
        if len(keys) > len(pages) or any(not 0 <= pages[b] < len(self.ref) or self.ref[pages[b]] == 0
                                         for b in range(len(keys))):
            raise PoolError("page")
        added = 0
        for b, key in enumerate(keys):
            if key in self.entries:
                self.entries[key]["last_use"] = now
            else:
                self.entries[key] = dict(page=pages[b], last_use=now)
                self.ref[pages[b]] += 1
                added += 1
        return added

    def _evictable(self):
        out = []
        for key, e in self.entries.items():
            has_child = any(len(k) == len(key) + self.P and k[:len(key)] == key for k in self.entries)
            if not has_child and self.ref[e["page"]] == 1:
                out.append((e["last_use"], e["page"], key))
        return sorted(out)

    def evict(self, now, ttl, want_free=0):
        dropped = 0
        while True:
            cand = [c for c in self._evictable() if now - c[0] > ttl]
            if not cand:
                break
            self._drop(cand[0][2])
            dropped += 1
        while self.free_count() < want_free:
            cand = self._evictable()
            if not cand:
                break
            self._drop(cand[0][2])
            dropped += 1
        return dropped

    def _drop(self, key):
        e = self.entries.pop(key)
        self.ref[e["page"]] -= 1

    def cache_size(self):
        return len(self.entries)

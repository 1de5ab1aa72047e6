"""The library's host page pool and prefix cache against the reference model
(randomised operation sequences, compared step by step), plus the sharing
pattern of the long-context shared-prefix workload built from real requests."""
import numpy as np
import pytest

from oracle.page_pool import PagePoolModel, PoolError
from paged_kv_attention_mapping_gb300 import binding


@pytest.fixture(scope="module")
def lib():
    from paged_kv_attention_mapping_gb300 import build
    build.build()
    return binding.lib()


def state(pool, model):
    assert pool.free_count() == model.free_count()
    assert [pool.refcount(p) for p in range(len(model.ref))] == model.ref
    assert pool.cache_size() == model.cache_size()


@pytest.mark.parametrize("seed", range(8))
def test_random_operations_match_the_model(lib, seed):
    rng = np.random.default_rng(seed)
    N, P = int(rng.integers(6, 30)), int(rng.choice([2, 3, 4]))
    pool, model = binding.PagePool(N, P), PagePoolModel(N, P)
    vocab = int(rng.integers(2, 4))           # small vocabulary: prompts share prefixes often
    held = []                                  # page lists held by live "requests"
    now = 0.0
    for _ in range(300):
        now += float(rng.uniform(0, 2))
        op = rng.integers(0, 6)
        if op == 0:                            # a request allocates pages
            n = int(rng.integers(0, 5))
            try:
                want = model.alloc(n)
            except PoolError:
                with pytest.raises(binding.PagedKVError):
                    pool.alloc(n)
                continue
            assert pool.alloc(n) == want
            held.append(want)
        elif op == 1 and held:                 # a request finishes
            pages = held.pop(int(rng.integers(0, len(held))))
            model.release(pages)
            pool.release(pages)
        elif op == 2:                          # a new request looks up its prompt
            toks = [int(x) for x in rng.integers(0, vocab, size=int(rng.integers(0, 4 * P + 2)))]
            got = pool.lookup(toks, now)
            assert got == model.lookup(toks, now)
            if got:
                held.append(got)
        elif op == 3 and held:                 # a request stores its completed prompt blocks
            pages = held[int(rng.integers(0, len(held)))]
            toks = [int(x) for x in rng.integers(0, vocab, size=len(pages) * P + int(rng.integers(0, P)))]
            assert pool.insert(toks, pages, now) == model.insert(toks, pages, now)
        elif op == 4:                          # eviction: TTL and memory pressure
            ttl, want = float(rng.uniform(0, 6)), int(rng.integers(0, N))
            assert pool.evict(now, ttl, want) == model.evict(now, ttl, want)
        elif op == 5 and held:                 # an extra holder of some pages
            pages = held[int(rng.integers(0, len(held)))]
            model.retain(pages)
            pool.retain(pages)
            held.append(list(pages))
        state(pool, model)


def test_errors_change_nothing(lib):
    pool, model = binding.PagePool(4, 2), PagePoolModel(4, 2)
    a = pool.alloc(2)
    model.alloc(2)
    for bad in ([5], [3], a + a + a):
        with pytest.raises(binding.PagedKVError):
            pool.release(bad)
    with pytest.raises(binding.PagedKVError):
        pool.alloc(3)
    with pytest.raises(binding.PagedKVError):
        pool.retain([3])
    state(pool, model)


def test_partial_blocks_are_not_cached_and_lookups_share_pages(lib):
    pool = binding.PagePool(8, 4)
    pages = pool.alloc(3)
    prompt = list(range(10))                   # 2 full blocks + 2 tokens
    assert pool.insert(prompt, pages, 0.0) == 2
    assert pool.lookup(prompt, 1.0) == pages[:2]
    assert pool.lookup([0, 1, 2, 3, 9, 9, 9, 9], 1.0) == pages[:1]   # diverges in block 2
    assert pool.lookup([1, 2, 3, 4], 1.0) == []                        # block 1 alone is not a chain start


def test_shared_prefix_tables_from_requests(lib):
    """16 requests with one 4096-token system prompt and private continuations:
    the first stores the prompt's 16 blocks, the others reuse its pages, which
    gives the page-table structure of the long-context shared-prefix workload."""
    P = 256
    pool = binding.PagePool(16 + 16 * 112 + 8, P)
    rng = np.random.default_rng(3)
    system = [int(x) for x in rng.integers(0, 32000, size=16 * P)]
    tables = []
    for r in range(16):
        got = pool.lookup(system, float(r))
        if r == 0:
            assert got == []
            got = pool.alloc(16)
            assert pool.insert(system, got, 0.0) == 16
        tail = pool.alloc(112)
        tables.append(got + tail)
    first = tables[0][:16]
    assert all(t[:16] == first for t in tables)
    priv = [p for t in tables for p in t[16:]]
    assert len(set(priv)) == len(priv) == 16 * 112
    assert all(pool.refcount(p) == 17 for p in first)     # 16 requests + the cache
    # all requests finish: only the cache keeps the prefix; eviction under pressure frees it
    for t in tables:
        pool.release(t)
    assert all(pool.refcount(p) == 1 for p in first)
    assert pool.evict(100.0, 1e9, want_free=pool.num_pages) == 16
    assert pool.free_count() == pool.num_pages


# ---------------------------------------------------------------------------
# the reference model itself, pinned to hand-worked sequences (Helios README,
# "Paged attention": a page is free again when its last holder lets go; Helios
# blog, "Prefix caching": full blocks only, longest chain reused, sliding TTL,
# unused leaf blocks evicted first)

def test_model_hand_worked_allocation_and_release():
    m = PagePoolModel(5, 2)
    assert m.alloc(2) == [0, 1] and m.alloc(1) == [2]       # lowest free ids first
    m.retain([1, 1])
    assert m.ref == [1, 3, 1, 0, 0]
    m.release([1, 0])
    assert m.ref == [0, 2, 1, 0, 0] and m.free_count() == 3
    assert m.alloc(1) == [0]                                 # a freed page is reused
    with pytest.raises(PoolError):
        m.release([3])                                       # free page
    with pytest.raises(PoolError):
        m.alloc(3)                                           # two pages left
    assert m.ref == [1, 2, 1, 0, 0]                          # failed calls changed nothing


def test_model_hand_worked_prefix_cache_and_eviction():
    m = PagePoolModel(6, 2)
    a = m.alloc(3)                                           # [0, 1, 2]
    assert m.insert([7, 7, 8, 8, 9], a, now=0.0) == 2        # blocks (7,7) and (7,7,8,8); 9 is partial
    assert m.ref == [2, 2, 1, 0, 0, 0]
    assert m.lookup([7, 7, 8, 8, 5, 5], now=1.0) == [0, 1]   # longest chain, caller gets a reference
    assert m.lookup([7, 7, 6, 6], now=2.0) == [0]            # diverges in the second block
    assert m.lookup([8, 8], now=2.0) == []                   # (8,8) is cached only after (7,7)
    assert m.ref == [4, 3, 1, 0, 0, 0]
    m.release(a)
    m.release([0, 1])
    m.release([0])
    assert m.ref == [1, 1, 0, 0, 0, 0]                       # only the cache holds 0 and 1
    # page 0 has a cached child (page 1), so the leaf 1 goes first, then 0
    assert m.evict(now=3.0, ttl=100.0, want_free=5) == 1
    assert m.ref == [1, 0, 0, 0, 0, 0] and m.cache_size() == 1
    assert m.evict(now=3.0, ttl=100.0, want_free=6) == 1
    assert m.cache_size() == 0 and m.free_count() == 6
    # TTL: an entry unused for longer than ttl goes even when no page is wanted
    b = m.alloc(1)
    m.insert([1, 2], b, now=10.0)
    m.release(b)
    assert m.evict(now=11.0, ttl=5.0) == 0
    assert m.evict(now=16.5, ttl=5.0) == 1

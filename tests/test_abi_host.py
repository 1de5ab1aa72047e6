"""The C-ABI library on the host: it loads, exports every call the header
declares, and its host-only packing matches the oracle bit for bit (no GPU)."""
import os
import re

import numpy as np
import pytest

import oracle
from paged_kv_attention_mapping_gb300 import binding
from paged_kv_attention_mapping_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_attention_mapping_gb300 import build
    build.build()
    return binding.lib()


def header_functions():
    text = open(os.path.join(ROOT, "include", "pagedkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_call(lib):
    names = header_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(binding.EXPORTED)
    assert "sm_103a" in binding.version()


def test_status_strings(lib):
    for code in range(-10, 1):
        assert binding.status_string(code) not in ("", "unknown status")
    assert binding.status_string(-99) == "unknown status"


def _rand_requests(rng, B, P):
    q_lens = [int(x) for x in rng.choice([0, 1, 1, 1, 2, 5, 17], size=B)]
    kv = [max(q, 1) + int(rng.integers(0, 40)) for q in q_lens]
    need = [-(-L // P) for L in kv]
    extra = [int(rng.integers(0, 2)) for _ in range(B)]
    n_pages = sum(n + e for n, e in zip(need, extra)) + 3
    perm = [int(p) for p in rng.permutation(n_pages)]
    pages, pos = [], 0
    for n, e in zip(need, extra):
        pages.append(perm[pos:pos + n + e])
        pos += n + e
    return q_lens, kv, pages, n_pages


@pytest.mark.parametrize("seed", range(6))
def test_pack_tick_matches_oracle(lib, seed):
    rng = np.random.default_rng(seed)
    P = int(rng.choice([1, 3, 16]))
    q_lens, kv, pages, n_pages = _rand_requests(rng, int(rng.integers(1, 12)), P)
    width = max(len(p) for p in pages) + int(rng.integers(0, 3))
    got = binding.pack_tick(q_lens, kv, pages, P, n_pages, width)
    want = oracle.pack_tick(q_lens, kv, pages, P, width)
    for k in ("order", "cu_seqlens_q", "kv_lens", "page_tables", "slot_mapping"):
        assert np.array_equal(got[k], want[k]), k


@pytest.mark.parametrize("name", W.WORKLOADS)
def test_pack_tick_matches_oracle_on_named_workloads(lib, name):
    w = W.make_workload(name)
    q = [r.q_len for r in w.requests]
    kv = [r.kv_len for r in w.requests]
    pg = [r.pages for r in w.requests]
    got = binding.pack_tick(q, kv, pg, w.shape.page_size, w.num_pages)
    want = oracle.pack_tick(q, kv, pg, w.shape.page_size)
    for k in ("order", "cu_seqlens_q", "kv_lens", "page_tables", "slot_mapping"):
        assert np.array_equal(got[k], want[k]), k


@pytest.mark.parametrize("seed", range(4))
def test_pack_tick_flat_into_preallocated_buffers(lib, seed):
    """The flat-array form writes the oracle's packing into caller buffers, and
    the same buffers can be reused for the next tick (stale contents overwritten)."""
    rng = np.random.default_rng(100 + seed)
    P = int(rng.choice([1, 3, 16]))
    q_lens, kv, pages, n_pages = _rand_requests(rng, int(rng.integers(1, 12)), P)
    B = len(q_lens)
    width = max(len(p) for p in pages) + int(rng.integers(0, 3))
    offs = np.zeros(B + 1, dtype=np.int32)
    offs[1:] = np.cumsum([len(p) for p in pages])
    ids = np.concatenate([np.asarray(p, dtype=np.int32) for p in pages])
    cap = max(sum(max(q, 0) for q in q_lens), 1)
    out = dict(order=np.full(B, 77, np.int32), cu_seqlens_q=np.full(B + 1, 77, np.int32),
               kv_lens=np.full(B, 77, np.int32), page_tables=np.full((B, width), 77, np.int32),
               slot_mapping=np.full(cap, 77, np.int64))
    want = oracle.pack_tick(q_lens, kv, pages, P, width)
    for _ in range(2):
        got = binding.pack_tick_flat(q_lens, kv, offs, ids, P, n_pages, width, out=out)
        for k in ("order", "cu_seqlens_q", "kv_lens", "page_tables", "slot_mapping"):
            assert np.array_equal(got[k], want[k]), k
            assert np.shares_memory(got[k], out[k]), k
    fresh = binding.pack_tick_flat(q_lens, kv, offs, ids, P, n_pages, width)
    for k in want:
        assert np.array_equal(fresh[k], want[k]), k


def test_pack_tick_flat_rejects_small_or_mistyped_buffers(lib):
    offs = np.array([0, 1, 2], np.int32)
    ids = np.array([0, 1], np.int32)
    good = dict(order=np.zeros(2, np.int32), cu_seqlens_q=np.zeros(3, np.int32), kv_lens=np.zeros(2, np.int32),
                page_tables=np.zeros((2, 1), np.int32), slot_mapping=np.zeros(2, np.int64))
    binding.pack_tick_flat([1, 1], [3, 3], offs, ids, 4, 2, 1, out=good)
    for key, bad in (("slot_mapping", np.zeros(1, np.int64)), ("slot_mapping", np.zeros(2, np.int32)),
                     ("page_tables", np.zeros((2, 2), np.int32)), ("cu_seqlens_q", np.zeros(2, np.int32))):
        o = dict(good)
        o[key] = bad
        with pytest.raises(ValueError):
            binding.pack_tick_flat([1, 1], [3, 3], offs, ids, 4, 2, 1, out=o)
    with pytest.raises(ValueError):
        binding.pack_tick_flat([1, 1], [3, 3], offs[:2], ids, 4, 2, 1)


def test_pack_tick_rejects_bad_inputs(lib):
    ok = dict(q_lens=[1, 3], kv_lens=[4, 3], pages=[[0], [1]], page_size=4, num_pages=2)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return binding.pack_tick(a["q_lens"], a["kv_lens"], a["pages"], a["page_size"], a["num_pages"],
                                 a.get("width"))

    call()
    with pytest.raises(binding.PagedKVError) as e:
        call(kv_lens=[4, 2])                 # kv_len < q_len
    assert e.value.status == -4
    with pytest.raises(binding.PagedKVError) as e:
        call(pages=[[0], [2]])               # page outside the pool
    assert e.value.status == -5
    with pytest.raises(binding.PagedKVError) as e:
        call(kv_lens=[5, 3])                 # 5 tokens need 2 pages of 4
    assert e.value.status == -5
    with pytest.raises(binding.PagedKVError) as e:
        call(q_lens=[-1, 3])
    assert e.value.status == -4
    with pytest.raises(binding.PagedKVError) as e:
        call(page_size=0)
    assert e.value.status == -3


def test_workspace_size(lib):
    import torch
    kc = torch.empty((8, 16, 2, 64), dtype=torch.bfloat16)
    n = binding.workspace_size(4, 10, 8, kc, 128)
    assert n > 0 and n % 256 == 0
    assert binding.workspace_size(4, 20, 8, kc, 128) >= n
    with pytest.raises(binding.PagedKVError):
        binding.workspace_size(4, 10, 7, kc, 128)   # Hq % Hkv != 0


def test_attention_rejects_unsupported_shapes_on_the_host(lib):
    """Group sizes outside 1..8 and 16, and head_dim outside {64, 128, 256}, are
    refused before any device work (PKV_E_SHAPE); an fp8 cache needs head_dim 128."""
    import ctypes
    fake = ctypes.c_void_p(256)
    for heads, kv_heads, d in ((40, 4, 128), (32, 8, 96), (36, 3, 128), (24, 1, 64), (8, 2, 192), (8, 2, 512)):
        desc = binding.CacheDesc(4, 16, kv_heads, d, binding.PKV_BF16)
        st = lib.pkv_paged_attention(fake, fake, fake, fake, 1, 1, heads, 1, 16, fake, fake, ctypes.byref(desc),
                                     ctypes.c_float(1.0), fake, None, fake, 1 << 20, None)
        assert st == -3, (heads, kv_heads, d, st)
        st = lib.pkv_paged_attention_no_alloc(fake, fake, fake, fake, 1, 1, heads, 1, 16, fake, fake,
                                              ctypes.byref(desc), ctypes.c_float(1.0), fake, None, None)
        assert st == -3, (heads, kv_heads, d, st)


def test_head_dim_256_is_accepted_on_the_host(lib):
    """head_dim 256 (every row on the CUDA-core rows kernel) gets a workspace
    size; an e4m3 cache at 256 is refused."""
    import ctypes
    desc = binding.CacheDesc(4, 16, 2, 256, binding.PKV_BF16)
    n = lib.pkv_paged_attention_workspace_size(4, 10, 8, ctypes.byref(desc), 512)
    assert n > 0 and n % 256 == 0
    fake = ctypes.c_void_p(256)
    fp8 = binding.CacheDesc(4, 16, 2, 256, binding.PKV_FP8_E4M3)
    scale = ctypes.c_float(1.0)
    st = lib.pkv_paged_attention_fp8(fake, binding.PKV_BF16, fake, fake, fake, 1, 1, 8, 1, 16, fake, fake,
                                     ctypes.byref(fp8), fake, fake, scale, fake, None, fake, 1 << 20, None)
    assert st == -3


def test_no_alloc_rejects_oversized_plans_on_the_host(lib):
    """A tick whose per-row plan does not fit the fixed scratch array is refused
    with PKV_E_WORKSPACE before the array or the device is touched."""
    import ctypes
    fake = ctypes.c_void_p(256)
    desc = binding.CacheDesc(4, 16, 2, 64, binding.PKV_BF16)
    st = lib.pkv_paged_attention_no_alloc(fake, fake, fake, fake, 1, 2_000_000, 8, 1, 16, fake, fake,
                                          ctypes.byref(desc), ctypes.c_float(0.1), fake, None, None)
    assert st == -6
    fp8 = binding.CacheDesc(4, 16, 2, 128, binding.PKV_FP8_E4M3)
    st = lib.pkv_paged_attention_no_alloc(fake, fake, fake, fake, 1, 1, 8, 1, 16, fake, fake,
                                          ctypes.byref(fp8), ctypes.c_float(0.1), fake, None, None)
    assert st == -2    # fp8 caches go through pkv_paged_attention_fp8


@pytest.mark.parametrize("call", ["paged_attention", "paged_attention_no_alloc"])
def test_binding_rejects_host_tensors_and_wide_indices(call):
    """The binding refuses, before any pointer reaches the library, tensors that
    are not on the GPU and index tensors that are not int32 (a CPU pointer or a
    64-bit table read as 32-bit ints would otherwise reach the kernels)."""
    import torch
    fn = getattr(binding, call)
    kc = torch.zeros((4, 16, 2, 64), dtype=torch.bfloat16)
    q = torch.zeros((1, 8, 64), dtype=torch.bfloat16)
    cu = torch.tensor([0, 1], dtype=torch.int32)
    kv = torch.tensor([1], dtype=torch.int32)
    pt = torch.zeros((1, 1), dtype=torch.int32)
    with pytest.raises(ValueError):
        fn(q, cu, kv, pt, kc, kc, 0.125, 16)                     # host tensors
    with pytest.raises(TypeError):
        fn(q, cu.long(), kv, pt, kc, kc, 0.125, 16)              # int64 cu_seqlens_q
    with pytest.raises(TypeError):
        fn(q, cu, kv, pt.long(), kc, kc, 0.125, 16)              # int64 page table
    with pytest.raises(TypeError):
        fn(q.half(), cu, kv, pt, kc, kc, 0.125, 16)              # q dtype != cache dtype

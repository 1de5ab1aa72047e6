"""pkv_paged_attention_no_alloc against the CPU oracle.

The no-allocation call serves callers that cannot allocate device memory (code
inside an allocator's or memory pool's own callbacks, or a plug-in handed only
its input and output tensors): it keeps its scratch (the work plan and the
split-KV partial results) in a fixed array inside the library. Its results are
compared with the oracle, not with the workspace call, because the two may
split a row's keys differently: the fixed array has less room for partial
results, so the planner widens the split until they fit. This file is collected
last so that a failure here stops a `-x` run only after every other test has run.
"""
import numpy as np
import pytest
import torch

from paged_kv_attention_mapping_gb300 import binding
from paged_kv_attention_mapping_gb300 import workloads as W

from tick_helpers import TOL_LSE, TOL_OUT, idx_dev, lists, oracle_tick, poison_unused, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from paged_kv_attention_mapping_gb300 import build
    build.build()
    binding.lib()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    binding.device_status()   # clear
    return d


def _partials_at_min_split(w, chunk):
    """Partial results the plan makes at its smallest split `chunk` keys: every
    row whose visible keys exceed the split writes ceil(keys / chunk) of them per
    KV head (rows of 64 or more in one sequence run on the prefill kernel and
    write none)."""
    n = 0
    for r in w.requests:
        if r.q_len >= 64:
            continue
        for i in range(r.q_len):
            k = r.kv_len - r.q_len + 1 + i
            if k > chunk:
                n += -(-k // chunk) * w.shape.num_kv_heads
    return n


CASES = [
    # long contexts with few sequences: the keys are split, so the scratch holds partials
    ("long-split", dict(seed=31, num_seqs=3, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=256,
                        dtype="bf16", q_lens=(1,), max_kv=20000, min_prefix=12000)),
    # a mixed tick with decode rows and short chunks
    ("mixed", dict(seed=32, num_seqs=6, num_q_heads=32, num_kv_heads=4, head_dim=64, page_size=16,
                   dtype="f16", q_lens=(1, 1, 40), max_kv=3000)),
    # 40-row chunks after 8k-token prefixes: at the smallest split (512 keys at
    # d 64) their partials exceed the room the fixed array leaves (about 8k of
    # 2080 bytes) but not the workspace call's 16384, so only this call widens
    # the split
    ("grow-split", dict(seed=33, num_seqs=4, num_q_heads=32, num_kv_heads=4, head_dim=64, page_size=16,
                        dtype="f16", q_lens=(40,), max_kv=8300, min_prefix=8000)),
    # 128-row and 200-row chunks and a decode row at the Qwen3-4B shape: the
    # tensor-core prefill kernel reads its tile list from the scratch array
    ("prefill-tc", dict(seed=37, num_seqs=4, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=256,
                        dtype="bf16", q_lens=(128, 200, 1), max_kv=1500)),
]


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_no_alloc_matches_oracle_twice(dev, name, kw):
    w = W.random_workload(**kw)
    if name == "grow-split":
        n = _partials_at_min_split(w, 512)
        assert 8100 < n <= 16384, n
    if name == "prefill-tc":
        assert max(r.q_len for r in w.requests) >= 128
    vals = W.host_values(w)
    ql, kl, pg = lists(w)
    packed = binding.pack_tick(ql, kl, pg, w.shape.page_size, w.num_pages)
    kc_h, vc_h = poison_unused(w, packed, vals.k_cache, vals.v_cache)
    ro, rl = oracle_tick(w, vals.q, vals.k_new, vals.v_new, kc_h, vc_h)
    dt = w.shape.dtype
    q = to_dev(vals.q, dt, dev)
    kc, vc = to_dev(kc_h, dt, dev), to_dev(vc_h, dt, dev)
    binding.kv_append(to_dev(vals.k_new, dt, dev), to_dev(vals.v_new, dt, dev),
                      idx_dev(packed["slot_mapping"], dev), kc, vc)
    cu, kv, pt = (idx_dev(packed[k], dev) for k in ("cu_seqlens_q", "kv_lens", "page_tables"))
    for _ in range(2):     # two calls in a row share the same scratch array
        out = torch.full_like(q, float("nan"))
        lse = torch.full((w.total_q, w.shape.num_q_heads), float("nan"), dtype=torch.float32, device=dev)
        binding.paged_attention_no_alloc(q, cu, kv, pt, kc, vc, w.scale, w.max_kv_len, out=out, lse=lse)
        torch.cuda.synchronize()
        assert binding.device_status() == 0
        go = to_host(out).astype(np.float64)
        assert np.isfinite(go).all()
        eo = float(np.abs(go - ro).max())
        el = float(np.abs(lse.cpu().numpy() - rl).max())
        assert eo <= TOL_OUT[dt], eo
        assert el <= TOL_LSE[dt], el


def test_no_alloc_rejects_sizes_beyond_its_scratch(dev):
    import ctypes
    kc = torch.zeros((4, 16, 2, 64), dtype=torch.bfloat16, device=dev)
    T = 2_000_000    # the per-row plan alone would exceed the fixed scratch array
    q = torch.zeros((1, 8, 64), dtype=torch.bfloat16, device=dev)
    desc = binding.cache_desc(kc)
    st = binding.lib().pkv_paged_attention_no_alloc(
        q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), 1, T, 8, 1, 16, kc.data_ptr(), kc.data_ptr(),
        ctypes.byref(desc), ctypes.c_float(0.1), q.data_ptr(), None, binding._stream_ptr())
    assert st == -6    # PKV_E_WORKSPACE, nothing launched
    torch.cuda.synchronize()
    assert binding.device_status() == 0

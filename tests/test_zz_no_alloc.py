"""pkv_paged_attention_no_alloc against pkv_paged_attention.

The no-allocation call serves callers that cannot allocate device memory (code
inside an allocator's or memory pool's own callbacks, or a plug-in handed only
its input and output tensors): it keeps its scratch in a fixed array inside the
library. This file is collected last so that a failure here stops a `-x` run
only after every other test has run.
"""
import numpy as np
import pytest
import torch

from paged_kv_attention_mapping_gb300 import binding
from paged_kv_attention_mapping_gb300 import workloads as W

from tick_helpers import TOL_LSE, TOL_OUT, idx_dev, lists, to_dev

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
    return d


CASES = [
    # long contexts with few sequences: the keys are split, so the scratch holds partials
    ("long-split", dict(seed=31, num_seqs=3, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=256,
                        dtype="bf16", q_lens=(1,), max_kv=20000, min_prefix=12000)),
    # a mixed tick with decode rows and chunks
    ("mixed", dict(seed=32, num_seqs=6, num_q_heads=32, num_kv_heads=4, head_dim=64, page_size=16,
                   dtype="f16", q_lens=(1, 1, 40), max_kv=3000)),
]


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_no_alloc_matches_workspace_call_twice(dev, name, kw):
    w = W.random_workload(**kw)
    vals = W.host_values(w)
    ql, kl, pg = lists(w)
    packed = binding.pack_tick(ql, kl, pg, w.shape.page_size, w.num_pages)
    dt = w.shape.dtype
    q = to_dev(vals.q, dt, dev)
    kc, vc = to_dev(vals.k_cache, dt, dev), to_dev(vals.v_cache, dt, dev)
    binding.kv_append(to_dev(vals.k_new, dt, dev), to_dev(vals.v_new, dt, dev),
                      idx_dev(packed["slot_mapping"], dev), kc, vc)
    cu, kv, pt = (idx_dev(packed[k], dev) for k in ("cu_seqlens_q", "kv_lens", "page_tables"))
    ref_out, ref_lse = binding.paged_attention(q, cu, kv, pt, kc, vc, w.scale, w.max_kv_len)
    torch.cuda.synchronize()
    for _ in range(2):     # two calls in a row share the same scratch array
        out = torch.full_like(q, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        binding.paged_attention_no_alloc(q, cu, kv, pt, kc, vc, w.scale, w.max_kv_len, out=out, lse=lse)
        torch.cuda.synchronize()
        assert binding.device_status() == 0
        eo = float((out.float() - ref_out.float()).abs().max())
        el = float((lse - ref_lse).abs().max())
        assert eo <= TOL_OUT[dt], eo
        assert el <= TOL_LSE[dt], el


def test_no_alloc_rejects_sizes_beyond_its_scratch(dev):
    kc = torch.zeros((4, 16, 2, 64), dtype=torch.bfloat16, device=dev)
    T = 2_000_000    # the per-row plan alone would exceed the fixed scratch array
    q = torch.zeros((1, 8, 64), dtype=torch.bfloat16, device=dev)
    with pytest.raises(binding.PagedKVError) as e:
        binding.lib()
        import ctypes
        desc = binding.cache_desc(kc)
        st = binding.lib().pkv_paged_attention_no_alloc(
            q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), 1, T, 8, 1, 16, kc.data_ptr(), kc.data_ptr(),
            ctypes.byref(desc), ctypes.c_float(0.1), q.data_ptr(), None, binding._stream_ptr())
        binding._check(st, "pkv_paged_attention_no_alloc")
    assert e.value.status == -6

"""A tick captured once in a CUDA graph and replayed with new lengths.

The work plan is computed on the device from cu_seqlens_q / kv_lens, so a
decode-only tick (every row one new token) can be captured once and replayed
every step with the same buffers: the caller rewrites q/k/v, the slot mapping,
kv_lens and page tables in place (Helios blog, "Continuous batching": decode-only
ticks reuse the decode page-table buffers; "CUDA Graphs" in its future-work
list). Each replay is checked against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_mapping_gb300 import binding
from paged_kv_attention_mapping_gb300 import workloads as W

from tick_helpers import TOL_LSE, TOL_OUT, lists

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


@pytest.mark.parametrize("dtype,Hq,Hkv,d,P", [("bf16", 32, 8, 128, 256), ("f16", 32, 4, 64, 16)])
def test_decode_tick_graph_replay_with_growing_lengths(dev, dtype, Hq, Hkv, d, P):
    rng = np.random.default_rng(77)
    B, steps = 6, 3
    w = W.random_workload(91, B, Hq, Hkv, d, P, dtype, (1,), 900, min_prefix=100, headroom=3.0)
    ql, kl, pg = lists(w)
    max_kv = max(kl) + steps
    # give every sequence room for `steps` more tokens (pages come from the pool's spare tail)
    used = {p for r in w.requests for p in r.pages}
    spare = [p for p in range(w.num_pages) if p not in used]
    pages = [list(r.pages) for r in w.requests]
    for b in range(B):
        while len(pages[b]) * P < kl[b] + steps:
            pages[b].append(spare.pop())
    width = max(len(p) for p in pages)
    vals = W.host_values(w)
    kc_h, vc_h = vals.k_cache.copy(), vals.v_cache.copy()
    t = lambda a: W.to_torch(a, dtype, dev)

    # device buffers reused by every replay
    q = torch.empty((B, Hq, d), dtype=W.torch_dtype(dtype), device=dev)
    kn = torch.empty((B, Hkv, d), dtype=q.dtype, device=dev)
    vn = torch.empty_like(kn)
    cu = torch.empty(B + 1, dtype=torch.int32, device=dev)
    kvl = torch.empty(B, dtype=torch.int32, device=dev)
    pt = torch.empty((B, width), dtype=torch.int32, device=dev)
    slots = torch.empty(B, dtype=torch.int64, device=dev)
    kc, vc = t(kc_h), t(vc_h)
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    ws = binding.alloc_workspace(B, B, Hq, kc, max_kv)

    def fill(step):
        lens = [L + step for L in kl]
        pk = oracle.pack_tick([1] * B, lens, pages, P, width)
        qh = W.round_to_dtype(rng.standard_normal((B, Hq, d), dtype=np.float32), dtype)
        kh = W.round_to_dtype(rng.standard_normal((B, Hkv, d), dtype=np.float32), dtype)
        vh = W.round_to_dtype(rng.standard_normal((B, Hkv, d), dtype=np.float32), dtype)
        q.copy_(t(qh)); kn.copy_(t(kh)); vn.copy_(t(vh))
        cu.copy_(torch.from_numpy(pk["cu_seqlens_q"])); kvl.copy_(torch.from_numpy(pk["kv_lens"]))
        pt.copy_(torch.from_numpy(pk["page_tables"])); slots.copy_(torch.from_numpy(pk["slot_mapping"]))
        return pk, qh, kh, vh

    def tick():
        binding.kv_append(kn, vn, slots, kc, vc)
        binding.paged_attention(q, cu, kvl, pt, kc, vc, w.scale, max_kv, out=out, lse=lse, workspace=ws)

    # warm up once outside capture (one-time set-up: attributes, device facts)
    pk, qh, kh, vh = fill(0)
    tick()
    torch.cuda.synchronize()
    kc.copy_(t(kc_h)); vc.copy_(t(vc_h))

    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            tick()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    kc.copy_(t(kc_h)); vc.copy_(t(vc_h))      # capture does not run the kernels

    for step in range(steps):
        pk, qh, kh, vh = fill(step)
        g.replay()
        torch.cuda.synchronize()
        assert binding.device_status() == 0
        kc_h, vc_h = oracle.kv_append(kc_h, vc_h, kh, vh, pk["slot_mapping"])
        ro, rl = oracle.paged_attention(qh, pk["cu_seqlens_q"], pk["kv_lens"], pk["page_tables"], kc_h, vc_h,
                                        w.scale)
        go = out.float().cpu().numpy()
        assert np.abs(go - ro).max() <= TOL_OUT[dtype], step
        assert np.abs(lse.cpu().numpy() - rl).max() <= TOL_LSE[dtype], step

"""Shared test plumbing: run one tick through the C ABI, and the oracle's
answer for the same inputs (computed only from host copies of the inputs)."""
import numpy as np
import torch

import oracle
from paged_kv_attention_mapping_gb300 import binding
from paged_kv_attention_mapping_gb300 import workloads as W

TOL_OUT = {"bf16": 1e-2, "f16": 5e-3, "f32": 1e-4}
TOL_LSE = {"bf16": 1e-3, "f16": 1e-3, "f32": 1e-5}


def lists(w):
    return ([r.q_len for r in w.requests], [r.kv_len for r in w.requests], [r.pages for r in w.requests])


def to_dev(a, dtype, dev):
    return W.to_torch(a, dtype, dev)


def idx_dev(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def poison_unused(w, packed, k_cache, v_cache):
    """NaN in every slot no sequence owns below its kv_len (host arrays)."""
    live = oracle.live_slots(w.num_pages, w.shape.page_size, packed["page_tables"], packed["kv_lens"])
    k_cache = k_cache.copy()
    v_cache = v_cache.copy()
    k_cache[~live] = np.nan
    v_cache[~live] = np.nan
    return k_cache, v_cache


def gpu_tick(w, packed, q, k_new, v_new, k_cache, v_cache, dev, want_lse=True, workspace=None):
    """Append then attend on the device; inputs are torch tensors on `dev`
    (caches are updated in place). Returns (out, lse) tensors."""
    binding.kv_append(k_new, v_new, idx_dev(packed["slot_mapping"], dev), k_cache, v_cache)
    out, lse = binding.paged_attention(q, idx_dev(packed["cu_seqlens_q"], dev), idx_dev(packed["kv_lens"], dev),
                                       idx_dev(packed["page_tables"], dev), k_cache, v_cache, w.scale,
                                       max(w.max_kv_len, 1), want_lse=want_lse, workspace=workspace)
    torch.cuda.synchronize()
    return out, lse


def oracle_tick(w, q, k_new, v_new, k_cache, v_cache, rows=None):
    """Oracle: pack, append, attend — from host arrays only."""
    ql, kl, pg = lists(w)
    p = oracle.pack_tick(ql, kl, pg, w.shape.page_size)
    kc, vc = oracle.kv_append(k_cache, v_cache, k_new, v_new, p["slot_mapping"])
    return oracle.paged_attention(q, p["cu_seqlens_q"], p["kv_lens"], p["page_tables"], kc, vc, w.scale, rows=rows)


def to_host(t):
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy()
    return t.cpu().numpy()


def sub_problem(w, packed, seqs, host_q, host_k_new, host_v_new, host_kc_pages, host_vc_pages):
    """The oracle's inputs for a subset of packed sequences: their pages are
    renumbered 0..n-1 in a compact pool (the oracle is invariant to page ids)."""
    cu = packed["cu_seqlens_q"]
    order = packed["order"]
    page_ids = sorted({p for b in seqs for p in w.requests[order[b]].pages})
    remap = {p: i for i, p in enumerate(page_ids)}
    reqs, rows = [], []
    for b in seqs:
        r = w.requests[order[b]]
        reqs.append(W.Request(r.q_len, r.kv_len, [remap[p] for p in r.pages]))
        rows.extend(range(cu[b], cu[b + 1]))
    sub = W.Workload(w.name + "-sub", w.shape, reqs, len(page_ids), w.scale, w.seed)
    kc = host_kc_pages(page_ids)
    vc = host_vc_pages(page_ids)
    rows = np.array(rows, dtype=np.int64)
    return sub, rows, host_q[rows], host_k_new[rows], host_v_new[rows], kc, vc

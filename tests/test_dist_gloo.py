"""World-size-2 runs of the multi-rank helpers on CPU (gloo).

Each rank runs its own replica of a small tick through the oracle; the
replicas must agree (no rank depends on another), and the timing aggregate is
the max over ranks of the per-rank step time.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import oracle
    from paged_kv_attention_mapping_gb300 import dist as D
    from paged_kv_attention_mapping_gb300 import workloads as W
    r, local, w = D.init("gloo")
    assert (r, w) == (rank, world)
    wl = W.random_workload(5, 3, 8, 2, 16, 4, "f32", (1, 3), 20)
    vals = W.host_values(wl)
    ql = [x.q_len for x in wl.requests]
    kl = [x.kv_len for x in wl.requests]
    pg = [x.pages for x in wl.requests]
    p = oracle.pack_tick(ql, kl, pg, 4)
    kc, vc = oracle.kv_append(vals.k_cache, vals.v_cache, vals.k_new, vals.v_new, p["slot_mapping"])
    out, lse = oracle.paged_attention(vals.q, p["cu_seqlens_q"], p["kv_lens"], p["page_tables"], kc, vc, wl.scale)
    # replicas agree
    t = torch.from_numpy(out.reshape(-1).copy())
    g = [torch.zeros_like(t) for _ in range(world)]
    dist.all_gather(g, t)
    assert all(torch.equal(g[0], x) for x in g)
    # step-time aggregate: max over ranks
    ms = [1.5 + rank, 0.25 * (rank + 1)]
    mx = D.max_over_ranks(ms)
    assert mx == [1.5 + world - 1, 0.25 * world]
    tok = D.aggregate_tokens_per_s(wl.total_q, mx[0], w)
    assert abs(tok - world * wl.total_q / (mx[0] / 1000.0)) < 1e-6
    D.barrier()
    np.save(os.path.join(out_dir, f"rank{rank}.npy"), np.array([tok]))
    dist.destroy_process_group()


def test_two_rank_replicas_and_aggregate(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    vals = [float(np.load(tmp_path / f"rank{r}.npy")[0]) for r in range(world)]
    assert vals[0] == vals[1]


def test_single_rank_is_identity():
    from paged_kv_attention_mapping_gb300 import dist as D
    assert D.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]
    assert D.aggregate_tokens_per_s(100, 2.0, 1) == 50000.0

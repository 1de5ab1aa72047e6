"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Append is compared bit for bit; attention within the tolerances of the
workload description (max abs error 1e-2 bf16, 5e-3 fp16, 1e-4 fp32 on
unit-normal inputs; lse 1e-3, 1e-5 for fp32). Every slot that no sequence owns
below its kv_len is NaN-poisoned in the small cases, so a read of a slot the
row may not see shows up as a NaN.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_mapping_gb300 import binding
from paged_kv_attention_mapping_gb300 import workloads as W

from tick_helpers import (TOL_LSE, TOL_OUT, gpu_tick, idx_dev, lists, oracle_tick, poison_unused, sub_problem,
                          to_dev, to_host)

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
    binding.device_status()  # clear
    return d


def run_and_compare(w, dev, poison=True, want_lse=True):
    vals = W.host_values(w)
    ql, kl, pg = lists(w)
    packed = binding.pack_tick(ql, kl, pg, w.shape.page_size, w.num_pages)
    kc_h, vc_h = vals.k_cache, vals.v_cache
    if poison:
        # NaN everywhere the tick will not own after the append
        kc_h, vc_h = poison_unused(w, packed, kc_h, vc_h)
    dt = w.shape.dtype
    kc, vc = to_dev(kc_h, dt, dev), to_dev(vc_h, dt, dev)
    out, lse = gpu_tick(w, packed, to_dev(vals.q, dt, dev), to_dev(vals.k_new, dt, dev), to_dev(vals.v_new, dt, dev),
                        kc, vc, dev, want_lse=want_lse)
    assert binding.device_status() == 0
    ro, rl = oracle_tick(w, vals.q, vals.k_new, vals.v_new, kc_h, vc_h)
    go = to_host(out).astype(np.float64)
    assert np.isfinite(go).all()
    eo = float(np.abs(go - ro).max())
    assert eo <= TOL_OUT[dt], eo
    if want_lse:
        el = float(np.abs(lse.cpu().numpy() - rl).max())
        assert el <= TOL_LSE[dt], el
    return out, lse


# ---------------------------------------------------------------------------
# append

@pytest.mark.parametrize("name,dtype", [("tiny_decode", "f32"), ("tiny_decode", "bf16"),
                                        ("tinyllama_decode", "f16")])
def test_append_bit_exact(dev, name, dtype):
    w = W.make_workload(name, dtype)
    vals = W.host_values(w)
    ql, kl, pg = lists(w)
    packed = binding.pack_tick(ql, kl, pg, w.shape.page_size, w.num_pages)
    kc, vc = to_dev(vals.k_cache, dtype, dev), to_dev(vals.v_cache, dtype, dev)
    binding.kv_append(to_dev(vals.k_new, dtype, dev), to_dev(vals.v_new, dtype, dev),
                      idx_dev(packed["slot_mapping"], dev), kc, vc)
    torch.cuda.synchronize()
    k2, v2 = oracle.kv_append(vals.k_cache, vals.v_cache, vals.k_new, vals.v_new, packed["slot_mapping"])
    want_k = W.to_torch(k2, dtype)
    want_v = W.to_torch(v2, dtype)
    assert torch.equal(kc.cpu().view(torch.int16 if dtype != "f32" else torch.int32),
                       want_k.view(torch.int16 if dtype != "f32" else torch.int32))
    assert torch.equal(vc.cpu().view(torch.int16 if dtype != "f32" else torch.int32),
                       want_v.view(torch.int16 if dtype != "f32" else torch.int32))


def test_append_skips_negative_and_flags_out_of_pool_slots(dev):
    N, P, H, D = 4, 16, 2, 64
    kc = torch.zeros((N, P, H, D), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    k = torch.randn((3, H, D), device=dev).to(torch.bfloat16)
    v = torch.randn((3, H, D), device=dev).to(torch.bfloat16)
    binding.kv_append(k, v, torch.tensor([5, -1, N * P + 3], dtype=torch.int64, device=dev), kc, vc)
    assert binding.device_status() == binding.DEV_BAD_SLOT
    flat = kc.view(N * P, H, D)
    assert torch.equal(flat[5], k[0])
    assert int((flat != 0).any(dim=(1, 2)).sum()) == 1
    assert binding.device_status() == 0


# ---------------------------------------------------------------------------
# attention, small cases against the whole oracle

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_tiny_decode(dev, dtype):
    run_and_compare(W.make_workload("tiny_decode", dtype), dev)


RAGGED = [
    # seed, B, Hq, Hkv, d, P, dtype, q_lens, max_kv
    (1, 8, 8, 2, 64, 16, "bf16", (1,), 300),
    (2, 6, 32, 8, 128, 256, "bf16", (1, 2, 17), 300),
    (3, 5, 32, 4, 64, 16, "f16", (1, 2, 17, 130), 300),
    (4, 4, 8, 8, 128, 16, "f32", (1, 2, 17), 200),
    (5, 3, 16, 2, 128, 256, "bf16", (130,), 300),
    (6, 8, 4, 1, 64, 16, "f16", (1, 17), 300),
    (7, 2, 32, 2, 64, 256, "bf16", (130, 1), 700),
    (8, 7, 16, 16, 64, 16, "f32", (1,), 300),
    (9, 3, 8, 8, 128, 256, "bf16", (130, 1), 400),      # g = 1: single-query-tile prefill kernel
    (10, 4, 16, 4, 64, 32, "f16", (200, 1, 70), 600),   # page 32 < tile: several pages per TMA tile
    (13, 3, 32, 2, 128, 256, "bf16", (130, 1), 500),    # g = 16: eight head pairs per KV head in the prefill kernel
    (14, 3, 8, 4, 64, 64, "f16", (150, 1), 400),        # g = 2, page 64: one page per decode tile
    (15, 3, 16, 8, 128, 128, "bf16", (140, 1), 600),    # page 128 = one prefill KV tile per page
    (16, 5, 64, 8, 128, 256, "bf16", (1, 2, 17), 2500),  # g = 8 at d 128: warp states merged in a K/V stage; splits
    (17, 4, 16, 1, 64, 16, "f32", (1, 3), 1200),        # g = 16 fp32: the same merge on the fp32 path; splits
    # many short chunks: each prefill CTA runs several 1-2 step work tiles back to
    # back through its 2-entry tile ring (Q reloads, V-tail fixes, tile hand-offs)
    (18, 24, 16, 4, 128, 256, "bf16", (64, 128, 129, 200), 600),
    (19, 24, 32, 4, 64, 16, "f16", (64, 100, 150, 1), 400),
    # groups of 3, 5, 6 and 7 q heads per KV head (the Qwen2.5 family has 5, 6
    # and 7): decode rows on the TMA kernel, chunks on the two-tile prefill
    # kernel (an odd group's last head as a solo tile), splits
    (51, 5, 24, 8, 128, 256, "bf16", (1, 2, 130), 2600),  # g = 3
    (52, 5, 40, 8, 128, 128, "bf16", (1, 150), 700),      # g = 5
    (53, 5, 12, 2, 64, 16, "f16", (1, 3, 100), 900),      # g = 6, two query tiles per CTA
    (54, 4, 28, 4, 128, 64, "f16", (1, 130), 2300),       # g = 7
    (55, 6, 21, 7, 64, 32, "f32", (1, 5), 1300),          # g = 3 over an fp32 cache
    # head_dim 256: every row (decode and chunk) on the TMA decode kernel over
    # 16-bit caches and the CUDA-core rows kernel over fp32 caches, rows past
    # 2048 keys split and merged by the combine kernel
    (61, 4, 16, 4, 256, 16, "bf16", (1, 2, 70), 2600),    # g = 4, splits
    (62, 3, 8, 8, 256, 64, "f16", (1, 130), 900),         # g = 1, a chunk of 130 rows
    (63, 3, 8, 1, 256, 32, "f32", (1, 3), 2500),          # g = 8 over an fp32 cache, splits
    (64, 2, 32, 2, 256, 256, "bf16", (1, 5), 4300),       # g = 16, two splits per row
]


@pytest.mark.parametrize("case", RAGGED, ids=[f"s{c[0]}-{c[6]}-d{c[4]}-P{c[5]}-g{c[2] // c[3]}" for c in RAGGED])
def test_ragged(dev, case):
    seed, B, Hq, Hkv, d, P, dt, ql, mk = case
    w = W.random_workload(seed, B, Hq, Hkv, d, P, dt, ql, mk)
    run_and_compare(w, dev)


# Page sizes that neither divide nor are multiples of the 64-key TMA tile (and
# pages smaller than one 16-byte-aligned box) run on the CUDA-core row kernel
# for every row, decode or chunk: it reads each key through the page table with
# vector loads and serves all g query heads of a KV head from each load.
ROWS_KERNEL = [
    # seed, B, Hq, Hkv, d, P, dtype, q_lens, max_kv
    (40, 6, 32, 8, 128, 24, "bf16", (1, 2, 17), 3000),   # rows past 2048 keys are split
    (41, 5, 32, 4, 64, 48, "f16", (1, 17, 70), 1500),    # a 70-row chunk row by row; 512-key splits
    (42, 4, 16, 16, 64, 24, "f32", (1, 3), 1200),        # g = 1
    (43, 3, 16, 1, 128, 96, "f32", (1, 5), 2500),        # g = 16 at d 128
    (44, 4, 8, 4, 128, 48, "bf16", (1, 130), 800),       # g = 2, a 130-row chunk
    (45, 5, 8, 2, 64, 4, "f16", (1, 9), 300),            # 4-token pages
    (46, 4, 16, 2, 64, 24, "bf16", (1,), 5000),          # g = 8, long decode rows split ten ways
    (47, 4, 24, 4, 128, 48, "f16", (1, 70), 1200),       # g = 6
    (48, 4, 15, 3, 64, 24, "f32", (1, 3), 900),          # g = 5
]


@pytest.mark.parametrize("case", ROWS_KERNEL,
                         ids=[f"s{c[0]}-{c[6]}-d{c[4]}-P{c[5]}-g{c[2] // c[3]}" for c in ROWS_KERNEL])
def test_rows_kernel_page_sizes(dev, case):
    seed, B, Hq, Hkv, d, P, dt, ql, mk = case
    w = W.random_workload(seed, B, Hq, Hkv, d, P, dt, ql, mk)
    binding.set_kernel_timing(True)
    try:
        run_and_compare(w, dev)
    finally:
        launched = binding.kernel_times()
        binding.set_kernel_timing(False)
    assert "rows" in launched and "decode" not in launched and "prefill_tc" not in launched, launched


def _sweep_cases(n=24, seed=20261202):
    """Seeded draws over the whole accepted shape space: group sizes 1-8 and 16,
    head_dim 64/128, pages from the TMA kernels' sizes and the rows kernel's,
    every dtype, decode rows, short chunks and chunks for the prefill kernels."""
    rng = np.random.default_rng(seed)
    out = []
    for k in range(n):
        g = int(rng.choice([1, 2, 3, 4, 5, 6, 7, 8, 16]))
        hkv = int(rng.choice([1, 2, 4, 8])) if g < 16 else int(rng.choice([1, 2]))
        d = int(rng.choice([64, 128]))
        P = int(rng.choice([8, 16, 32, 64, 128, 256, 24, 40]))
        dt = str(rng.choice(["f32", "f16", "bf16"]))
        ql = tuple(int(x) for x in rng.choice([1, 1, 2, 7, 64, 100, 140], size=3))
        B = int(rng.integers(1, 7))
        mk = int(rng.choice([200, 700, 2500]))
        out.append((1000 + k, B, g * hkv, hkv, d, P, dt, ql, mk))
    return out


@pytest.mark.parametrize("case", _sweep_cases(),
                         ids=[f"w{c[0]}-{c[6]}-d{c[4]}-P{c[5]}-g{c[2] // c[3]}" for c in _sweep_cases()])
def test_seeded_shape_sweep(dev, case):
    seed, B, Hq, Hkv, d, P, dt, ql, mk = case
    w = W.random_workload(seed, B, Hq, Hkv, d, P, dt, ql, mk)
    run_and_compare(w, dev)


def test_chunk_among_idle_sequences_takes_row_path(dev):
    """A tick with no more rows than sequences skips the tensor-core prefill
    kernel; a 64-row chunk whose 63 companions are idle is then attended row by
    row, with the same results as the oracle."""
    rng = np.random.default_rng(31)
    P, B = 16, 64
    shape = W.TickShape(8, 2, 64, P, "bf16")
    reqs, pool = [], list(rng.permutation(400))
    for b in range(B):
        q = 64 if b == 17 else 0
        L = 64 + int(rng.integers(1, 120)) if q else int(rng.integers(1, 40))
        n = (L + P - 1) // P
        reqs.append(W.Request(q, L, [int(x) for x in pool[:n]]))
        pool = pool[n:]
    w = W.Workload("idle_chunk", shape, reqs, 400, 0.125, 31)
    assert w.total_q == B
    run_and_compare(w, dev)


def test_without_lse(dev):
    w = W.random_workload(11, 4, 8, 2, 64, 16, "bf16", (1, 17), 120)
    run_and_compare(w, dev, want_lse=False)


def test_idle_sequences_and_empty_tick(dev):
    w = W.random_workload(12, 6, 8, 2, 64, 16, "bf16", (0, 1, 0, 5), 100)
    run_and_compare(w, dev)
    # a tick with no rows at all is a no-op that returns OK
    kc = torch.zeros((2, 16, 2, 64), dtype=torch.bfloat16, device=dev)
    q = torch.zeros((0, 8, 64), dtype=torch.bfloat16, device=dev)
    ws = binding.alloc_workspace(1, 0, 8, kc, 16)
    binding.paged_attention(q, torch.tensor([0, 0], dtype=torch.int32, device=dev),
                            torch.tensor([5], dtype=torch.int32, device=dev),
                            torch.zeros((1, 1), dtype=torch.int32, device=dev), kc, kc, 0.125, 16, workspace=ws)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f16", 64), ("f32", 64)])
def test_one_key_context_returns_v(dev, dtype, d):
    """A context of one key (the token just appended): out is that token's V
    exactly, lse is scale * q.k (the softmax of one score is 1)."""
    B, Hq, Hkv, P = 5, 16, 4, 16
    rng = np.random.default_rng(21)
    q = W.round_to_dtype(rng.standard_normal((B, Hq, d), dtype=np.float32), dtype)
    k = W.round_to_dtype(rng.standard_normal((B, Hkv, d), dtype=np.float32), dtype)
    v = W.round_to_dtype(rng.standard_normal((B, Hkv, d), dtype=np.float32), dtype)
    pages = [[b] for b in range(B)]
    packed = binding.pack_tick([1] * B, [1] * B, pages, P, B)
    kc = torch.full((B, P, Hkv, d), float("nan"), dtype=W.torch_dtype(dtype), device=dev)
    vc = kc.clone()
    scale = 1.0 / np.sqrt(d)
    binding.kv_append(to_dev(k, dtype, dev), to_dev(v, dtype, dev), idx_dev(packed["slot_mapping"], dev), kc, vc)
    out, lse = binding.paged_attention(to_dev(q, dtype, dev), idx_dev(packed["cu_seqlens_q"], dev),
                                       idx_dev(packed["kv_lens"], dev), idx_dev(packed["page_tables"], dev), kc,
                                       vc, scale, 1)
    torch.cuda.synchronize()
    g = Hq // Hkv
    want = np.repeat(np.asarray(v, np.float32), g, axis=1)        # q head h reads KV head h // g
    assert np.array_equal(to_host(out).astype(np.float32), want)
    qk = np.einsum("bhd,bhd->bh", np.asarray(q, np.float64), np.repeat(np.asarray(k, np.float64), g, axis=1))
    assert np.abs(lse.cpu().numpy() - scale * qk).max() <= TOL_LSE[dtype]


def test_back_to_back_ticks_without_sync(dev):
    """Two ticks (chunks and decode rows) issued one after the other on one
    stream with no host synchronisation, then the first again into the same
    buffers: both match the oracle and the repeat is bit-identical."""
    ws_ = []
    res = []
    for seed in (31, 32):
        w = W.random_workload(seed, 6, 16, 4, 128, 256, "bf16", (1, 1, 150), 900)
        vals = W.host_values(w)
        ql, kl, pg = lists(w)
        packed = binding.pack_tick(ql, kl, pg, w.shape.page_size, w.num_pages)
        kc, vc = to_dev(vals.k_cache, "bf16", dev), to_dev(vals.v_cache, "bf16", dev)
        args = (to_dev(vals.q, "bf16", dev), idx_dev(packed["cu_seqlens_q"], dev), idx_dev(packed["kv_lens"], dev),
                idx_dev(packed["page_tables"], dev), kc, vc, w.scale, w.max_kv_len)
        ws_.append((w, vals, packed, args, to_dev(vals.k_new, "bf16", dev), to_dev(vals.v_new, "bf16", dev)))
    for w, vals, packed, args, kn, vn in ws_:
        binding.kv_append(kn, vn, idx_dev(packed["slot_mapping"], dev), args[4], args[5])
        res.append(binding.paged_attention(*args))
    w, vals, packed, args, kn, vn = ws_[0]
    again = binding.paged_attention(*args)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    for (w, vals, packed, args, kn, vn), (out, lse) in zip(ws_, res):
        ro, rl = oracle_tick(w, vals.q, vals.k_new, vals.v_new, vals.k_cache, vals.v_cache)
        assert np.abs(to_host(out).astype(np.float64) - ro).max() <= TOL_OUT["bf16"]
        assert np.abs(lse.cpu().numpy() - rl).max() <= TOL_LSE["bf16"]
    assert torch.equal(again[0], res[0][0]) and torch.equal(again[1], res[0][1])


def test_packing_does_not_change_a_row(dev):
    """A decode row gives bit-identical output alone and inside a mixed tick."""
    w = W.random_workload(13, 6, 32, 8, 128, 256, "bf16", (1, 1, 40), 3000)
    vals = W.host_values(w)
    ql, kl, pg = lists(w)
    packed = binding.pack_tick(ql, kl, pg, w.shape.page_size, w.num_pages)
    dt = w.shape.dtype
    kc, vc = to_dev(vals.k_cache, dt, dev), to_dev(vals.v_cache, dt, dev)
    out, lse = gpu_tick(w, packed, to_dev(vals.q, dt, dev), to_dev(vals.k_new, dt, dev),
                        to_dev(vals.v_new, dt, dev), kc, vc, dev)
    cu = packed["cu_seqlens_q"]
    order = packed["order"]
    for b in range(len(order)):
        if cu[b + 1] - cu[b] != 1:
            continue
        r = w.requests[order[b]]
        one = W.Workload("one", w.shape, [r], w.num_pages, w.scale, w.seed)
        p1 = binding.pack_tick([1], [r.kv_len], [r.pages], w.shape.page_size, w.num_pages)
        q1 = to_dev(vals.q, dt, dev)[cu[b]:cu[b] + 1].contiguous()
        o1, l1 = binding.paged_attention(q1, idx_dev(p1["cu_seqlens_q"], dev), idx_dev(p1["kv_lens"], dev),
                                         idx_dev(p1["page_tables"], dev), kc, vc, w.scale, w.max_kv_len)
        torch.cuda.synchronize()
        assert torch.equal(o1[0], out[cu[b]]) and torch.equal(l1[0], lse[cu[b]])


def test_bad_page_id_sets_status_and_skips_row(dev):
    w = W.random_workload(14, 3, 8, 2, 64, 16, "bf16", (1,), 100)
    vals = W.host_values(w)
    ql, kl, pg = lists(w)
    packed = binding.pack_tick(ql, kl, pg, w.shape.page_size, w.num_pages)
    tables = packed["page_tables"].copy()
    tables[1, 0] = w.num_pages + 7          # outside the pool
    dt = w.shape.dtype
    kc, vc = to_dev(vals.k_cache, dt, dev), to_dev(vals.v_cache, dt, dev)
    out = torch.full((w.total_q, 8, 64), 7.0, dtype=torch.bfloat16, device=dev)
    binding.paged_attention(to_dev(vals.q, dt, dev), idx_dev(packed["cu_seqlens_q"], dev),
                            idx_dev(packed["kv_lens"], dev), idx_dev(tables, dev), kc, vc, w.scale, w.max_kv_len,
                            out=out)
    assert binding.device_status() & binding.DEV_BAD_PAGE
    assert bool((out[1].float() == 7.0).all())           # the bad row is left unwritten
    assert not bool((out[0].float() == 7.0).all())
    assert binding.device_status() == 0


def test_bad_lengths_set_status(dev):
    kc = torch.zeros((4, 16, 2, 64), dtype=torch.bfloat16, device=dev)
    q = torch.zeros((3, 8, 64), dtype=torch.bfloat16, device=dev)
    binding.paged_attention(q, torch.tensor([0, 1, 3], dtype=torch.int32, device=dev),
                            torch.tensor([40, 1], dtype=torch.int32, device=dev),   # 40 > 2 pages * 16; 1 < 2
                            torch.zeros((2, 2), dtype=torch.int32, device=dev), kc, kc, 0.125, 64)
    assert binding.device_status() & binding.DEV_BAD_LENGTHS



def _attend_after_append(w, dev, kv_lens=None, cu=None):
    """Caches appended on the host by the oracle; attention alone on the device
    with (possibly altered) lengths, into an output pre-filled with 7.0."""
    vals = W.host_values(w)
    ql, kl, pg = lists(w)
    packed = binding.pack_tick(ql, kl, pg, w.shape.page_size, w.num_pages)
    kc_h, vc_h = oracle.kv_append(vals.k_cache, vals.v_cache, vals.k_new, vals.v_new, packed["slot_mapping"])
    dt = w.shape.dtype
    out = torch.full((w.total_q, w.shape.num_q_heads, w.shape.head_dim), 7.0, dtype=W.torch_dtype(dt), device=dev)
    binding.paged_attention(to_dev(vals.q, dt, dev), idx_dev(packed["cu_seqlens_q"] if cu is None else cu, dev),
                            idx_dev(packed["kv_lens"] if kv_lens is None else kv_lens, dev),
                            idx_dev(packed["page_tables"], dev), to_dev(kc_h, dt, dev), to_dev(vc_h, dt, dev),
                            w.scale, w.max_kv_len, out=out)
    torch.cuda.synchronize()
    return vals, packed, kc_h, vc_h, out


def test_bad_sequence_skipped_others_exact(dev):
    # long contexts so that the good decode rows are split; sequence 1 too long
    w = W.random_workload(21, 4, 32, 8, 128, 256, "bf16", (1, 17, 130), 9500)
    ql, kl, pg = lists(w)
    packed = binding.pack_tick(ql, kl, pg, w.shape.page_size, w.num_pages)
    bad_kv = packed["kv_lens"].copy()
    bad_kv[1] = w.max_kv_len + 1
    vals, packed, kc_h, vc_h, out = _attend_after_append(w, dev, kv_lens=bad_kv)
    assert binding.device_status() & binding.DEV_BAD_LENGTHS
    cu = packed["cu_seqlens_q"]
    bad_rows = list(range(cu[1], cu[2]))
    good_rows = [r for r in range(w.total_q) if r not in bad_rows]
    assert bool((out[bad_rows].float() == 7.0).all())
    ro, _ = oracle.paged_attention(vals.q, cu, packed["kv_lens"], packed["page_tables"], kc_h, vc_h, w.scale,
                                   rows=good_rows)
    eo = float(np.abs(to_host(out[good_rows]).astype(np.float64) - ro).max())
    assert eo <= TOL_OUT["bf16"], eo


def test_decreasing_cu_seqlens_skips_every_row(dev):
    w = W.random_workload(22, 3, 8, 2, 64, 16, "bf16", (1, 17), 300)
    ql, kl, pg = lists(w)
    packed = binding.pack_tick(ql, kl, pg, w.shape.page_size, w.num_pages)
    cu = packed["cu_seqlens_q"].copy()
    assert cu[1] < cu[2]
    cu[1], cu[2] = cu[2], cu[1]              # one q_len < 0: the rows no longer partition
    _, _, _, _, out = _attend_after_append(w, dev, cu=cu)
    assert binding.device_status() & binding.DEV_BAD_LENGTHS
    assert bool((out.float() == 7.0).all())
    assert binding.device_status() == 0

def test_host_checks_reject_without_launch(dev):
    kc = torch.zeros((4, 16, 2, 64), dtype=torch.bfloat16, device=dev)
    q = torch.zeros((1, 24, 64), dtype=torch.bfloat16, device=dev)   # Hq=24, Hkv=2 -> g=12 unsupported
    with pytest.raises(binding.PagedKVError) as e:
        binding.paged_attention(q, torch.tensor([0, 1], dtype=torch.int32, device=dev),
                                torch.tensor([1], dtype=torch.int32, device=dev),
                                torch.zeros((1, 1), dtype=torch.int32, device=dev), kc, kc, 0.1, 16,
                                workspace=torch.empty(1 << 20, dtype=torch.uint8, device=dev))
    assert e.value.status == -3
    q = torch.zeros((1, 8, 64), dtype=torch.bfloat16, device=dev)
    with pytest.raises(binding.PagedKVError) as e:
        binding.paged_attention(q, torch.tensor([0, 1], dtype=torch.int32, device=dev),
                                torch.tensor([1], dtype=torch.int32, device=dev),
                                torch.zeros((1, 1), dtype=torch.int32, device=dev), kc, kc, 0.1, 16,
                                workspace=torch.empty(256, dtype=torch.uint8, device=dev))
    assert e.value.status == -6


# ---------------------------------------------------------------------------
# the named workloads at full size, on sampled sequences and rows

def full_size_check(name, dev, n_decode=12, chunk_rows=48, seed=0):
    w = W.make_workload(name) if isinstance(name, str) else name
    dt = w.shape.dtype
    ql, kl, pg = lists(w)
    packed = binding.pack_tick(ql, kl, pg, w.shape.page_size, w.num_pages)
    ref = oracle.pack_tick(ql, kl, pg, w.shape.page_size)
    for k in ref:
        assert np.array_equal(packed[k], ref[k]), k
    vals = W.device_values(w, dev)
    # host copies of what the oracle needs, taken before the append
    host_q, host_k, host_v = (to_host(vals[k]) for k in ("q", "k_new", "v_new"))
    kc, vc = vals["k_cache"], vals["v_cache"]
    cu = packed["cu_seqlens_q"]
    B = len(packed["order"])
    rng = np.random.default_rng(seed)
    dec = [b for b in range(B) if cu[b + 1] - cu[b] == 1]
    chunks = [b for b in range(B) if cu[b + 1] - cu[b] > 1]
    seqs = sorted(set(rng.choice(dec, size=min(n_decode, len(dec)), replace=False).tolist()) | set(chunks))
    # always include the longest decode sequence
    if dec:
        seqs = sorted(set(seqs) | {max(dec, key=lambda b: packed["kv_lens"][b])})
    page_ids_cache = {}

    def pages_of(cache):
        def get(ids):
            t = cache[torch.tensor(ids, device=dev, dtype=torch.long)]
            return to_host(t)
        return get

    sub, rows, q_s, k_s, v_s, kc_s, vc_s = sub_problem(w, packed, seqs, host_q, host_k, host_v,
                                                       pages_of(kc), pages_of(vc))
    kc_before, vc_before = kc.clone(), vc.clone()
    out, lse = gpu_tick(w, packed, vals["q"], vals["k_new"], vals["v_new"], kc, vc, dev)
    assert binding.device_status() == 0
    # the append over the whole tick, bit for bit: every slot of the slot
    # mapping holds its token's K and V row, every other slot is unchanged
    bits = torch.int32 if dt == "f32" else torch.int16
    s_ = w.shape
    slots_t = torch.from_numpy(packed["slot_mapping"]).to(dev)
    for cache, before, new in ((kc, kc_before, vals["k_new"]), (vc, vc_before, vals["v_new"])):
        flat = cache.view(-1, s_.num_kv_heads, s_.head_dim).view(bits)
        flat_before = before.view(-1, s_.num_kv_heads, s_.head_dim).view(bits)
        assert torch.equal(flat[slots_t], new.view(bits))
        keep = torch.ones(flat.shape[0], dtype=torch.bool, device=dev)
        keep[slots_t] = False
        assert torch.equal(flat[keep], flat_before[keep])
    del kc_before, vc_before
    # rows to check: all decode rows of the sample, and a spread of chunk rows
    sub_cu = oracle.pack_tick(*lists(sub), sub.shape.page_size)["cu_seqlens_q"]
    check = []
    for i in range(len(seqs)):
        n = sub_cu[i + 1] - sub_cu[i]
        if n <= 1:
            check += list(range(sub_cu[i], sub_cu[i + 1]))
        else:
            pick = set(rng.choice(n, size=min(chunk_rows, n), replace=False).tolist()) | {0, n - 1, min(127, n - 1),
                                                                                         min(128, n - 1)}
            check += [sub_cu[i] + j for j in sorted(pick)]
    ro, rl = oracle_tick(sub, q_s, k_s, v_s, kc_s, vc_s, rows=check)
    go = to_host(out)[rows[check]].astype(np.float64)
    gl = lse.cpu().numpy()[rows[check]]
    eo = float(np.abs(go - ro).max())
    el = float(np.abs(gl - rl).max())
    assert np.isfinite(go).all()
    assert eo <= TOL_OUT[dt], eo
    assert el <= TOL_LSE[dt], el
    return out, lse


@pytest.mark.parametrize("name", ["tinyllama_decode", "qwen3_decode", "mixed_tick", "shared_prefix_long",
                                  "mixed_decode_heavy", "mixed_many_chunks"])
def test_full_size_workload(dev, name):
    full_size_check(name, dev)


@pytest.mark.parametrize("hq,hkv", [(28, 4), (24, 8)])
def test_full_size_mixed_tick_odd_groups(dev, hq, hkv):
    """The mixed tick's requests (96 decodes, two 2048-row chunks) with groups of
    7 and 3 q heads per KV head: the chunks run on the two-tile prefill kernel
    with each group's last head as a solo tile, beside the decode rows."""
    w0 = W.make_workload("mixed_tick")
    s0 = w0.shape
    shape = W.TickShape(hq, hkv, s0.head_dim, s0.page_size, s0.dtype)
    w = W.Workload(f"mixed_tick_{hq}x{hkv}", shape, w0.requests, w0.num_pages, w0.scale, w0.seed + hq)
    binding.set_kernel_timing(True)
    binding.kernel_times()
    try:
        full_size_check(w, dev)
        launched = binding.kernel_times()
    finally:
        binding.set_kernel_timing(False)
    assert "prefill_tc" in launched and "decode" in launched, launched


def test_more_than_256_prefill_tiles(dev):
    """300 sequences of one 64-row chunk each (prefixes of 0-256 keys, head_dim 64,
    pages of 16, group 4): 300 (sequence, q tile) pairs, more than the plan ranks
    directly, so its counting sort orders the prefill kernel's tiles. Every chunk
    is in the checked sub-problem; a few rows of each are compared."""
    w = W.random_workload(71, 300, 8, 2, 64, 16, "bf16", (64,), 320)
    assert sum(r.q_len for r in w.requests) == 300 * 64
    full_size_check(w, dev, n_decode=0, chunk_rows=6, seed=3)

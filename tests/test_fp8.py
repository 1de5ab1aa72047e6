"""FP8 (e4m3) KV cache: the oracle codec pinned to the format's fixed points,
and (GPU) the quantising append and attention over fp8 pages."""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8 as F
from paged_kv_attention_mapping_gb300 import binding
from paged_kv_attention_mapping_gb300 import workloads as W

from tick_helpers import TOL_LSE, TOL_OUT, idx_dev, lists, to_dev


def test_table_fixed_points():
    t = F.e4m3_table()
    assert t[0x7E] == 448.0 and np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert t[0x08] == 2.0 ** -6 and t[0x01] == 2.0 ** -9 and t[0x38] == 1.0 and t[0x80] == 0.0
    assert np.all(np.diff(t[:127]) > 0)
    assert np.array_equal(t[128:255], -t[:127])


def test_quantize_rounding_and_saturation():
    one = np.ones(1, dtype=np.float32)
    q = lambda v: int(F.quantize(np.array([[v]], dtype=np.float32), one)[0, 0])
    assert q(1.0) == 0x38 and q(-1.0) == 0xB8
    assert q(1.0 + 1 / 16) == 0x38          # halfway 1 .. 1.125: even mantissa (1)
    assert q(1.0 + 3 / 16) == 0x3A          # halfway 1.125 .. 1.25: even mantissa (1.25)
    assert q(1000.0) == 0x7E and q(-1e9) == 0xFE and q(460.0) == 0x7E
    assert q(2.0 ** -10) == 0x00            # halfway 0 .. 2^-9: even (0)
    assert q(3 * 2.0 ** -11) == 0x01
    t = F.e4m3_table()
    vals = t[np.isfinite(t)].astype(np.float32)
    codes = F.quantize(vals[None, :], one)[0]
    assert np.array_equal(t[codes], vals.astype(np.float64))   # representable values are fixed points


def test_quotient_is_rounded_to_float32_before_the_e4m3_rounding():
    # x / s is 34.000000353 exactly but 34.0 (the midpoint of 32 and 36) in
    # float32; ties-to-even then gives 32 (code 0x60). Dividing in float64
    # would give 36 (0x61).
    x = np.array([0x42B7F396], dtype=np.uint32).view(np.float32)
    s = np.array([0x402D217E], dtype=np.uint32).view(np.float32)
    assert float(np.float64(x[0]) / np.float64(s[0])) > 34.0
    assert int(F.quantize(x.reshape(1, 1), s)[0, 0]) == 0x60


def test_dequantize_scales_per_head():
    codes = np.array([[[0x38, 0x40], [0x38, 0xB8]]], dtype=np.uint8)   # [1, 2 heads, 2]
    v = F.dequantize(codes, np.array([0.5, 3.0]))
    assert np.array_equal(v, [[[0.5, 1.0], [3.0, -3.0]]])


# ---------------------------------------------------------------------------
# host-side checks of the fp8 entry points (no device work happens before them)

def _desc(N, P, H, D, dtype):
    return binding.CacheDesc(N, P, H, D, dtype)


def test_fp8_entry_points_reject_wrong_types_on_the_host():
    import ctypes
    L = binding.lib()
    fp8 = _desc(4, 16, 2, 128, binding.PKV_FP8_E4M3)
    bf16 = _desc(4, 16, 2, 128, binding.PKV_BF16)
    fake = ctypes.c_void_p(256)
    # the 16-bit entry points refuse an fp8 cache
    assert L.pkv_kv_append(fake, fake, fake, 1, fake, fake, ctypes.byref(fp8), None) == -2
    assert L.pkv_paged_attention(fake, fake, fake, fake, 1, 1, 4, 1, 16, fake, fake, ctypes.byref(fp8),
                                 ctypes.c_float(1.0), fake, None, fake, 1 << 20, None) == -2
    assert L.pkv_rope_kv_append(fake, fake, fake, fake, fake, 8, fake, 1, 4, fake, fake, ctypes.byref(fp8), fake,
                                None) == -2
    # the fp8 entry points refuse a 16-bit cache, an fp32 query and head_dim 64
    assert L.pkv_paged_attention_fp8(fake, binding.PKV_BF16, fake, fake, fake, 1, 1, 4, 1, 16, fake, fake,
                                     ctypes.byref(bf16), fake, fake, ctypes.c_float(1.0), fake, None, fake, 1 << 20,
                                     None) == -2
    assert L.pkv_paged_attention_fp8(fake, binding.PKV_F32, fake, fake, fake, 1, 1, 4, 1, 16, fake, fake,
                                     ctypes.byref(fp8), fake, fake, ctypes.c_float(1.0), fake, None, fake, 1 << 20,
                                     None) == -2
    d64 = _desc(4, 16, 2, 64, binding.PKV_FP8_E4M3)
    assert L.pkv_paged_attention_fp8(fake, binding.PKV_BF16, fake, fake, fake, 1, 1, 4, 1, 16, fake, fake,
                                     ctypes.byref(d64), fake, fake, ctypes.c_float(1.0), fake, None, fake, 1 << 20,
                                     None) == -3
    assert L.pkv_kv_append_quant(fake, fake, binding.PKV_BF16, fake, 1, fake, fake, ctypes.byref(bf16), fake, fake,
                                 None) == -2
    d40 = _desc(4, 16, 2, 40, binding.PKV_FP8_E4M3)
    assert L.pkv_kv_append_quant(fake, fake, binding.PKV_BF16, fake, 1, fake, fake, ctypes.byref(d40), fake, fake,
                                 None) == -3
    # missing scales
    assert L.pkv_paged_attention_fp8(fake, binding.PKV_BF16, fake, fake, fake, 1, 1, 4, 1, 16, fake, fake,
                                     ctypes.byref(fp8), None, fake, ctypes.c_float(1.0), fake, None, fake, 1 << 20,
                                     None) == -1
    assert L.pkv_kv_append_quant(fake, fake, binding.PKV_BF16, fake, 1, fake, fake, ctypes.byref(fp8), fake, None,
                                 None) == -1


# ---------------------------------------------------------------------------
# GPU: the quantising append (bit-exact) and attention over fp8 pages

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


def _hard_values(rng, shape, dtype):
    """Unit normals times 40 (some saturate at small scales), with exact ties
    of the e4m3 grid, tiny values and signed zeros mixed in."""
    x = rng.standard_normal(shape, dtype=np.float32) * 40.0
    flat = x.reshape(-1)
    n = flat.size
    ties = np.array([1.0625, 1.1875, -1.0625, 2 ** -10, -3 * 2 ** -11, 0.0, -0.0, 448.0, 464.0, -1e6],
                    dtype=np.float32)
    pick = rng.choice(n, size=n // 8, replace=False)
    flat[pick] = ties[rng.integers(0, len(ties), size=len(pick))]
    return W.round_to_dtype(x, dtype)


@pytest.mark.gpu
@pytest.mark.parametrize("src,D", [("bf16", 128), ("f16", 128), ("f32", 128), ("bf16", 64)])
def test_append_quant_bit_exact(dev, src, D):
    rng = np.random.default_rng(5)
    N, P, H, T = 12, 16, 4, 57
    slots = rng.permutation(N * P)[:T].astype(np.int64)
    slots[[3, 20]] = -1
    k = _hard_values(rng, (T, H, D), src)
    v = _hard_values(rng, (T, H, D), src)
    # scale 1 keeps the ties on the grid; the others move them off it
    ks = np.array([1.0, 0.05, 0.3, 7.0], dtype=np.float32)
    vs = np.array([0.2, 1.0, 3.0, 0.011], dtype=np.float32)
    init = rng.integers(0, 256, size=(N, P, H, D), dtype=np.uint8)
    kc = torch.from_numpy(init.copy()).to(dev)
    vc = torch.from_numpy(init.copy()).to(dev)
    binding.kv_append_quant(to_dev(k, src, dev), to_dev(v, src, dev), idx_dev(slots, dev), kc, vc,
                            torch.from_numpy(ks).to(dev), torch.from_numpy(vs).to(dev))
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    src32 = lambda a: np.asarray(a, dtype=np.float32)
    want_k, want_v = oracle.kv_append(init, init, F.quantize(src32(k), ks), F.quantize(src32(v), vs), slots)
    assert np.array_equal(kc.cpu().numpy(), want_k)
    assert np.array_equal(vc.cpu().numpy(), want_v)


def _fp8_tick(w, dev, qdt, seed=0, poison=True):
    """Quantise a workload's cache on the host (oracle codec), run append +
    attention on the device, and compare with the oracle over the dequantised
    pages (fp64)."""
    s = w.shape
    vals = W.host_values(w)
    ql, kl, pg = lists(w)
    packed = binding.pack_tick(ql, kl, pg, s.page_size, w.num_pages)
    rng = np.random.default_rng([w.seed, seed])
    ks = (np.abs(vals.k_cache).max(axis=(0, 1, 3)) / 448.0 * rng.uniform(0.5, 2.0, s.num_kv_heads)).astype(np.float32)
    vs = (np.abs(vals.v_cache).max(axis=(0, 1, 3)) / 448.0 * rng.uniform(0.5, 2.0, s.num_kv_heads)).astype(np.float32)
    kc_codes = F.quantize(vals.k_cache, ks)
    vc_codes = F.quantize(vals.v_cache, vs)
    if poison:
        live = oracle.live_slots(w.num_pages, s.page_size, packed["page_tables"], packed["kv_lens"])
        kc_codes[~live] = 0x7F   # NaN code
        vc_codes[~live] = 0xFF
    kc = torch.from_numpy(kc_codes.copy()).to(dev)
    vc = torch.from_numpy(vc_codes.copy()).to(dev)
    ks_d, vs_d = torch.from_numpy(ks).to(dev), torch.from_numpy(vs).to(dev)
    qh = W.round_to_dtype(vals.q, qdt)
    kn = W.round_to_dtype(vals.k_new, qdt)
    vn = W.round_to_dtype(vals.v_new, qdt)
    # device: quantising append, then attention
    binding.kv_append_quant(to_dev(kn, qdt, dev), to_dev(vn, qdt, dev), idx_dev(packed["slot_mapping"], dev), kc, vc,
                            ks_d, vs_d)
    out, lse = binding.paged_attention_fp8(to_dev(qh, qdt, dev), idx_dev(packed["cu_seqlens_q"], dev),
                                           idx_dev(packed["kv_lens"], dev), idx_dev(packed["page_tables"], dev),
                                           kc, vc, ks_d, vs_d, w.scale, max(w.max_kv_len, 1))
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    # oracle: the same codes, appended in packed order, then attention over their values
    ok, ov = oracle.kv_append(kc_codes, vc_codes, F.quantize(np.asarray(kn, np.float32), ks),
                              F.quantize(np.asarray(vn, np.float32), vs), packed["slot_mapping"])
    assert np.array_equal(kc.cpu().numpy(), ok) and np.array_equal(vc.cpu().numpy(), ov)
    # q rows in packed order, as the device got them
    ro, rl = oracle.paged_attention(np.asarray(qh, np.float64), packed["cu_seqlens_q"], packed["kv_lens"],
                                    packed["page_tables"], F.dequantize(ok, ks), F.dequantize(ov, vs), w.scale)
    go = out.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(go).all()
    eo = float(np.abs(go - ro).max())
    el = float(np.abs(lse.cpu().numpy() - rl).max())
    assert eo <= TOL_OUT[qdt], eo
    assert el <= TOL_LSE[qdt], el
    return eo, el


@pytest.mark.gpu
@pytest.mark.parametrize("qdt,Hq,Hkv,P,q_lens,max_kv", [
    ("bf16", 32, 8, 16, (1,), 700),              # decode rows, GQA 4, small pages
    ("f16", 32, 8, 256, (1,), 3000),             # long rows split over several items
    ("bf16", 16, 1, 16, (1, 1, 3, 17, 80), 900), # GQA 16 with chunk rows (causal, row kernel)
    ("bf16", 8, 8, 64, (1, 2, 9), 400),          # no grouping (G = 1)
    ("f16", 16, 8, 32, (1, 33), 520),            # G = 2
    ("bf16", 32, 8, 64, (1, 1, 5), 9500),        # rows split over several items, combined in the kernel
    # chunks of 64 rows or more: the tensor-core prefill kernel with the codes
    # widened to fp16 in shared memory (causal inside the chunk, ragged tails)
    ("bf16", 32, 8, 256, (1, 130, 200), 1500),   # GQA 4, one page per KV tile, bf16 q narrowed to fp16
    ("f16", 32, 8, 16, (1, 70, 129), 700),       # 16-token pages: eight pages per KV tile
    ("bf16", 16, 8, 64, (2, 150), 600),          # G = 2, two pages per KV tile
    ("f16", 32, 2, 128, (1, 96, 300), 900),      # G = 16
    ("bf16", 24, 8, 256, (1, 130, 200), 1500),   # G = 3: each group's last head runs as a solo tile
    ("f16", 8, 8, 128, (1, 100), 600),           # G = 1: every tile solo
])
def test_attention_over_fp8_pages(dev, qdt, Hq, Hkv, P, q_lens, max_kv):
    seed = 300 + Hq + P + (max(q_lens) if max(q_lens) >= 64 else 0)   # chunk cases drawn apart from the rest
    w = W.random_workload(seed, 9, Hq, Hkv, 128, P, qdt, q_lens, max_kv)
    _fp8_tick(w, dev, qdt)


@pytest.mark.gpu
def test_fp8_decode_full_size_sampled(dev):
    """qwen3_decode shapes (128 sequences, 512-8192 context, page 256, GQA 4)
    with the cache quantised on the device, attention checked on sampled rows."""
    w = W.make_workload("qwen3_decode")
    s = w.shape
    vals = W.device_values(w, dev)
    ks = torch.full((s.num_kv_heads,), 4.0 / 448.0, device=dev)
    vs = torch.full((s.num_kv_heads,), 4.5 / 448.0, device=dev)
    N, P = w.num_pages, s.page_size
    kc = torch.empty((N, P, s.num_kv_heads, s.head_dim), dtype=torch.uint8, device=dev)
    vc = torch.empty_like(kc)
    # quantise the whole pool with the library's own append (slot i <- row i)
    all_slots = torch.arange(N * P, dtype=torch.int64, device=dev)
    binding.kv_append_quant(vals["k_cache"].reshape(N * P, s.num_kv_heads, s.head_dim),
                            vals["v_cache"].reshape(N * P, s.num_kv_heads, s.head_dim), all_slots, kc, vc, ks, vs)
    ql, kl, pg = lists(w)
    packed = binding.pack_tick(ql, kl, pg, P, N)
    binding.kv_append_quant(vals["k_new"], vals["v_new"], idx_dev(packed["slot_mapping"], dev), kc, vc, ks, vs)
    out, lse = binding.paged_attention_fp8(vals["q"], idx_dev(packed["cu_seqlens_q"], dev),
                                           idx_dev(packed["kv_lens"], dev), idx_dev(packed["page_tables"], dev),
                                           kc, vc, ks, vs, w.scale, w.max_kv_len)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    ks_h, vs_h = ks.cpu().numpy(), vs.cpu().numpy()
    rows = np.random.default_rng(3).choice(w.total_q, size=6, replace=False)
    cu, kvl, pt = packed["cu_seqlens_q"], packed["kv_lens"], packed["page_tables"]
    qh = vals["q"].float().cpu().numpy().astype(np.float64)
    for r in rows:
        b = int(np.searchsorted(cu, r, side="right") - 1)
        L = int(kvl[b])
        npg = -(-L // P)
        pages = torch.from_numpy(pt[b, :npg].astype(np.int64)).to(dev)
        kseq = F.dequantize(kc[pages].cpu().numpy(), ks_h).reshape(-1, s.num_kv_heads,
                                                                                            s.head_dim)[:L]
        vseq = F.dequantize(vc[pages].cpu().numpy(), vs_h).reshape(-1, s.num_kv_heads,
                                                                                            s.head_dim)[:L]
        ro, rl = oracle.attend_row(qh[r], kseq, vseq, L, w.scale)   # a decode row sees all L keys
        assert np.abs(out[r].float().cpu().numpy() - ro).max() <= TOL_OUT["bf16"]
        assert np.abs(lse[r].cpu().numpy() - rl).max() <= TOL_LSE["bf16"]


def _quantised_pool(w, dev, ks, vs):
    """The workload's synthetic pool drawn on the device and quantised by the
    library's own append (slot i <- row i), plus the tick's packing."""
    s = w.shape
    vals = W.device_values(w, dev)
    N, P = w.num_pages, s.page_size
    kc = torch.empty((N, P, s.num_kv_heads, s.head_dim), dtype=torch.uint8, device=dev)
    vc = torch.empty_like(kc)
    all_slots = torch.arange(N * P, dtype=torch.int64, device=dev)
    binding.kv_append_quant(vals["k_cache"].reshape(N * P, s.num_kv_heads, s.head_dim),
                            vals["v_cache"].reshape(N * P, s.num_kv_heads, s.head_dim), all_slots, kc, vc, ks, vs)
    ql, kl, pg = lists(w)
    packed = binding.pack_tick(ql, kl, pg, P, N)
    return vals, kc, vc, packed


@pytest.mark.gpu
def test_fp8_mixed_tick_full_size_sampled(dev):
    """The mixed tick (96 decode rows, two 2048-row chunks after prefixes of 0
    and 3072, Qwen3-4B shape, page 256) over an e4m3 cache: the chunks run on
    the tensor-core prefill kernel with widened tiles. Sampled rows of every
    kind against the oracle over the dequantised pages."""
    w = W.make_workload("mixed_tick")
    s = w.shape
    ks = torch.full((s.num_kv_heads,), 4.0 / 448.0, device=dev)
    vs = torch.full((s.num_kv_heads,), 4.5 / 448.0, device=dev)
    vals, kc, vc, packed = _quantised_pool(w, dev, ks, vs)
    binding.kv_append_quant(vals["k_new"], vals["v_new"], idx_dev(packed["slot_mapping"], dev), kc, vc, ks, vs)
    binding.set_kernel_timing(True)
    try:
        out, lse = binding.paged_attention_fp8(vals["q"], idx_dev(packed["cu_seqlens_q"], dev),
                                               idx_dev(packed["kv_lens"], dev), idx_dev(packed["page_tables"], dev),
                                               kc, vc, ks, vs, w.scale, w.max_kv_len)
        torch.cuda.synchronize()
    finally:
        launched = binding.kernel_times()
        binding.set_kernel_timing(False)
    assert "prefill_tc" in launched, launched
    assert binding.device_status() == 0
    ks_h, vs_h = ks.cpu().numpy(), vs.cpu().numpy()
    cu, kvl, pt = packed["cu_seqlens_q"], packed["kv_lens"], packed["page_tables"]
    qh = vals["q"].float().cpu().numpy().astype(np.float64)
    rng = np.random.default_rng(5)
    B = len(kvl)
    chunks = [b for b in range(B) if cu[b + 1] - cu[b] > 1]
    rows = list(rng.choice(int(cu[len(kvl) - len(chunks)]), size=6, replace=False))
    for b in chunks:
        n = int(cu[b + 1] - cu[b])
        pick = set(rng.choice(n, size=24, replace=False).tolist()) | {0, 127, 128, n - 1}
        rows += [int(cu[b]) + j for j in sorted(pick)]
    cache = {}
    for r in rows:
        b = int(np.searchsorted(cu, r, side="right") - 1)
        L = int(kvl[b])
        if b not in cache:
            npg = -(-L // s.page_size)
            pages = torch.from_numpy(pt[b, :npg].astype(np.int64)).to(dev)
            cache[b] = (F.dequantize(kc[pages].cpu().numpy(), ks_h).reshape(-1, s.num_kv_heads, s.head_dim)[:L],
                        F.dequantize(vc[pages].cpu().numpy(), vs_h).reshape(-1, s.num_kv_heads, s.head_dim)[:L])
        kseq, vseq = cache[b]
        n_visible = L - int(cu[b + 1] - cu[b]) + (r - int(cu[b])) + 1   # bottom-right causal rule
        ro, rl = oracle.attend_row(qh[r], kseq, vseq, n_visible, w.scale)
        assert np.abs(out[r].float().cpu().numpy() - ro).max() <= TOL_OUT["bf16"], r
        assert np.abs(lse[r].cpu().numpy() - rl).max() <= TOL_LSE["bf16"], r


@pytest.mark.gpu
def test_append_quant_divides_in_float32(dev):
    """The float32 quotient case of the codec pin, through the kernel."""
    H, D = 2, 128
    x = np.array([0x42B7F396], dtype=np.uint32).view(np.float32)[0]
    s = np.array([0x402D217E], dtype=np.uint32).view(np.float32)[0]
    k = np.full((1, H, D), x, dtype=np.float32)
    scales = np.array([s, s], dtype=np.float32)
    kc = torch.zeros((1, 16, H, D), dtype=torch.uint8, device=dev)
    vc = torch.zeros_like(kc)
    binding.kv_append_quant(torch.from_numpy(k).to(dev), torch.from_numpy(k).to(dev),
                            torch.zeros(1, dtype=torch.int64, device=dev), kc, vc,
                            torch.from_numpy(scales).to(dev), torch.from_numpy(scales).to(dev))
    torch.cuda.synchronize()
    assert bool((kc[0, 0] == 0x60).all()) and bool((vc[0, 0] == 0x60).all())
    assert int(kc[0, 1:].sum()) == 0

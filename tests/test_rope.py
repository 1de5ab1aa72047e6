"""RoPE: the oracle pinned to closed forms, the library's cos/sin table against
the oracle's angles, and (GPU) the fused rotate-and-append kernel."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle.rope import apply_rope, positions_of_tick, rope_angles
from paged_kv_attention_mapping_gb300 import binding
from paged_kv_attention_mapping_gb300 import workloads as W

from tick_helpers import TOL_LSE, TOL_OUT, idx_dev, lists, to_dev


# ---------------------------------------------------------------------------
# oracle pins (CPU)

def test_two_dims_rotate_by_the_position():
    x = np.array([[[1.0, 0.0]], [[0.3, -2.0]]])
    y = apply_rope(x, [0, 5], 10000.0)
    assert np.allclose(y[0], x[0], atol=0)                                   # position 0: identity
    c, s = math.cos(5.0), math.sin(5.0)                                     # d = 2: frequency 1
    assert np.allclose(y[1, 0], [0.3 * c + 2.0 * s, -2.0 * c + 0.3 * s], atol=1e-15)


def test_pairs_are_i_and_i_plus_half():
    d, p, base = 8, 3, 100.0
    for i in range(d // 2):
        e = np.zeros((1, 1, d))
        e[0, 0, i] = 1.0
        y = apply_rope(e, [p], base)[0, 0]
        a = p * base ** (-2.0 * i / d)
        want = np.zeros(d)
        want[i], want[i + d // 2] = math.cos(a), math.sin(a)
        assert np.allclose(y, want, atol=1e-15)


def test_norm_kept_and_scores_depend_on_distance_only():
    rng = np.random.default_rng(1)
    q, k = rng.standard_normal((1, 1, 16)), rng.standard_normal((1, 1, 16))
    assert abs(np.linalg.norm(apply_rope(q, [7], 1e4)) - np.linalg.norm(q)) < 1e-12
    dots = [float(apply_rope(q, [p + 9], 1e4).ravel() @ apply_rope(k, [p], 1e4).ravel()) for p in (0, 5, 40)]
    assert max(dots) - min(dots) < 1e-12


def test_positions_of_tick():
    assert list(positions_of_tick([0, 1, 4, 4], [10, 7, 3])) == [9, 4, 5, 6]


def test_library_positions_match_the_oracle(lib):
    for name in W.WORKLOADS:
        w = W.make_workload(name)
        p = oracle.pack_tick(*lists(w), w.shape.page_size)
        assert np.array_equal(binding.tick_positions(p["cu_seqlens_q"], p["kv_lens"]),
                              positions_of_tick(p["cu_seqlens_q"], p["kv_lens"]))


# ---------------------------------------------------------------------------
# library table (CPU)

@pytest.fixture(scope="module")
def lib():
    from paged_kv_attention_mapping_gb300 import build
    build.build()
    return binding.lib()


@pytest.mark.parametrize("base,d", [(10000.0, 64), (1e6, 128)])
def test_library_table_matches_the_angles(lib, base, d):
    tab = binding.rope_table(base, d, 9000)
    a = rope_angles(base, d, np.arange(9000))
    assert np.abs(tab[..., 0] - np.cos(a)).max() < 1e-7
    assert np.abs(tab[..., 1] - np.sin(a)).max() < 1e-7
    with pytest.raises(binding.PagedKVError):
        binding.rope_table(1.0, d, 10)


# ---------------------------------------------------------------------------
# GPU: fused rotate-and-append, and attention after it

def ulp_err(got, want, x, dtype):
    """|got - want| over (one dtype spacing at |want| + one at the row's largest
    input): fp32 rotation error is relative to the operands, final rounding to
    the result."""
    mant = {"bf16": 7, "f16": 10, "f32": 23}[dtype]
    sp = lambda m: np.exp2(np.floor(np.log2(np.maximum(m, 2.0 ** -14))) - mant)
    rowmax = np.abs(np.asarray(x, dtype=np.float64)).max(axis=-1, keepdims=True)
    return float((np.abs(got - want) / (sp(np.abs(want)) + sp(rowmax))).max())


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,Hq,Hkv,d,P", [("bf16", 32, 8, 128, 256), ("f16", 32, 4, 64, 16), ("f32", 8, 2, 64, 16)])
def test_rope_append_then_attention(dtype, Hq, Hkv, d, P):
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    binding.lib()
    dev = torch.device("cuda:0")
    base = 1e6 if d == 128 else 1e4
    w = W.random_workload(61, 5, Hq, Hkv, d, P, dtype, (1, 1, 150), 700)
    vals = W.host_values(w)
    ql, kl, pg = lists(w)
    pk = binding.pack_tick(ql, kl, pg, P, w.num_pages)
    pos = positions_of_tick(pk["cu_seqlens_q"], pk["kv_lens"])
    tab = torch.from_numpy(binding.rope_table(base, d, max(kl) + 1)).to(dev)
    kc, vc = to_dev(vals.k_cache, dtype, dev), to_dev(vals.v_cache, dtype, dev)
    q = to_dev(vals.q, dtype, dev)
    q_rot = binding.rope_kv_append(q, to_dev(vals.k_new, dtype, dev), to_dev(vals.v_new, dtype, dev),
                                   idx_dev(pos, dev), tab, idx_dev(pk["slot_mapping"], dev), kc, vc)
    out, lse = binding.paged_attention(q_rot, idx_dev(pk["cu_seqlens_q"], dev), idx_dev(pk["kv_lens"], dev),
                                       idx_dev(pk["page_tables"], dev), kc, vc, w.scale, w.max_kv_len)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    # oracle: rotate (float64), round to the dtype, append, attend
    q_ref = W.round_to_dtype(apply_rope(vals.q, pos, base).astype(np.float32), dtype)
    k_ref = W.round_to_dtype(apply_rope(vals.k_new, pos, base).astype(np.float32), dtype)
    to_np = lambda t: t.float().cpu().numpy()
    assert ulp_err(to_np(q_rot), apply_rope(vals.q, pos, base), vals.q, dtype) <= 1.0
    kc2, vc2 = oracle.kv_append(vals.k_cache, vals.v_cache, k_ref, vals.v_new, pk["slot_mapping"])
    flat = lambda c: c.reshape(-1, Hkv, d)
    slots = pk["slot_mapping"]
    got_k = to_np(kc).reshape(-1, Hkv, d)[slots]
    assert ulp_err(got_k, apply_rope(vals.k_new, pos, base), vals.k_new, dtype) <= 1.0
    assert np.array_equal(to_np(vc).reshape(-1, Hkv, d)[slots], flat(vc2)[slots].astype(np.float32))
    # attention on the GPU's own rotated values equals the oracle on them
    ro, rl = oracle.paged_attention(to_np(q_rot).astype(vals.q.dtype) if dtype != "bf16" else to_np(q_rot),
                                    pk["cu_seqlens_q"], pk["kv_lens"], pk["page_tables"],
                                    to_np(kc).astype(vals.k_cache.dtype) if dtype != "bf16" else to_np(kc),
                                    to_np(vc).astype(vals.v_cache.dtype) if dtype != "bf16" else to_np(vc), w.scale)
    assert np.abs(to_np(out) - ro).max() <= TOL_OUT[dtype]
    assert np.abs(lse.cpu().numpy() - rl).max() <= TOL_LSE[dtype]


@pytest.mark.gpu
def test_rope_append_flags_bad_positions():
    binding.lib()
    dev = torch.device("cuda:0")
    kc = torch.zeros((2, 16, 2, 64), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    q = torch.ones((2, 4, 64), dtype=torch.bfloat16, device=dev)
    k = torch.ones((2, 2, 64), dtype=torch.bfloat16, device=dev)
    tab = torch.from_numpy(binding.rope_table(1e4, 64, 8)).to(dev)
    binding.rope_kv_append(q, k, k, torch.tensor([3, 8], dtype=torch.int32, device=dev), tab,
                           torch.tensor([0, 1], dtype=torch.int64, device=dev), kc, vc)
    assert binding.device_status() & binding.DEV_BAD_POSITION
    assert binding.device_status() == 0

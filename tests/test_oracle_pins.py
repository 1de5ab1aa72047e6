"""Pins of the CPU oracle to facts outside itself (no GPU).

Each pin is chosen so that a plausible slip in the oracle (a dropped scale, a
wrong GQA head map, a causal offset off by one, a transposed page index, a
missing normalisation) fails at least one of them; the mutation tests at the
end plant such slips in the oracle and check that they are caught.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import oracle.core as OPA
from paged_kv_attention_mapping_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# test-local builders (independent of the oracle's own index arithmetic)

def build_paged(dense_k, dense_v, page_size, rng, extra_pages=3):
    """Scatter per-sequence dense K/V [L, Hkv, d] into a random page pool by
    walking the positions one by one; returns (k_pool, v_pool, page lists)."""
    need = [-(-k.shape[0] // page_size) for k in dense_k]
    n_pages = sum(need) + extra_pages
    perm = list(rng.permutation(n_pages))
    Hkv, d = dense_k[0].shape[1:]
    kp = rng.standard_normal((n_pages, page_size, Hkv, d))
    vp = rng.standard_normal((n_pages, page_size, Hkv, d))
    pages = []
    for k, v, n in zip(dense_k, dense_v, need):
        mine = [int(perm.pop()) for _ in range(n)]
        pages.append(mine)
        pos = 0
        for page in mine:
            for off in range(page_size):
                if pos < k.shape[0]:
                    kp[page, off] = k[pos]
                    vp[page, off] = v[pos]
                pos += 1
    return kp, vp, pages


def table(pages, width=None):
    width = width or max(len(p) for p in pages)
    t = np.full((len(pages), width), -1, dtype=np.int32)
    for b, p in enumerate(pages):
        t[b, :len(p)] = p
    return t


def sdpa_dense(q, K, V, scale):
    """torch SDPA in float64 on dense K/V with KV heads repeated per group and
    an explicit bottom-right causal mask; returns (out [Lq,Hq,d], lse [Lq,Hq])."""
    Lq, Hq, d = q.shape
    L, Hkv, _ = K.shape
    g = Hq // Hkv
    qt = torch.from_numpy(q).double().permute(1, 0, 2)
    kt = torch.from_numpy(K).double().repeat_interleave(g, dim=1).permute(1, 0, 2)
    vt = torch.from_numpy(V).double().repeat_interleave(g, dim=1).permute(1, 0, 2)
    i = torch.arange(Lq)[:, None]
    j = torch.arange(L)[None, :]
    mask = j <= (L - Lq + i)
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    scores = (qt @ kt.transpose(-1, -2)) * scale
    lse = torch.logsumexp(scores.masked_fill(~mask, float("-inf")), dim=-1)
    return out.permute(1, 0, 2).numpy(), lse.permute(1, 0).numpy()


def random_case(seed, B=3, Hq=8, Hkv=2, d=16, P=4, q_lens=(1, 1, 5), prefix=(6, 0, 7)):
    rng = np.random.default_rng(seed)
    dk, dv, qs = [], [], []
    for b in range(B):
        L = prefix[b] + q_lens[b]
        dk.append(rng.standard_normal((L, Hkv, d)))
        dv.append(rng.standard_normal((L, Hkv, d)))
        qs.append(rng.standard_normal((q_lens[b], Hq, d)))
    kp, vp, pages = build_paged(dk, dv, P, rng)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    kv = np.array([p + q for p, q in zip(prefix, q_lens)], dtype=np.int32)
    return dict(dk=dk, dv=dv, qs=qs, q=np.concatenate(qs), kp=kp, vp=vp, pages=pages,
                cu=cu, kv=kv, pt=table(pages), scale=1.0 / math.sqrt(d))


def max_err_vs_sdpa(c):
    out, lse = oracle.paged_attention(c["q"], c["cu"], c["kv"], c["pt"], c["kp"], c["vp"], c["scale"])
    e_o = e_l = 0.0
    for b in range(len(c["qs"])):
        r0, r1 = c["cu"][b], c["cu"][b + 1]
        ro, rl = sdpa_dense(c["qs"][b], c["dk"][b], c["dv"][b], c["scale"])
        e_o = max(e_o, float(np.abs(out[r0:r1] - ro).max()))
        e_l = max(e_l, float(np.abs(lse[r0:r1] - rl).max()))
    return e_o, e_l


# ---------------------------------------------------------------------------
# pin 1: a library special case (dense unpaged attention)

@pytest.mark.parametrize("seed,Hq,Hkv,P,q_lens,prefix", [
    (0, 8, 2, 4, (1, 1, 5), (6, 0, 7)),
    (1, 4, 4, 3, (3, 1, 2), (0, 9, 4)),
    (2, 6, 1, 16, (1, 17, 1), (40, 20, 0)),
    (3, 8, 4, 5, (9, 1, 1), (11, 3, 1)),
])
def test_matches_dense_sdpa(seed, Hq, Hkv, P, q_lens, prefix):
    c = random_case(seed, Hq=Hq, Hkv=Hkv, P=P, q_lens=q_lens, prefix=prefix)
    e_o, e_l = max_err_vs_sdpa(c)
    assert e_o < 1e-12 and e_l < 1e-12, (e_o, e_l)


# ---------------------------------------------------------------------------
# pin 2: brute force on tiny inputs with Python floats

def brute(qs, dk, dv, scale):
    res_o, res_l = [], []
    for b in range(len(qs)):
        Lq, Hq, d = qs[b].shape
        L, Hkv, _ = dk[b].shape
        for i in range(Lq):
            row_o, row_l = [], []
            for h in range(Hq):
                kvh = h * Hkv // Hq
                s = []
                for j in range(L - Lq + i + 1):
                    s.append(scale * sum(float(qs[b][i, h, c]) * float(dk[b][j, kvh, c]) for c in range(d)))
                m = max(s)
                tot = sum(math.exp(x - m) for x in s)
                lse = m + math.log(tot)
                o = [sum(math.exp(s[j] - lse) * float(dv[b][j, kvh, c]) for j in range(len(s))) for c in range(d)]
                row_o.append(o)
                row_l.append(lse)
            res_o.append(row_o)
            res_l.append(row_l)
    return np.array(res_o), np.array(res_l)


@pytest.mark.parametrize("seed", range(4))
def test_matches_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    B = 3
    q_lens = [int(x) for x in rng.integers(1, 4, size=B)]
    prefix = [int(x) for x in rng.integers(0, 3, size=B)]
    c = random_case(100 + seed, B=B, Hq=4, Hkv=2, d=4, P=2, q_lens=q_lens, prefix=prefix)
    out, lse = oracle.paged_attention(c["q"], c["cu"], c["kv"], c["pt"], c["kp"], c["vp"], c["scale"])
    bo, bl = brute(c["qs"], c["dk"], c["dv"], c["scale"])
    assert np.abs(out - bo).max() < 1e-12
    assert np.abs(lse - bl).max() < 1e-12


# ---------------------------------------------------------------------------
# pin 3: one-key context returns V exactly

def test_one_key_context_returns_v():
    rng = np.random.default_rng(7)
    k = rng.standard_normal((1, 2, 8))
    v = rng.standard_normal((1, 2, 8))
    q = rng.standard_normal((1, 4, 8))
    kp, vp, pages = build_paged([k], [v], 4, rng)
    out, lse = oracle.paged_attention(q, np.array([0, 1]), np.array([1]), table(pages), kp, vp, 0.37)
    assert np.array_equal(out[0], np.repeat(v[0], 2, axis=0))
    for h in range(4):
        assert abs(lse[0, h] - 0.37 * float(np.dot(q[0, h], k[0, h // 2]))) < 1e-14


# ---------------------------------------------------------------------------
# pin 4: closed forms

def test_zero_scale_gives_mean_of_visible_values():
    c = random_case(11, q_lens=(1, 6, 3), prefix=(5, 0, 4))
    out, lse = oracle.paged_attention(c["q"], c["cu"], c["kv"], c["pt"], c["kp"], c["vp"], 0.0)
    for b in range(3):
        Lq = c["cu"][b + 1] - c["cu"][b]
        L = int(c["kv"][b])
        for i in range(Lq):
            n = L - Lq + i + 1          # keys the row sees
            want = np.repeat(c["dv"][b][:n].mean(axis=0), 4, axis=0)
            assert np.abs(out[c["cu"][b] + i] - want).max() < 1e-13
            assert np.abs(lse[c["cu"][b] + i] - math.log(n)).max() < 1e-13


def test_identical_keys_and_identical_values():
    rng = np.random.default_rng(12)
    L, Hkv, d, Hq = 9, 2, 8, 4
    k = np.repeat(rng.standard_normal((1, Hkv, d)), L, axis=0)
    v = rng.standard_normal((L, Hkv, d))
    q = rng.standard_normal((3, Hq, d))
    kp, vp, pages = build_paged([k], [v], 4, rng)
    out, lse = oracle.paged_attention(q, np.array([0, 3]), np.array([L]), table(pages), kp, vp, 0.5)
    for i in range(3):
        n = L - 3 + i + 1
        for h in range(Hq):
            s = 0.5 * float(np.dot(q[i, h], k[0, h // 2]))
            assert abs(lse[i, h] - (s + math.log(n))) < 1e-12
            assert np.abs(out[i, h] - v[:n, h // 2].mean(axis=0)).max() < 1e-12
    c_val = rng.standard_normal((1, Hkv, d))
    v2 = np.repeat(c_val, L, axis=0)
    k2 = rng.standard_normal((L, Hkv, d))
    kp, vp, pages = build_paged([k2], [v2], 4, rng)
    out, _ = oracle.paged_attention(q, np.array([0, 3]), np.array([L]), table(pages), kp, vp, 0.5)
    for h in range(Hq):
        assert np.abs(out[:, h] - c_val[0, h // 2]).max() < 1e-12


def test_future_keys_do_not_matter():
    """Changing K/V at positions a row may not see leaves that row unchanged."""
    c = random_case(13, q_lens=(1, 6, 1), prefix=(3, 2, 8))
    out, lse = oracle.paged_attention(c["q"], c["cu"], c["kv"], c["pt"], c["kp"], c["vp"], c["scale"])
    b, Lq, L = 1, 6, 8
    for i in range(Lq):
        dk = [x.copy() for x in c["dk"]]
        dv = [x.copy() for x in c["dv"]]
        dk[b][L - Lq + i + 1:] += 5.0
        dv[b][L - Lq + i + 1:] -= 3.0
        rng = np.random.default_rng(0)
        kp, vp, pages = build_paged(dk, dv, 4, rng)
        o2, l2 = oracle.paged_attention(c["q"], c["cu"], c["kv"], table(pages), kp, vp, c["scale"])
        r = c["cu"][b] + i
        assert np.abs(o2[r] - out[r]).max() < 1e-13 and np.abs(l2[r] - lse[r]).max() < 1e-13
        if i < Lq - 1:   # the next row does see the change
            assert np.abs(o2[r + 1] - out[r + 1]).max() > 1e-3


# ---------------------------------------------------------------------------
# pin 5: invariants

def test_page_permutation_is_bit_exact():
    c = random_case(21, q_lens=(1, 4, 2), prefix=(9, 3, 5))
    out, lse = oracle.paged_attention(c["q"], c["cu"], c["kv"], c["pt"], c["kp"], c["vp"], c["scale"])
    rng = np.random.default_rng(5)
    N = c["kp"].shape[0]
    perm = rng.permutation(N)          # new page id of old page p is perm[p]
    kp2, vp2 = np.empty_like(c["kp"]), np.empty_like(c["vp"])
    kp2[perm] = c["kp"]
    vp2[perm] = c["vp"]
    pt2 = np.where(c["pt"] >= 0, perm[np.maximum(c["pt"], 0)], -1).astype(np.int32)
    o2, l2 = oracle.paged_attention(c["q"], c["cu"], c["kv"], pt2, kp2, vp2, c["scale"])
    assert np.array_equal(out, o2) and np.array_equal(lse, l2)


def test_shared_prefix_pages_equal_private_copies():
    rng = np.random.default_rng(22)
    P, Hkv, d, Hq = 4, 2, 8, 4
    prefix_k = rng.standard_normal((8, Hkv, d))
    prefix_v = rng.standard_normal((8, Hkv, d))
    tails = [(rng.standard_normal((n, Hkv, d)), rng.standard_normal((n, Hkv, d))) for n in (3, 6)]
    dk = [np.concatenate([prefix_k, t[0]]) for t in tails]
    dv = [np.concatenate([prefix_v, t[1]]) for t in tails]
    q = rng.standard_normal((2, Hq, d))
    kp, vp, pages = build_paged(dk, dv, P, rng)                   # private copies
    o1, l1 = oracle.paged_attention(q, np.array([0, 1, 2]), np.array([11, 14]), table(pages), kp, vp, 0.3)
    # shared: sequence 1 points its first two logical pages at sequence 0's pages
    pages_sh = [pages[0], pages[0][:2] + pages[1][2:]]
    o2, l2 = oracle.paged_attention(q, np.array([0, 1, 2]), np.array([11, 14]), table(pages_sh), kp, vp, 0.3)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_packing_order_does_not_change_rows():
    c = random_case(23, q_lens=(1, 4, 3), prefix=(5, 2, 6))
    out, lse = oracle.paged_attention(c["q"], c["cu"], c["kv"], c["pt"], c["kp"], c["vp"], c["scale"])
    order = [2, 0, 1]
    q2 = np.concatenate([c["qs"][b] for b in order])
    cu2 = np.concatenate([[0], np.cumsum([len(c["qs"][b]) for b in order])])
    o2, l2 = oracle.paged_attention(q2, cu2, c["kv"][order], c["pt"][order], c["kp"], c["vp"], c["scale"])
    for new_b, b in enumerate(order):
        a0, a1 = c["cu"][b], c["cu"][b + 1]
        n0 = cu2[new_b]
        assert np.array_equal(out[a0:a1], o2[n0:n0 + a1 - a0])
        assert np.array_equal(lse[a0:a1], l2[n0:n0 + a1 - a0])


def test_chunk_equals_successive_decodes():
    c = random_case(24, B=1, q_lens=(7,), prefix=(10,))
    out, lse = oracle.paged_attention(c["q"], c["cu"], c["kv"], c["pt"], c["kp"], c["vp"], c["scale"])
    for i in range(7):
        o1, l1 = oracle.paged_attention(c["q"][i:i + 1], np.array([0, 1]), np.array([10 + i + 1]),
                                        c["pt"], c["kp"], c["vp"], c["scale"])
        assert np.abs(o1[0] - out[i]).max() < 1e-13 and np.abs(l1[0] - lse[i]).max() < 1e-13


def test_unused_slots_are_never_read():
    c = random_case(25, q_lens=(1, 3, 2), prefix=(6, 1, 9))
    out, lse = oracle.paged_attention(c["q"], c["cu"], c["kv"], c["pt"], c["kp"], c["vp"], c["scale"])
    live = oracle.live_slots(c["kp"].shape[0], c["kp"].shape[1], c["pt"], c["kv"])
    kp, vp = c["kp"].copy(), c["vp"].copy()
    kp[~live] = np.nan
    vp[~live] = np.inf
    o2, l2 = oracle.paged_attention(c["q"], c["cu"], c["kv"], c["pt"], kp, vp, c["scale"])
    assert np.array_equal(out, o2) and np.array_equal(lse, l2)
    # live_slots itself, by enumeration of (page, offset) pairs
    want = np.zeros_like(live)
    for b, pg in enumerate(c["pages"]):
        pos = 0
        for page in pg:
            for off in range(c["kp"].shape[1]):
                if pos < c["kv"][b]:
                    want[page, off] = True
                pos += 1
    assert np.array_equal(live, want)


# ---------------------------------------------------------------------------
# pin 6: split identity

@pytest.mark.parametrize("cuts", [(5,), (0, 7), (3, 3, 9), (1, 2, 4, 8, 12)])
def test_split_merge_equals_unsplit(cuts):
    rng = np.random.default_rng(31)
    L, Hkv, d, Hq = 14, 2, 8, 6
    K = rng.standard_normal((L, Hkv, d))
    V = rng.standard_normal((L, Hkv, d))
    q = rng.standard_normal((Hq, d))
    o, lse = oracle.attend_row(q, K, V, L, 0.4)
    bounds = [0] + list(cuts) + [L]
    parts = [oracle.attend_partial(q, K, V, a, b, 0.4) for a, b in zip(bounds, bounds[1:])]
    om, lm = oracle.combine_splits(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    assert np.abs(om - o).max() < 1e-12 and np.abs(lm - lse).max() < 1e-12


def test_combine_closed_form_two_equal_parts():
    """Two parts with equal lse: lse grows by ln 2 and o is the average."""
    o = np.array([[[1.0, 3.0]], [[3.0, -1.0]]])
    lse = np.array([[0.25], [0.25]])
    om, lm = oracle.combine_splits(o, lse)
    assert np.allclose(om, [[2.0, 1.0]], atol=1e-15) and abs(lm[0] - (0.25 + math.log(2))) < 1e-15


# ---------------------------------------------------------------------------
# pin 7: layout arithmetic printed on the pages

def test_pool_size_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "kv_pool_layout.json")))
    n = oracle.pool_bytes(g["dims"], g["elt_bytes"])
    assert n == g["bytes"]
    assert round(n / 1e6, 1) == g["printed_megabytes"]


# ---------------------------------------------------------------------------
# pin 8: append

def test_append_round_trip_and_untouched_slots():
    rng = np.random.default_rng(41)
    N, P, Hkv, d, T = 6, 4, 2, 8, 7
    kc = rng.standard_normal((N, P, Hkv, d)).astype(np.float32)
    vc = rng.standard_normal((N, P, Hkv, d)).astype(np.float32)
    k = rng.standard_normal((T, Hkv, d)).astype(np.float32)
    v = rng.standard_normal((T, Hkv, d)).astype(np.float32)
    slots = np.array([5, 23, -1, 0, 17, 9, -7], dtype=np.int64)
    k2, v2 = oracle.kv_append(kc, vc, k, v, slots)
    flat_k, flat_v = k2.reshape(N * P, Hkv, d), v2.reshape(N * P, Hkv, d)
    touched = set()
    for t, s in enumerate(slots):
        if s >= 0:
            assert flat_k[s].tobytes() == k[t].tobytes() and flat_v[s].tobytes() == v[t].tobytes()
            touched.add(int(s))
    for s in range(N * P):
        if s not in touched:
            assert flat_k[s].tobytes() == kc.reshape(N * P, Hkv, d)[s].tobytes()
    with pytest.raises(oracle.OracleInputError):
        oracle.kv_append(kc, vc, k, v, np.array([1, 1, 2, 3, 4, 5, 6]))
    with pytest.raises(oracle.OracleInputError):
        oracle.kv_append(kc, vc, k, v, np.array([1, 2, 3, 4, 5, 6, N * P]))


# ---------------------------------------------------------------------------
# pin 9: packing

def test_pack_tick_by_enumeration():
    rng = np.random.default_rng(51)
    P = 4
    q_lens = [3, 1, 0, 1, 5, 1]
    kv_lens = [7, 9, 2, 1, 5, 12]
    n_pages = sum(-(-L // P) for L in kv_lens) + 2
    perm = list(rng.permutation(n_pages))
    pages = [[int(perm.pop()) for _ in range(-(-L // P))] for L in kv_lens]
    p = oracle.pack_tick(q_lens, kv_lens, pages, P, max_pages_per_seq=4)
    assert list(p["order"]) == [1, 3, 5, 0, 2, 4]      # decode rows first, arrival order kept
    assert list(p["cu_seqlens_q"]) == [0, 1, 2, 3, 6, 6, 11]
    assert list(p["kv_lens"]) == [9, 1, 12, 7, 2, 5]
    assert p["page_tables"].shape == (6, 4)
    want = []
    for b in p["order"]:
        slots = [page * P + off for page in pages[b] for off in range(P)][:kv_lens[b]]
        want += slots[kv_lens[b] - q_lens[b]:]
    assert list(p["slot_mapping"]) == want
    for row, b in enumerate(p["order"]):
        assert list(p["page_tables"][row, :len(pages[b])]) == pages[b]
        assert all(x == -1 for x in p["page_tables"][row, len(pages[b]):])


def test_workloads_match_their_description():
    w = W.make_workload("mixed_tick")
    assert [r.q_len for r in w.requests].count(1) == 96 and w.total_q == 96 + 4096
    assert [(r.q_len, r.kv_len) for r in w.requests[-2:]] == [(2048, 2048), (2048, 5120)]
    w5 = W.make_workload("shared_prefix_long")
    assert all(r.pages[:16] == w5.requests[0].pages[:16] for r in w5.requests)
    priv = [p for r in w5.requests for p in r.pages[16:]]
    assert len(set(priv)) == len(priv) == 16 * 112 and w5.num_pages == math.ceil(1.25 * 1808)
    w1 = W.make_workload("tiny_decode")
    assert [r.kv_len for r in w1.requests] == [17, 64, 100, 255] and w1.num_pages == 64


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5], dtype=np.float32)
    r = W.round_to_dtype(x, "bf16")
    t = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    assert np.array_equal(r, t)


# ---------------------------------------------------------------------------
# planted slips: each must be caught by a pin above

def _wrong_head_map(q_row, K, V, n_visible, scale):
    Hq, d = q_row.shape
    Hkv = K.shape[1]
    o = np.empty((Hq, d))
    lse = np.empty(Hq)
    for h in range(Hq):
        kvh = h % Hkv                       # slip: interleaved instead of grouped
        s = scale * (K[:n_visible, kvh] @ q_row[h])
        lse[h] = s.max() + np.log(np.exp(s - s.max()).sum())
        o[h] = np.exp(s - lse[h]) @ V[:n_visible, kvh]
    return o, lse


def _off_by_one_causal(q_row, K, V, n_visible, scale):
    return ORIG_ATTEND(q_row, K, V, max(1, n_visible - 1), scale)


def _missing_scale(q_row, K, V, n_visible, scale):
    return ORIG_ATTEND(q_row, K, V, n_visible, 1.0)


ORIG_ATTEND = OPA.attend_row


@pytest.mark.parametrize("slip", [_wrong_head_map, _off_by_one_causal, _missing_scale])
def test_planted_slips_are_caught(monkeypatch, slip):
    monkeypatch.setattr(OPA, "attend_row", slip)
    c = random_case(0, Hq=8, Hkv=2, P=4, q_lens=(1, 1, 5), prefix=(6, 0, 7))
    e_o, e_l = max_err_vs_sdpa(c)
    assert max(e_o, e_l) > 1e-3


def test_planted_page_index_slip_is_caught(monkeypatch):
    def wrong_gather(cache, row, kv_len):
        N, P = cache.shape[:2]
        out = np.empty((kv_len,) + cache.shape[2:])
        for j in range(kv_len):
            out[j] = cache[row[j % P] if j % P < len(row) else row[0], j // P % P]   # slip: swapped
        return out
    monkeypatch.setattr(OPA, "gather_sequence", wrong_gather)
    c = random_case(3, Hq=8, Hkv=4, P=5, q_lens=(9, 1, 1), prefix=(11, 3, 1))
    e_o, _ = max_err_vs_sdpa(c)
    assert e_o > 1e-3

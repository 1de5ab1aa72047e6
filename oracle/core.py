"""CPU oracle for attention over a paged KV cache in one packed tick.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module; the library never does,
and it shares no code with the CUDA path. Everything here is plain NumPy on the
host: index work in Python integers, floating point in float64 on the stored
(dtype-rounded) values widened exactly.

What it computes, and where the serving pages define it:

* the KV page pool: a fixed pool of fixed-size pages, per layer laid out
  ``[pages, page_size, kv_heads, head_dim]`` for K and for V
  (llm-serving-engine README, component table "KV Cache" row and the
  "KV cache memory layout" figure; Helios README, "Paged attention");
* per-sequence page tables that map a position to a page
  (mini-vLLM, "Paged KV-cache"; Helios README, "Paged attention");
* the slot write of each new token before attention (Helios blog, "Prefill vs
  Decode": decode writes the slot of the new token; Helios README, "Paged
  attention": prefill and decode write K and V into the pages, then attend);
* attention softmax(Q K^T * scale) V (Helios blog, "torch.sdpa and Flash
  Attention"), with grouped-query heads sharing KV heads (same section;
  llm-serving-engine README, component table "GQA" row);
* the causal rule: a decode row sees the whole context, a prefill chunk that
  continues after cached K/V sees the whole prefix and is causal inside the
  chunk (llm-serving-engine README, engine step trace, "_step_prefill" /
  "_step_decode"; Helios README, "Paged attention": causal paged attention);
* one packed forward over decode tokens and prefill chunks with independent
  positions and page tables, decode tokens taken first (Helios README,
  "Continuous batching"; Helios blog, "Continuous batching").

Readings taken where the pages are silent (each also listed in the design notes):
query i of a sequence with q_len rows and kv_len keys sits at position
kv_len - q_len + i and sees keys 0..kv_len - q_len + i; kv_len counts the
tokens appended this tick; q head h reads KV head h // (Hq / Hkv); lse is the
natural log of sum_j exp(scale * q.k_j); slot = page * page_size + offset,
negative slots are skipped; the packed row order is decode rows (q_len == 1)
first, then the other sequences, each group in arrival order.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np


class OracleInputError(ValueError):
    """The inputs break the contract of the operation."""


# ---------------------------------------------------------------------------
# layout arithmetic

def pool_bytes(dims: Sequence[int], elt_bytes: int) -> int:
    """Bytes of a pre-allocated KV tensor of the given dimensions
    (llm-serving-engine README, "KV cache memory layout": the tensor
    [layers, 2, blocks, block_size, kv_heads, head_dim] is one allocation)."""
    n = 1
    for x in dims:
        n *= int(x)
    return n * int(elt_bytes)


# ---------------------------------------------------------------------------
# a1: packing one tick

def pack_tick(q_lens: Sequence[int], kv_lens: Sequence[int], pages: Sequence[Sequence[int]],
              page_size: int, max_pages_per_seq: Optional[int] = None):
    """Order the sequences (decode rows first, then the rest, each in arrival
    order) and build the packed metadata of the tick.

    Returns a dict with
      order          [B]      int32, arrival index of each packed sequence
      cu_seqlens_q   [B + 1]  int32, row offsets of the packed sequences
      kv_lens        [B]      int32
      page_tables    [B, max_pages_per_seq] int32, unused entries -1
      slot_mapping   [T]      int64, slot of each packed row's new token
    """
    B = len(q_lens)
    if not (len(kv_lens) == B and len(pages) == B):
        raise OracleInputError("per-sequence lists differ in length")
    P = int(page_size)
    if P <= 0:
        raise OracleInputError("page_size must be positive")
    for q, L, pg in zip(q_lens, kv_lens, pages):
        if q < 0 or L < q or (q > 0 and L < 1):
            raise OracleInputError("need 0 <= q_len <= kv_len and kv_len >= 1 when q_len > 0")
        if len(pg) * P < L:
            raise OracleInputError("a sequence owns fewer pages than its length needs")
    width = max((len(pg) for pg in pages), default=0) if max_pages_per_seq is None else int(max_pages_per_seq)
    if any(len(pg) > width for pg in pages):
        raise OracleInputError("max_pages_per_seq is smaller than a page list")

    order = [b for b in range(B) if q_lens[b] == 1] + [b for b in range(B) if q_lens[b] != 1]
    cu = [0]
    for b in order:
        cu.append(cu[-1] + int(q_lens[b]))
    tables = np.full((B, width), -1, dtype=np.int32)
    slots = []
    for row, b in enumerate(order):
        pg = list(pages[b])
        tables[row, :len(pg)] = pg
        L, q = int(kv_lens[b]), int(q_lens[b])
        for i in range(q):
            pos = L - q + i                      # position of the i-th new token
            slots.append(int(pg[pos // P]) * P + pos % P)
    return dict(
        order=np.array(order, dtype=np.int32),
        cu_seqlens_q=np.array(cu, dtype=np.int32),
        kv_lens=np.array([kv_lens[b] for b in order], dtype=np.int32),
        page_tables=tables,
        slot_mapping=np.array(slots, dtype=np.int64),
    )


# ---------------------------------------------------------------------------
# a2: slot-mapping append

def kv_append(k_cache: np.ndarray, v_cache: np.ndarray, k: np.ndarray, v: np.ndarray,
              slot_mapping: np.ndarray):
    """Write each new token's K and V rows into its slot; return new caches.

    k_cache, v_cache [N, P, Hkv, d]; k, v [T, Hkv, d]; slot_mapping [T].
    Row t goes to page slot // P, offset slot % P; a negative slot is skipped.
    The copy is exact (same dtype in and out)."""
    N, P = k_cache.shape[:2]
    T = k.shape[0]
    if v.shape != k.shape or v_cache.shape != k_cache.shape or slot_mapping.shape != (T,):
        raise OracleInputError("shape mismatch")
    if k.shape[1:] != k_cache.shape[2:] or k.dtype != k_cache.dtype:
        raise OracleInputError("token rows do not match the cache rows")
    live = [int(s) for s in slot_mapping if s >= 0]
    if len(set(live)) != len(live):
        raise OracleInputError("duplicate slot in one append")
    if any(s >= N * P for s in live):
        raise OracleInputError("slot outside the pool")
    kc, vc = k_cache.copy(), v_cache.copy()
    for t in range(T):
        s = int(slot_mapping[t])
        if s < 0:
            continue
        kc[s // P, s % P] = k[t]
        vc[s // P, s % P] = v[t]
    return kc, vc


# ---------------------------------------------------------------------------
# a3/a5: attention through the page table

def gather_sequence(cache: np.ndarray, page_table_row: np.ndarray, kv_len: int) -> np.ndarray:
    """K (or V) of one sequence, positions 0..kv_len-1, as float64 [kv_len, Hkv, d].

    Logical page n of the sequence is physical page page_table_row[n]; position
    j lives at offset j % P of logical page j // P."""
    N, P = cache.shape[:2]
    out = np.empty((kv_len,) + cache.shape[2:], dtype=np.float64)
    for n in range(-(-kv_len // P)):
        page = int(page_table_row[n])
        if not 0 <= page < N:
            raise OracleInputError(f"page id {page} outside the pool")
        rows = min(P, kv_len - n * P)
        out[n * P:n * P + rows] = cache[page, :rows].astype(np.float64)
    return out


def attend_row(q_row: np.ndarray, K: np.ndarray, V: np.ndarray, n_visible: int, scale: float):
    """One query row (all Hq heads) against keys 0..n_visible-1.

    q_row [Hq, d]; K, V [>= n_visible, Hkv, d] float64.
    Returns (o [Hq, d], lse [Hq]) in float64: for each head h with KV head
    h // (Hq / Hkv), s_j = scale * q_h . k_j, lse = ln sum_j exp(s_j),
    o = sum_j exp(s_j - lse) v_j."""
    Hq, d = q_row.shape
    Hkv = K.shape[1]
    g = Hq // Hkv
    q64 = q_row.astype(np.float64)
    o = np.empty((Hq, d), dtype=np.float64)
    lse = np.empty(Hq, dtype=np.float64)
    for kvh in range(Hkv):
        heads = slice(kvh * g, (kvh + 1) * g)
        s = scale * (K[:n_visible, kvh, :] @ q64[heads].T)        # [n, g]
        m = s.max(axis=0)
        lse[heads] = m + np.log(np.exp(s - m).sum(axis=0))
        w = np.exp(s - lse[heads])                                # softmax weights
        o[heads] = w.T @ V[:n_visible, kvh, :]
    return o, lse


def paged_attention(q: np.ndarray, cu_seqlens_q: np.ndarray, kv_lens: np.ndarray,
                    page_tables: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                    scale: float, rows: Optional[Sequence[int]] = None):
    """Attention of every packed query row over its sequence's pages.

    q [T, Hq, d]; cu_seqlens_q [B+1]; kv_lens [B] (after the append);
    page_tables [B, W]; caches [N, P, Hkv, d]. Row i of sequence b attends keys
    0..kv_lens[b] - q_len_b + i. Returns float64 (out [R, Hq, d], lse [R, Hq])
    for the requested rows (all rows when rows is None)."""
    T, Hq, d = q.shape
    N, P, Hkv, dk = k_cache.shape
    if dk != d or Hq % Hkv != 0 or v_cache.shape != k_cache.shape:
        raise OracleInputError("head shapes do not match")
    cu = [int(x) for x in cu_seqlens_q]
    B = len(cu) - 1
    if cu[0] != 0 or cu[-1] != T or any(b < a for a, b in zip(cu, cu[1:])):
        raise OracleInputError("cu_seqlens_q must start at 0, end at T and not decrease")
    want = list(range(T)) if rows is None else [int(r) for r in rows]
    out = np.zeros((len(want), Hq, d), dtype=np.float64)
    lse = np.zeros((len(want), Hq), dtype=np.float64)
    by_seq = {}
    for k, r in enumerate(want):
        b = int(np.searchsorted(cu, r, side="right")) - 1
        by_seq.setdefault(b, []).append((k, r))
    for b, items in by_seq.items():
        Lq, L = cu[b + 1] - cu[b], int(kv_lens[b])
        if L < Lq or L < 1:
            raise OracleInputError("kv_len must be >= q_len and >= 1")
        K = gather_sequence(k_cache, page_tables[b], L)
        V = gather_sequence(v_cache, page_tables[b], L)
        for k, r in items:
            i = r - cu[b]
            n_visible = L - Lq + i + 1
            out[k], lse[k] = attend_row(q[r], K, V, n_visible, scale)
    return out, lse


# ---------------------------------------------------------------------------
# a4: split-KV merge

def attend_partial(q_row: np.ndarray, K: np.ndarray, V: np.ndarray, lo: int, hi: int, scale: float):
    """Partial result over keys lo..hi-1 of one row: (o normalised within the
    part, lse of the part). An empty part gives (0, -inf)."""
    Hq, d = q_row.shape
    if hi <= lo:
        return np.zeros((Hq, d)), np.full(Hq, -np.inf)
    o, lse = attend_row(q_row, K[lo:hi], V[lo:hi], hi - lo, scale)
    return o, lse


def combine_splits(o_parts: np.ndarray, lse_parts: np.ndarray):
    """Merge partial results over disjoint key ranges (axis 0 = part):
    lse = ln sum_s exp(lse_s); o = sum_s exp(lse_s - lse) o_s."""
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    o_parts = np.asarray(o_parts, dtype=np.float64)
    m = lse_parts.max(axis=0)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    lse = m_safe + np.log(np.exp(lse_parts - m_safe).sum(axis=0))
    w = np.exp(lse_parts - lse)                                    # [S, ...]
    o = (w[..., None] * o_parts).sum(axis=0)
    return o, lse


# ---------------------------------------------------------------------------
# helpers for building test inputs

def live_slots(num_pages: int, page_size: int, page_tables: np.ndarray, kv_lens: np.ndarray) -> np.ndarray:
    """Boolean [N, P]: slots that hold a position < kv_len of some sequence."""
    live = np.zeros((num_pages, page_size), dtype=bool)
    for b in range(len(kv_lens)):
        L = int(kv_lens[b])
        for j in range(L):
            live[int(page_tables[b][j // page_size]), j % page_size] = True
    return live


"""Seeded synthetic inputs for one packed paged-KV attention tick.

This module only draws random numbers: sequence lengths, which physical pages a
sequence owns, and the N(0, 1) values of Q, K, V and of the page pool, rounded to
the cache dtype. It holds none of the attention arithmetic (no slot numbers, no
masking, no softmax, no packing); both the CUDA path's tests/benchmark and the
CPU oracle are fed from it.

The five named workloads follow the shapes the serving pages describe:
a TinyLlama-shaped cache (32 query heads, 4 KV heads, head_dim 64, 16-token
blocks; llm-serving-engine README, component table "GQA" row and the
"KV cache memory layout" figure) and Helios' Qwen3-4B engine with 256-token
pages (Helios README, "Paged attention"). The Qwen3-4B head counts (32/8,
head_dim 128) are not printed on the pages and are taken as stated in the
workload description.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np

DTYPES = ("f32", "f16", "bf16")


@dataclasses.dataclass(frozen=True)
class TickShape:
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    dtype: str  # one of DTYPES

    @property
    def elt_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2


@dataclasses.dataclass
class Request:
    """One sequence in the tick.

    q_len:  tokens this sequence contributes to the tick (1 for a decode step,
            the chunk length for a prefill chunk, 0 for an idle sequence).
    kv_len: context length after this tick's tokens are written (it counts them).
    pages:  physical page ids the sequence owns, in logical order
            (len == ceil(kv_len / page_size)).
    """
    q_len: int
    kv_len: int
    pages: List[int]


@dataclasses.dataclass
class Workload:
    name: str
    shape: TickShape
    requests: List[Request]
    num_pages: int
    scale: float
    seed: int

    @property
    def total_q(self) -> int:
        return sum(r.q_len for r in self.requests)

    @property
    def num_seqs(self) -> int:
        return len(self.requests)

    @property
    def max_kv_len(self) -> int:
        return max((r.kv_len for r in self.requests), default=0)

    @property
    def max_pages_per_seq(self) -> int:
        return max((len(r.pages) for r in self.requests), default=0)


QWEN3_4B = dict(num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=256)
TINYLLAMA = dict(num_q_heads=32, num_kv_heads=4, head_dim=64, page_size=16)

WORKLOADS = (
    "tiny_decode",         # 4 seqs, kv {17,64,100,255}, 8/2 heads, d 64, page 16
    "tinyllama_decode",    # 64 seqs, kv U[128,2048], 32/4 heads, d 64, page 16, fp16
    "qwen3_decode",        # 128 seqs, kv U[512,8192], 32/8 heads, d 128, page 256, bf16
    "mixed_tick",          # 96 decodes + 2 prefill chunks of 2048, Qwen3-4B shape, bf16
    "shared_prefix_long",  # 16 seqs of 32768, 16 shared prefix pages, Qwen3-4B shape, bf16
    # two more packings of the mixed tick's kind, to check how the prefill /
    # decode share of the SMs holds up away from the named tick
    "mixed_decode_heavy",  # 256 decodes + one 1024-token chunk after 2048, Qwen3-4B shape, bf16
    "mixed_many_chunks",   # 32 decodes + four 512-token chunks after 0/1024/2048/4096, Qwen3-4B shape
)
BASE_SEED = 20261202


def _pages_needed(kv_len: int, page_size: int) -> int:
    # how many pages a sequence of this length occupies (allocation size only)
    return -(-kv_len // page_size)


def _scatter_pages(rng, lens_pages: List[int], headroom: float = 1.25):
    need = sum(lens_pages)
    num_pages = max(1, math.ceil(headroom * need))
    perm = rng.permutation(num_pages)
    out, pos = [], 0
    for n in lens_pages:
        out.append([int(p) for p in perm[pos:pos + n]])
        pos += n
    return out, num_pages


def make_workload(name: str, dtype: Optional[str] = None) -> Workload:
    """The five named tick workloads, drawn from seed BASE_SEED + index."""
    idx = WORKLOADS.index(name)
    seed = BASE_SEED + idx
    rng = np.random.default_rng(seed)
    if name == "tiny_decode":
        shape = TickShape(8, 2, 64, 16, dtype or "f32")
        lens = [17, 64, 100, 255]
        num_pages = 64
        perm = rng.permutation(num_pages)
        reqs, pos = [], 0
        for L in lens:
            n = _pages_needed(L, 16)
            reqs.append(Request(1, L, [int(p) for p in perm[pos:pos + n]]))
            pos += n
    elif name == "tinyllama_decode":
        shape = TickShape(**TINYLLAMA, dtype=dtype or "f16")
        lens = [int(x) for x in rng.integers(128, 2048 + 1, size=64)]
        pages, num_pages = _scatter_pages(rng, [_pages_needed(L, 16) for L in lens])
        reqs = [Request(1, L, p) for L, p in zip(lens, pages)]
    elif name == "qwen3_decode":
        shape = TickShape(**QWEN3_4B, dtype=dtype or "bf16")
        lens = [int(x) for x in rng.integers(512, 8192 + 1, size=128)]
        pages, num_pages = _scatter_pages(rng, [_pages_needed(L, 256) for L in lens])
        reqs = [Request(1, L, p) for L, p in zip(lens, pages)]
    elif name == "mixed_tick":
        shape = TickShape(**QWEN3_4B, dtype=dtype or "bf16")
        lens = [int(x) for x in rng.integers(256, 4096 + 1, size=96)]
        q_lens = [1] * 96 + [2048, 2048]
        kv = lens + [2048, 3072 + 2048]
        pages, num_pages = _scatter_pages(rng, [_pages_needed(L, 256) for L in kv])
        reqs = [Request(q, L, p) for q, L, p in zip(q_lens, kv, pages)]
    elif name in ("mixed_decode_heavy", "mixed_many_chunks"):
        shape = TickShape(**QWEN3_4B, dtype=dtype or "bf16")
        n_dec, chunks = (256, [(1024, 2048)]) if name == "mixed_decode_heavy" else \
            (32, [(512, 0), (512, 1024), (512, 2048), (512, 4096)])
        lens = [int(x) for x in rng.integers(256, 4096 + 1, size=n_dec)]
        q_lens = [1] * n_dec + [q for q, _ in chunks]
        kv = lens + [pre + q for q, pre in chunks]
        pages, num_pages = _scatter_pages(rng, [_pages_needed(L, 256) for L in kv])
        reqs = [Request(q, L, p) for q, L, p in zip(q_lens, kv, pages)]
    elif name == "shared_prefix_long":
        shape = TickShape(**QWEN3_4B, dtype=dtype or "bf16")
        B, L, shared = 16, 32768, 16
        per_seq = _pages_needed(L, 256)  # 128
        need = shared + B * (per_seq - shared)  # 1808
        num_pages = math.ceil(1.25 * need)
        perm = [int(p) for p in rng.permutation(num_pages)]
        prefix = perm[:shared]
        reqs, pos = [], shared
        for _ in range(B):
            priv = perm[pos:pos + per_seq - shared]
            pos += per_seq - shared
            reqs.append(Request(1, L, prefix + priv))
    else:  # pragma: no cover
        raise ValueError(name)
    return Workload(name, shape, reqs, num_pages, 1.0 / math.sqrt(shape.head_dim), seed)


def random_workload(seed: int, num_seqs: int, num_q_heads: int, num_kv_heads: int,
                    head_dim: int, page_size: int, dtype: str, q_lens, max_kv: int,
                    min_prefix: int = 0, headroom: float = 1.5) -> Workload:
    """A small ragged tick: q_len drawn from `q_lens`, prefix length from
    [min_prefix, max_kv - q_len], pages scattered over a pool with headroom."""
    rng = np.random.default_rng(seed)
    qs, kvs = [], []
    for _ in range(num_seqs):
        q = int(rng.choice(q_lens))
        hi = max(min_prefix, max_kv - q)
        prefix = int(rng.integers(min_prefix, hi + 1))
        if q == 0 and prefix == 0:
            prefix = 1
        qs.append(q)
        kvs.append(prefix + q)
    pages, num_pages = _scatter_pages(rng, [_pages_needed(L, page_size) for L in kvs], headroom)
    shape = TickShape(num_q_heads, num_kv_heads, head_dim, page_size, dtype)
    reqs = [Request(q, L, p) for q, L, p in zip(qs, kvs, pages)]
    return Workload(f"random{seed}", shape, reqs, num_pages, 1.0 / math.sqrt(head_dim), seed)


# ---------------------------------------------------------------------------
# values

def round_to_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round fp32 values to the cache dtype (round to nearest even).

    f32 -> float32, f16 -> float16, bf16 -> float32 holding bf16 values."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f32":
        return x
    if dtype == "f16":
        return x.astype(np.float16)
    if dtype == "bf16":
        b = x.view(np.uint32)
        b = b + (np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1)))
        return (b & np.uint32(0xFFFF0000)).view(np.float32)
    raise ValueError(dtype)


@dataclasses.dataclass
class TickValues:
    """Host arrays, in the row order of the workload's requests.

    q [T, Hq, d]; k_new, v_new [T, Hkv, d]; k_cache, v_cache [N, P, Hkv, d].
    bf16 values are held in float32 arrays (exactly representable)."""
    q: np.ndarray
    k_new: np.ndarray
    v_new: np.ndarray
    k_cache: np.ndarray
    v_cache: np.ndarray


def host_values(w: Workload) -> TickValues:
    s = w.shape
    rng = np.random.default_rng([w.seed, 1])
    T = w.total_q

    def draw(*shape):
        return round_to_dtype(rng.standard_normal(shape, dtype=np.float32), s.dtype)

    q = draw(T, s.num_q_heads, s.head_dim)
    k_new = draw(T, s.num_kv_heads, s.head_dim)
    v_new = draw(T, s.num_kv_heads, s.head_dim)
    k_cache = draw(w.num_pages, s.page_size, s.num_kv_heads, s.head_dim)
    v_cache = draw(w.num_pages, s.page_size, s.num_kv_heads, s.head_dim)
    return TickValues(q, k_new, v_new, k_cache, v_cache)


def torch_dtype(dtype: str):
    import torch
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]


def to_torch(x: np.ndarray, dtype: str, device="cpu"):
    """Host array (as produced above) -> torch tensor of the cache dtype."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x))
    return t.to(torch_dtype(dtype)).to(device)


def device_values(w: Workload, device="cuda"):
    """Same shapes as host_values, drawn on the device by torch's seeded
    generator (fast for multi-GB pools). Returns a dict of torch tensors."""
    import torch
    s = w.shape
    g = torch.Generator(device=device)
    g.manual_seed(w.seed)
    T = w.total_q
    dt = torch_dtype(s.dtype)

    def draw(*shape):
        return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(dt)

    return dict(
        q=draw(T, s.num_q_heads, s.head_dim),
        k_new=draw(T, s.num_kv_heads, s.head_dim),
        v_new=draw(T, s.num_kv_heads, s.head_dim),
        k_cache=draw(w.num_pages, s.page_size, s.num_kv_heads, s.head_dim),
        v_cache=draw(w.num_pages, s.page_size, s.num_kv_heads, s.head_dim),
    )

"""Thin ctypes binding of libpagedkv (declared in include/pagedkv.h).

Argument marshalling only: torch tensors become device pointers and the
current torch stream becomes the cudaStream_t; every step of the computation
runs in the library's kernels. There is no fallback: if the library is missing
or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import itertools
import os
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpagedkv.so")

PKV_F32, PKV_F16, PKV_BF16, PKV_FP8_E4M3 = 0, 1, 2, 3
DEV_BAD_SLOT, DEV_BAD_LENGTHS, DEV_BAD_PAGE, DEV_TIMEOUT, DEV_BAD_POSITION = 0x1, 0x2, 0x4, 0x8, 0x10

EXPORTED = (
    "pkv_pack_tick",
    "pkv_kv_append",
    "pkv_paged_attention_workspace_size",
    "pkv_paged_attention",
    "pkv_paged_attention_no_alloc",
    "pkv_status_string",
    "pkv_get_device_status",
    "pkv_selftest_bounded_wait",
    "pkv_set_kernel_timing",
    "pkv_kernel_times",
    "pkv_version",
    "pkv_last_error",
    "pkv_pool_create",
    "pkv_pool_destroy",
    "pkv_pool_alloc",
    "pkv_pool_retain",
    "pkv_pool_release",
    "pkv_pool_free_count",
    "pkv_pool_refcount",
    "pkv_prefix_lookup",
    "pkv_prefix_insert",
    "pkv_prefix_evict",
    "pkv_prefix_size",
    "pkv_rope_table",
    "pkv_rope_kv_append",
    "pkv_tick_positions",
    "pkv_kv_append_quant",
    "pkv_paged_attention_fp8",
)


class PagedKVError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = f"; {lib().pkv_last_error().decode()}" if status == -8 else ""
        super().__init__(f"{where}: {status_string(status)} (status {status}){detail}")


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_pages", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32)]


_lib = None


def lib():
    """Load libpagedkv.so (built by paged_kv_attention_mapping_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libpagedkv.so is not built ({LIB_PATH}); run "
                           "`python -c 'import __graft_entry__ as g; g.build()'` first")
    L = ctypes.CDLL(LIB_PATH)
    i32, i64, vp, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
    P32, P64 = ctypes.POINTER(i32), ctypes.POINTER(i64)
    L.pkv_pack_tick.argtypes = [i32, vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
    L.pkv_pack_tick.restype = ctypes.c_int
    L.pkv_kv_append.argtypes = [vp, vp, vp, i32, vp, vp, ctypes.POINTER(CacheDesc), vp]
    L.pkv_kv_append.restype = ctypes.c_int
    L.pkv_paged_attention_workspace_size.argtypes = [i32, i32, i32, ctypes.POINTER(CacheDesc), i32]
    L.pkv_paged_attention_workspace_size.restype = sz
    L.pkv_paged_attention.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp,
                                      ctypes.POINTER(CacheDesc), ctypes.c_float, vp, vp, vp, sz, vp]
    L.pkv_paged_attention.restype = ctypes.c_int
    L.pkv_paged_attention_no_alloc.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp,
                                               ctypes.POINTER(CacheDesc), ctypes.c_float, vp, vp, vp]
    L.pkv_paged_attention_no_alloc.restype = ctypes.c_int
    L.pkv_status_string.argtypes = [ctypes.c_int]
    L.pkv_status_string.restype = ctypes.c_char_p
    L.pkv_get_device_status.argtypes = [P32, vp]
    L.pkv_get_device_status.restype = ctypes.c_int
    L.pkv_selftest_bounded_wait.argtypes = [i32, vp, vp]
    L.pkv_selftest_bounded_wait.restype = ctypes.c_int
    L.pkv_set_kernel_timing.argtypes = [ctypes.c_int]
    L.pkv_set_kernel_timing.restype = ctypes.c_int
    L.pkv_kernel_times.argtypes = [ctypes.POINTER(ctypes.c_char_p), P32, ctypes.POINTER(ctypes.c_double), i32]
    L.pkv_kernel_times.restype = ctypes.c_int
    L.pkv_last_error.argtypes = []
    L.pkv_last_error.restype = ctypes.c_char_p
    L.pkv_pool_create.argtypes = [i32, i32, ctypes.POINTER(vp)]
    L.pkv_pool_create.restype = ctypes.c_int
    L.pkv_pool_destroy.argtypes = [vp]
    L.pkv_pool_destroy.restype = None
    for name in ("pkv_pool_alloc", "pkv_pool_retain", "pkv_pool_release"):
        getattr(L, name).argtypes = [vp, P32, i32] if name != "pkv_pool_alloc" else [vp, i32, P32]
        getattr(L, name).restype = ctypes.c_int
    L.pkv_pool_free_count.argtypes = [vp]
    L.pkv_pool_free_count.restype = ctypes.c_int
    L.pkv_pool_refcount.argtypes = [vp, i32]
    L.pkv_pool_refcount.restype = ctypes.c_int
    L.pkv_prefix_lookup.argtypes = [vp, P32, i32, ctypes.c_double, P32, i32]
    L.pkv_prefix_lookup.restype = ctypes.c_int
    L.pkv_prefix_insert.argtypes = [vp, P32, i32, P32, i32, ctypes.c_double]
    L.pkv_prefix_insert.restype = ctypes.c_int
    L.pkv_prefix_evict.argtypes = [vp, ctypes.c_double, ctypes.c_double, i32]
    L.pkv_prefix_evict.restype = ctypes.c_int
    L.pkv_prefix_size.argtypes = [vp]
    L.pkv_prefix_size.restype = ctypes.c_int
    L.pkv_rope_table.argtypes = [ctypes.c_double, i32, i32, ctypes.POINTER(ctypes.c_float)]
    L.pkv_rope_table.restype = ctypes.c_int
    L.pkv_rope_kv_append.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, vp, vp, ctypes.POINTER(CacheDesc), vp, vp]
    L.pkv_rope_kv_append.restype = ctypes.c_int
    L.pkv_kv_append_quant.argtypes = [vp, vp, i32, vp, i32, vp, vp, ctypes.POINTER(CacheDesc), vp, vp, vp]
    L.pkv_kv_append_quant.restype = ctypes.c_int
    L.pkv_paged_attention_fp8.argtypes = [vp, i32, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp,
                                          ctypes.POINTER(CacheDesc), vp, vp, ctypes.c_float, vp, vp, vp, sz, vp]
    L.pkv_paged_attention_fp8.restype = ctypes.c_int
    L.pkv_tick_positions.argtypes = [i32, P32, P32, P32, i32]
    L.pkv_tick_positions.restype = ctypes.c_int
    L.pkv_version.argtypes = []
    L.pkv_version.restype = ctypes.c_char_p
    _lib = L
    return L


def status_string(status: int) -> str:
    return lib().pkv_status_string(int(status)).decode()


def version() -> str:
    return lib().pkv_version().decode()


def _check(status: int, where: str):
    if status != 0:
        raise PagedKVError(status, where)


# ---------------------------------------------------------------------------
# host packing

def pack_tick(q_lens: Sequence[int], kv_lens: Sequence[int], pages: Sequence[Sequence[int]], page_size: int,
              num_pages: int, max_pages_per_seq: Optional[int] = None):
    """Host packing of one tick (pkv_pack_tick). Returns numpy arrays:
    order, cu_seqlens_q, kv_lens, page_tables [B, W] (-1 padded), slot_mapping."""
    B = len(q_lens)
    counts = [len(p) for p in pages]
    offs = np.zeros(B + 1, dtype=np.int32)
    if B:
        np.cumsum(counts, out=offs[1:])
    ids = np.fromiter(itertools.chain.from_iterable(pages), dtype=np.int32, count=int(offs[-1]))
    return pack_tick_flat(np.asarray(q_lens, dtype=np.int32), np.asarray(kv_lens, dtype=np.int32), offs, ids,
                          page_size, num_pages, max_pages_per_seq)


def pack_tick_flat(q_lens, kv_lens, page_offsets, page_ids, page_size: int, num_pages: int,
                   max_pages_per_seq: Optional[int] = None, out: Optional[dict] = None):
    """pack_tick on flat int32 arrays, the form a scheduler keeps its block
    tables in: sequence b owns page_ids[page_offsets[b]:page_offsets[b + 1]].

    `out` may hold preallocated (for example pinned) numpy arrays to write into:
    order [>= B], cu_seqlens_q [B + 1], kv_lens [>= B], page_tables [B, W] and
    slot_mapping [>= sum of q_lens] (int64), so that a serving loop packs each
    tick without allocating. Returns the same dict as pack_tick (views of `out`)."""
    ql = np.ascontiguousarray(q_lens, dtype=np.int32)
    kl = np.ascontiguousarray(kv_lens, dtype=np.int32)
    offs = np.ascontiguousarray(page_offsets, dtype=np.int32)
    ids = np.ascontiguousarray(page_ids, dtype=np.int32)
    B = int(ql.shape[0])
    if offs.shape[0] != B + 1:
        raise ValueError("page_offsets must have num_seqs + 1 entries")
    if ids.size == 0:
        ids = np.zeros(1, dtype=np.int32)
    if max_pages_per_seq is not None:
        W = int(max_pages_per_seq)
    else:
        W = int(np.max(np.diff(offs))) if B else 1
    W = max(W, 1)
    cap = int(max(int(ql.clip(min=0).sum()), 1))
    if out is None:
        out = dict(order=np.zeros(max(B, 1), dtype=np.int32), cu_seqlens_q=np.zeros(B + 1, dtype=np.int32),
                   kv_lens=np.zeros(max(B, 1), dtype=np.int32), page_tables=np.zeros((max(B, 1), W), dtype=np.int32),
                   slot_mapping=np.zeros(cap, dtype=np.int64))
    order, cu, kv_out, tables, slots = (out["order"], out["cu_seqlens_q"], out["kv_lens"], out["page_tables"],
                                        out["slot_mapping"])
    if (order.dtype != np.int32 or cu.dtype != np.int32 or kv_out.dtype != np.int32 or tables.dtype != np.int32
            or slots.dtype != np.int64):
        raise ValueError("pack_tick_flat: out arrays must be int32 (slot_mapping int64)")
    if (order.size < max(B, 1) or cu.size < B + 1 or kv_out.size < max(B, 1) or tables.ndim != 2
            or tables.shape[0] < max(B, 1) or tables.shape[1] != W or slots.size < cap):
        raise ValueError("pack_tick_flat: out arrays too small for this tick")
    for a in (order, cu, kv_out, tables, slots):
        if not a.flags.c_contiguous:
            raise ValueError("pack_tick_flat: out arrays must be C-contiguous")
    total = np.zeros(1, dtype=np.int32)
    st = lib().pkv_pack_tick(B, ql.ctypes.data if B else None, kl.ctypes.data if B else None, offs.ctypes.data,
                             ids.ctypes.data, int(page_size), int(num_pages), W, cap, order.ctypes.data,
                             cu.ctypes.data, kv_out.ctypes.data, tables.ctypes.data, slots.ctypes.data,
                             total.ctypes.data)
    _check(st, "pkv_pack_tick")
    T = int(total[0])
    return dict(order=order[:B], cu_seqlens_q=cu[:B + 1], kv_lens=kv_out[:B], page_tables=tables[:B],
                slot_mapping=slots[:T])


# ---------------------------------------------------------------------------
# device calls (torch tensors)

def _dtype_code(t) -> int:
    import torch
    m = {torch.float32: PKV_F32, torch.float16: PKV_F16, torch.bfloat16: PKV_BF16,
         torch.uint8: PKV_FP8_E4M3}
    if hasattr(torch, "float8_e4m3fn"):
        m[torch.float8_e4m3fn] = PKV_FP8_E4M3
    if t.dtype not in m:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return m[t.dtype]


def cache_desc(k_cache) -> CacheDesc:
    if k_cache.dim() != 4 or not k_cache.is_contiguous():
        raise ValueError("cache must be a contiguous [num_pages, page_size, num_kv_heads, head_dim] tensor")
    N, P, H, D = k_cache.shape
    return CacheDesc(N, P, H, D, _dtype_code(k_cache))


def _stream_ptr(stream=None) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _ptr(t) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


def kv_append(k, v, slot_mapping, k_cache, v_cache, stream=None):
    """Write new tokens' K/V rows into their slots (pkv_kv_append)."""
    for t in (k, v, slot_mapping, k_cache, v_cache):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("kv_append needs contiguous CUDA tensors")
    import torch
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    desc = cache_desc(k_cache)
    st = lib().pkv_kv_append(_ptr(k), _ptr(v), _ptr(slot_mapping), int(k.shape[0]), _ptr(k_cache), _ptr(v_cache),
                             ctypes.byref(desc), _stream_ptr(stream))
    _check(st, "pkv_kv_append")


def workspace_size(num_seqs: int, total_q: int, num_q_heads: int, k_cache, max_kv_len: int) -> int:
    desc = cache_desc(k_cache)
    n = lib().pkv_paged_attention_workspace_size(int(num_seqs), int(total_q), int(num_q_heads), ctypes.byref(desc),
                                                 int(max_kv_len))
    if n == 0:
        raise PagedKVError(-3, "pkv_paged_attention_workspace_size")
    return int(n)


def alloc_workspace(num_seqs, total_q, num_q_heads, k_cache, max_kv_len):
    import torch
    n = workspace_size(num_seqs, total_q, num_q_heads, k_cache, max_kv_len)
    return torch.empty(n, dtype=torch.uint8, device=k_cache.device)


def _check_attention_args(where, q, cu_seqlens_q, kv_lens, page_tables, k_cache, v_cache, out, lse,
                          extra=(), q_matches_cache=True):
    """The checks every attention call makes before any pointer reaches the
    library: CUDA, contiguous, int32 index tensors, consistent dtypes and shapes."""
    import torch
    for t in (cu_seqlens_q, kv_lens, page_tables):
        if t.dtype != torch.int32:
            raise TypeError(f"{where}: index tensors must be int32")
    if v_cache.dtype != k_cache.dtype or v_cache.shape != k_cache.shape:
        raise TypeError(f"{where}: k_cache and v_cache must share one dtype and shape")
    if q_matches_cache and q.dtype != k_cache.dtype:
        raise TypeError(f"{where}: q, k_cache and v_cache must share one dtype")
    for t in (q, cu_seqlens_q, kv_lens, page_tables, k_cache, v_cache) + tuple(extra):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{where} needs contiguous CUDA tensors")
    if q.dim() != 3 or page_tables.dim() != 2 or cu_seqlens_q.dim() != 1 or kv_lens.dim() != 1:
        raise ValueError(f"{where}: q [T, Hq, d], cu_seqlens_q [B+1], kv_lens [B], page_tables [B, W]")
    B = int(cu_seqlens_q.shape[0]) - 1
    if B < 0 or int(kv_lens.shape[0]) < B or int(page_tables.shape[0]) < B:
        raise ValueError(f"{where}: cu_seqlens_q, kv_lens and page_tables disagree on the number of sequences")
    if out is not None:
        if not out.is_cuda or not out.is_contiguous() or out.dtype != q.dtype or out.shape != q.shape:
            raise ValueError(f"{where}: out must be a contiguous CUDA tensor shaped and typed like q")
    if lse is not None:
        if (not lse.is_cuda or not lse.is_contiguous() or lse.dtype != torch.float32
                or tuple(lse.shape) != tuple(q.shape[:2])):
            raise ValueError(f"{where}: lse must be a contiguous float32 CUDA tensor [T, Hq]")


def paged_attention(q, cu_seqlens_q, kv_lens, page_tables, k_cache, v_cache, scale: float, max_kv_len: int,
                    out=None, lse=None, workspace=None, want_lse: bool = True, stream=None):
    """Attention of packed query rows over their pages (pkv_paged_attention).

    q [T, Hq, d] (cache dtype); cu_seqlens_q int32 [B+1]; kv_lens int32 [B];
    page_tables int32 [B, W]; caches [N, P, Hkv, d]. Returns (out, lse)."""
    import torch
    _check_attention_args("paged_attention", q, cu_seqlens_q, kv_lens, page_tables, k_cache, v_cache, out, lse)
    T, Hq, D = q.shape
    B = int(cu_seqlens_q.shape[0]) - 1
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(B, T, Hq, k_cache, max_kv_len)
    elif not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("paged_attention: workspace must be a contiguous CUDA tensor")
    desc = cache_desc(k_cache)
    st = lib().pkv_paged_attention(_ptr(q), _ptr(cu_seqlens_q), _ptr(kv_lens), _ptr(page_tables), B, int(T), int(Hq),
                                   int(page_tables.shape[1]), int(max_kv_len), _ptr(k_cache), _ptr(v_cache),
                                   ctypes.byref(desc), ctypes.c_float(scale), _ptr(out), _ptr(lse), _ptr(workspace),
                                   int(workspace.numel() * workspace.element_size()), _stream_ptr(stream))
    _check(st, "pkv_paged_attention")
    return out, lse


def paged_attention_no_alloc(q, cu_seqlens_q, kv_lens, page_tables, k_cache, v_cache, scale: float,
                             max_kv_len: int, out=None, lse=None, want_lse: bool = True, stream=None):
    """pkv_paged_attention_no_alloc: as paged_attention, but the library uses its
    own fixed device scratch array instead of a caller workspace (for callers
    that cannot allocate device memory). Output buffers may still be passed in;
    when they are not, this wrapper allocates them with torch (the C call
    itself never allocates)."""
    import torch
    _check_attention_args("paged_attention_no_alloc", q, cu_seqlens_q, kv_lens, page_tables, k_cache, v_cache,
                          out, lse)
    T, Hq, D = q.shape
    B = int(cu_seqlens_q.shape[0]) - 1
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device)
    desc = cache_desc(k_cache)
    st = lib().pkv_paged_attention_no_alloc(_ptr(q), _ptr(cu_seqlens_q), _ptr(kv_lens), _ptr(page_tables), B,
                                            int(T), int(Hq), int(page_tables.shape[1]), int(max_kv_len),
                                            _ptr(k_cache), _ptr(v_cache), ctypes.byref(desc), ctypes.c_float(scale),
                                            _ptr(out), _ptr(lse), _stream_ptr(stream))
    _check(st, "pkv_paged_attention_no_alloc")
    return out, lse


def kv_append_quant(k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale, stream=None):
    """Quantise new tokens' K/V rows to e4m3 codes of x / scale[head] and write
    them into their slots of an fp8 cache (pkv_kv_append_quant). Caches are
    uint8 (or float8_e4m3fn) [N, P, Hkv, d]; scales float32 [Hkv] on the device."""
    import torch
    for t in (k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("kv_append_quant needs contiguous CUDA tensors")
    if slot_mapping.dtype != torch.int64 or k_scale.dtype != torch.float32 or v_scale.dtype != torch.float32:
        raise TypeError("slot_mapping int64, scales float32")
    desc = cache_desc(k_cache)
    st = lib().pkv_kv_append_quant(_ptr(k), _ptr(v), _dtype_code(k), _ptr(slot_mapping), int(k.shape[0]),
                                   _ptr(k_cache), _ptr(v_cache), ctypes.byref(desc), _ptr(k_scale), _ptr(v_scale),
                                   _stream_ptr(stream))
    _check(st, "pkv_kv_append_quant")


def paged_attention_fp8(q, cu_seqlens_q, kv_lens, page_tables, k_cache, v_cache, k_scale, v_scale, scale: float,
                        max_kv_len: int, out=None, lse=None, workspace=None, want_lse: bool = True, stream=None):
    """Attention over an fp8 e4m3 cache (pkv_paged_attention_fp8): q/out bf16 or
    f16 [T, Hq, d]; caches uint8 codes [N, P, Hkv, d]; element = code * scale[head]."""
    import torch
    _check_attention_args("paged_attention_fp8", q, cu_seqlens_q, kv_lens, page_tables, k_cache, v_cache, out, lse,
                          extra=(k_scale, v_scale), q_matches_cache=False)
    if k_scale.dtype != torch.float32 or v_scale.dtype != torch.float32:
        raise TypeError("paged_attention_fp8: scales must be float32")
    T, Hq, D = q.shape
    B = int(cu_seqlens_q.shape[0]) - 1
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(B, T, Hq, k_cache, max_kv_len)
    elif not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("paged_attention_fp8: workspace must be a contiguous CUDA tensor")
    desc = cache_desc(k_cache)
    st = lib().pkv_paged_attention_fp8(_ptr(q), _dtype_code(q), _ptr(cu_seqlens_q), _ptr(kv_lens),
                                       _ptr(page_tables), B, int(T), int(Hq), int(page_tables.shape[1]),
                                       int(max_kv_len), _ptr(k_cache), _ptr(v_cache), ctypes.byref(desc),
                                       _ptr(k_scale), _ptr(v_scale), ctypes.c_float(scale), _ptr(out), _ptr(lse),
                                       _ptr(workspace), int(workspace.numel() * workspace.element_size()),
                                       _stream_ptr(stream))
    _check(st, "pkv_paged_attention_fp8")
    return out, lse


def tick_positions(cu_seqlens_q, kv_lens) -> np.ndarray:
    """Position of every packed row (pkv_tick_positions), host int32 array."""
    cu = np.ascontiguousarray(cu_seqlens_q, dtype=np.int32)
    kl = np.ascontiguousarray(kv_lens, dtype=np.int32)
    out = np.zeros(max(int(cu[-1]), 1), dtype=np.int32)
    P32 = ctypes.POINTER(ctypes.c_int32)
    _check(lib().pkv_tick_positions(len(kl), cu.ctypes.data_as(P32), kl.ctypes.data_as(P32),
                                    out.ctypes.data_as(P32), len(out)), "pkv_tick_positions")
    return out[:int(cu[-1])]


def rope_table(base: float, head_dim: int, max_pos: int) -> np.ndarray:
    """Host cos/sin table [max_pos, head_dim/2, 2] float32 (pkv_rope_table)."""
    out = np.zeros((max_pos, head_dim // 2, 2), dtype=np.float32)
    _check(lib().pkv_rope_table(float(base), int(head_dim), int(max_pos),
                                out.ctypes.data_as(ctypes.POINTER(ctypes.c_float))), "pkv_rope_table")
    return out


def rope_kv_append(q, k, v, positions, cos_sin, slot_mapping, k_cache, v_cache, q_out=None, stream=None):
    """Rotate K and write it with V to the slots; rotate Q into q_out
    (pkv_rope_kv_append). cos_sin: device float32 [max_pos, d/2, 2]."""
    import torch
    for t in (q, k, v, positions, cos_sin, slot_mapping, k_cache, v_cache):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("rope_kv_append needs contiguous CUDA tensors")
    if positions.dtype != torch.int32 or slot_mapping.dtype != torch.int64 or cos_sin.dtype != torch.float32:
        raise TypeError("positions int32, slot_mapping int64, cos_sin float32")
    if q_out is None:
        q_out = torch.empty_like(q)
    desc = cache_desc(k_cache)
    st = lib().pkv_rope_kv_append(_ptr(q), _ptr(k), _ptr(v), _ptr(positions), _ptr(cos_sin), int(cos_sin.shape[0]),
                                  _ptr(slot_mapping), int(k.shape[0]), int(q.shape[1]), _ptr(k_cache),
                                  _ptr(v_cache), ctypes.byref(desc), _ptr(q_out), _stream_ptr(stream))
    _check(st, "pkv_rope_kv_append")
    return q_out


def selftest_bounded_wait(limit_us: int, result=None, stream=None) -> None:
    """Enqueue the failure-path self-test (pkv_selftest_bounded_wait): a CTA laid
    out like the prefill kernel's waits on barriers that nothing completes; the
    producer warp gives up after ~limit_us and sets PKV_DEV_TIMEOUT, the other
    warps drain through the abort flag. `result`: optional device int32 [2]
    tensor (error word, warps that returned)."""
    if result is not None:
        import torch
        if not result.is_cuda or result.dtype != torch.int32 or result.numel() < 2 or not result.is_contiguous():
            raise ValueError("selftest_bounded_wait: result must be a contiguous int32 CUDA tensor of 2 entries")
    _check(lib().pkv_selftest_bounded_wait(int(limit_us), _ptr(result), _stream_ptr(stream)),
           "pkv_selftest_bounded_wait")


def device_status(stream=None) -> int:
    """OR of the device status bits since the last call (then cleared)."""
    code = ctypes.c_int32(0)
    _check(lib().pkv_get_device_status(ctypes.byref(code), _stream_ptr(stream)), "pkv_get_device_status")
    return int(code.value)


def set_kernel_timing(enable: bool):
    _check(lib().pkv_set_kernel_timing(1 if enable else 0), "pkv_set_kernel_timing")


def kernel_times(max_kernels: int = 32):
    """{kernel name: (launches, total ms)} recorded since the last call."""
    names = (ctypes.c_char_p * max_kernels)()
    launches = (ctypes.c_int32 * max_kernels)()
    total = (ctypes.c_double * max_kernels)()
    n = lib().pkv_kernel_times(names, launches, total, max_kernels)
    if n < 0:
        raise PagedKVError(n, "pkv_kernel_times")
    return {names[i].decode(): (int(launches[i]), float(total[i])) for i in range(n)}


# ---------------------------------------------------------------------------
# host page pool and prefix cache

class PagePool:
    """The library's host page pool (pkv_pool_*, pkv_prefix_*)."""

    def __init__(self, num_pages: int, page_size: int):
        self._h = ctypes.c_void_p()
        _check(lib().pkv_pool_create(int(num_pages), int(page_size), ctypes.byref(self._h)), "pkv_pool_create")
        self.num_pages, self.page_size = int(num_pages), int(page_size)

    def close(self):
        if self._h:
            lib().pkv_pool_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @staticmethod
    def _arr(xs):
        a = np.ascontiguousarray(np.asarray(xs, dtype=np.int32))
        return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))

    def alloc(self, n: int):
        a = np.zeros(max(n, 1), dtype=np.int32)
        _check(lib().pkv_pool_alloc(self._h, int(n), a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))), "pkv_pool_alloc")
        return [int(x) for x in a[:n]]

    def retain(self, pages):
        a, p = self._arr(pages)
        _check(lib().pkv_pool_retain(self._h, p, len(a)), "pkv_pool_retain")

    def release(self, pages):
        a, p = self._arr(pages)
        _check(lib().pkv_pool_release(self._h, p, len(a)), "pkv_pool_release")

    def free_count(self) -> int:
        return int(lib().pkv_pool_free_count(self._h))

    def refcount(self, page: int) -> int:
        r = lib().pkv_pool_refcount(self._h, int(page))
        if r < 0:
            raise PagedKVError(r, "pkv_pool_refcount")
        return int(r)

    def lookup(self, tokens, now: float, max_pages: int = 1 << 20):
        t, tp = self._arr(tokens if len(tokens) else [0])
        n_max = min(max_pages, len(tokens) // self.page_size)
        out = np.zeros(max(n_max, 1), dtype=np.int32)
        n = lib().pkv_prefix_lookup(self._h, tp, len(tokens), float(now),
                                    out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), int(n_max))
        if n < 0:
            raise PagedKVError(n, "pkv_prefix_lookup")
        return [int(x) for x in out[:n]]

    def insert(self, tokens, pages, now: float) -> int:
        t, tp = self._arr(tokens if len(tokens) else [0])
        a, ap = self._arr(pages if len(pages) else [0])
        n = lib().pkv_prefix_insert(self._h, tp, len(tokens), ap, len(pages), float(now))
        if n < 0:
            raise PagedKVError(n, "pkv_prefix_insert")
        return int(n)

    def evict(self, now: float, ttl: float, want_free: int = 0) -> int:
        n = lib().pkv_prefix_evict(self._h, float(now), float(ttl), int(want_free))
        if n < 0:
            raise PagedKVError(n, "pkv_prefix_evict")
        return int(n)

    def cache_size(self) -> int:
        return int(lib().pkv_prefix_size(self._h))

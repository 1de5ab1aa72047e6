"""Rotary position embedding — TEST INFRASTRUCTURE (CPU oracle, float64).

Q and K are rotated by position before attention (Helios blog, "torch.sdpa and
Flash Attention"; llm-serving-engine README, component table "RoPE from
scratch"). The pages do not say which variant; the reading taken is the
half-split form: pair i < d/2 of a head row joins x_i and x_{i+d/2}, rotated by
angle p * base**(-2 i / d).
"""
from __future__ import annotations

import numpy as np


def rope_angles(base: float, head_dim: int, positions) -> np.ndarray:
    """[len(positions), d/2] angles p * base**(-2 i / d) in float64."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    inv_freq = base ** (-2.0 * i / head_dim)
    return np.asarray(positions, dtype=np.float64)[:, None] * inv_freq[None, :]


def apply_rope(x: np.ndarray, positions, base: float) -> np.ndarray:
    """Rotate rows x [T, H, d] (any float dtype, widened exactly) at positions [T]."""
    x = np.asarray(x, dtype=np.float64)
    T, H, d = x.shape
    a = rope_angles(base, d, positions)[:, None, :]           # [T, 1, d/2]
    c, s = np.cos(a), np.sin(a)
    x1, x2 = x[..., : d // 2], x[..., d // 2:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def positions_of_tick(cu_seqlens_q, kv_lens) -> np.ndarray:
    """Position of every packed row: kv_len - q_len + i for row i of a sequence."""
    out = []
    for b in range(len(kv_lens)):
        q = int(cu_seqlens_q[b + 1]) - int(cu_seqlens_q[b])
        out += [int(kv_lens[b]) - q + i for i in range(q)]
    return np.array(out, dtype=np.int32)

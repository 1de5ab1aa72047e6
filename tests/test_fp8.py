"""FP8 (e4m3) KV cache: the oracle codec pinned to the format's fixed points,
and (GPU) the quantising append and attention over fp8 pages."""
import numpy as np

from oracle import fp8 as F


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


def test_dequantize_scales_per_head():
    codes = np.array([[[0x38, 0x40], [0x38, 0xB8]]], dtype=np.uint8)   # [1, 2 heads, 2]
    v = F.dequantize(codes, np.array([0.5, 3.0]))
    assert np.array_equal(v, [[[0.5, 1.0], [3.0, -3.0]]])

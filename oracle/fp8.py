"""Oracle: the FP8-E4M3 KV cache (decode, encode, the window write).

Test infrastructure only (see the package docstring).

Source: [TS] "One tree attention", FP8 paragraph. An FP8 KV cache is E4M3 and
unscaled: a stored byte is the value itself, with no per-tensor or per-head
scale. The window kernel widens the window's FP8 K/V to the model dtype after
loading them and takes the unquantized query.

E4M3 (the "fn" variant of the OCP 8-bit floating-point formats): one sign bit,
four exponent bits with bias 7, three mantissa bits.
  * exponent field e = 1..15: value (-1)^s * 2^(e - 7) * (1 + m / 8)
  * exponent field e = 0: subnormal, (-1)^s * 2^-6 * (m / 8)
  * S.1111.111 (0x7F, 0xFF) is NaN; there is no infinity, so the largest
    finite magnitude is 2^8 * 1.75 = 448 (0x7E).

Readings where the pages are silent:
  * rounding into E4M3 is to nearest, ties to even, and saturating
    (magnitudes past 448 store 448; NaN stays NaN). The pages give no cast
    mode. Saturation is the hardware conversion's mode, and a KV entry never
    comes near 448.
  * the window's rotated key is first rounded to the model dtype (bf16, as
    the bf16 cache stores it), then cast to E4M3. The value is taken as is.
"""
from __future__ import annotations

import numpy as np

from . import rope
from .attention import round_bf16, widen

E4M3_MAX = 448.0
E4M3_NAN = 0x7F


def decode_e4m3(codes) -> np.ndarray:
    """E4M3 bytes (uint8) -> fp64, exactly, from the field definition above."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = np.ldexp(1.0 + m / 8.0, e - 7)
    sub = np.ldexp(m / 8.0, -6)
    v = s * np.where(e == 0, sub, normal)
    return np.where((c & 0x7F) == 0x7F, np.nan, v)


def encode_e4m3(x) -> np.ndarray:
    """fp64 -> E4M3 bytes: round to nearest, ties to even, saturating at 448.

    Stated as the grid search it is: the representable magnitudes are the 127
    non-negative codes 0x00..0x7E, in increasing order; a magnitude takes the
    nearest one, and of two equally near the one whose code is even (the
    code's last bit is the mantissa's last bit). Beyond 448 the nearest is 448.
    """
    x = np.asarray(x, dtype=np.float64)
    grid = decode_e4m3(np.arange(0x7F, dtype=np.uint8))          # 0 .. 448, increasing
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.clip(np.searchsorted(grid, a, side="left"), 0, 0x7E)  # first grid value >= a
    lo = np.maximum(hi - 1, 0)
    d_lo = a - grid[lo]
    d_hi = grid[hi] - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(take_hi, hi, lo).astype(np.int64)
    code = np.where(a == grid[hi], hi, code)                       # exact values
    sign = np.where(np.signbit(x), 0x80, 0)
    out = (code | sign).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(E4M3_NAN), out).astype(np.uint8)


def window_kv_fp8(k_new, v_new, positions, theta: float):
    """The window write into an FP8 cache, per node row: K = e4m3(bf16(RoPE(k,
    position))), V = e4m3(v). k_new, v_new: [rows][Hkv][d] bf16 bits;
    positions: [rows]. Returns (k8, v8) uint8 [rows][Hkv][d]."""
    pos = np.asarray(positions, dtype=np.int64).reshape(-1)[:, None]
    k = round_bf16(rope.rotate(widen(k_new), pos, theta))
    return encode_e4m3(k), encode_e4m3(widen(v_new))

"""Pins for oracle.fp8 (the E4M3 KV cache): the format's fixed points, a
library routine on its whole code space, round-trip identity, the tie rule,
saturation, and the window write at position 0 (no rotation)."""
import numpy as np
import pytest

import oracle.fp8 as F
from oracle import rope as OR

torch = pytest.importorskip("torch")


def _torch_e4m3(x):
    """torch's own float8_e4m3fn cast (round to nearest even, no saturation:
    magnitudes from 464 up become NaN), as bytes."""
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_decode_fixed_points():
    """Values that follow from the field layout alone (1 sign, 4 exponent
    bits with bias 7, 3 mantissa bits, S.1111.111 = NaN)."""
    for code, val in [(0x00, 0.0), (0x38, 1.0), (0x3C, 1.5), (0x40, 2.0), (0xC0, -2.0), (0x7E, 448.0),
                      (0x08, 2.0 ** -6), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x30, 0.5), (0x77, 240.0)]:
        assert F.decode_e4m3(np.uint8(code)) == val, hex(code)
    assert np.signbit(F.decode_e4m3(np.uint8(0x80)))
    assert np.isnan(F.decode_e4m3(np.array([0x7F, 0xFF], np.uint8))).all()
    # every finite code is distinct and the 127 non-negative ones increase
    g = F.decode_e4m3(np.arange(0x7F, dtype=np.uint8))
    assert (np.diff(g) > 0).all()


def test_decode_matches_torch_on_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.tensor(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = F.decode_e4m3(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert (got[ok] == ref[ok]).all()
    assert (np.signbit(got[ok]) == np.signbit(ref[ok])).all()


def test_encode_round_trips_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert (F.encode_e4m3(F.decode_e4m3(codes)) == codes).all()


def test_encode_matches_torch_below_saturation():
    """In range the cast is torch's: random values, every midpoint between
    neighbouring codes (the ties) and points just beside them."""
    rng = np.random.default_rng(7)
    g = F.decode_e4m3(np.arange(0x7F, dtype=np.uint8))
    mid = (g[:-1] + g[1:]) / 2
    x = np.concatenate([rng.normal(0, 1, 4000), rng.normal(0, 60, 4000), rng.uniform(-2.0 ** -5, 2.0 ** -5, 2000),
                        mid, -mid, mid * (1 + 2.0 ** -20), mid * (1 - 2.0 ** -20), g, -g])
    x = x[np.abs(x) < 464]
    x = x.astype(np.float32).astype(np.float64)   # torch casts from float32
    assert (F.encode_e4m3(x) == _torch_e4m3(x)).all()


def test_encode_ties_to_even_and_saturates():
    # 1 + 1/16 lies halfway between 1 (0x38, even) and 1.125 (0x39): even wins
    assert F.encode_e4m3(1.0625) == 0x38
    # 1.1875 lies halfway between 1.125 (0x39) and 1.25 (0x3A): even wins
    assert F.encode_e4m3(1.1875) == 0x3A
    # half the smallest subnormal rounds to zero, three halves of it to 2^-9 * 2
    assert F.encode_e4m3(2.0 ** -10) == 0x00
    assert F.encode_e4m3(3 * 2.0 ** -10) == 0x02
    # saturation: everything past 448 stores 448 (torch would store NaN there)
    assert (F.encode_e4m3([464.0, 1000.0, 1e30, np.inf]) == 0x7E).all()
    assert (F.encode_e4m3([-464.0, -np.inf]) == 0xFE).all()
    assert F.encode_e4m3(np.nan) == 0x7F
    assert F.encode_e4m3(-0.0) == 0x80


def test_window_kv_fp8_at_position_zero_is_the_plain_cast():
    """At position 0 the rotation is the identity, so the window write
    reduces to torch's cast of the bf16 inputs (no value here nears 464)."""
    rng = np.random.default_rng(3)
    bits = (rng.normal(0, 1, (6, 2, 128)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    vbits = (rng.normal(0, 1, (6, 2, 128)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    k8, v8 = F.window_kv_fp8(bits, vbits, np.zeros(6, np.int64), 10000.0)
    as_f = lambda b: (b.astype(np.uint32) << 16).view(np.float32)
    assert (k8 == _torch_e4m3(as_f(bits))).all()
    assert (v8 == _torch_e4m3(as_f(vbits))).all()


def test_window_kv_fp8_rotates_before_the_cast():
    """Away from position 0 the key is the bf16 rotation, then the cast: the
    decoded key lies within one E4M3 step (relative 2^-3, plus half the
    subnormal spacing) of the exact rotation."""
    rng = np.random.default_rng(5)
    bits = (rng.normal(0, 1, (4, 1, 128)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    pos = np.array([1, 17, 300, 4097])
    k8, _ = F.window_kv_fp8(bits, bits, pos, 10000.0)
    exact = OR.rotate((bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64), pos[:, None], 10000.0)
    got = F.decode_e4m3(k8)
    assert (np.abs(got - exact) <= np.abs(exact) * 2.0 ** -3 + 2.0 ** -9).all()
    # position 1 changes the key: the cast really comes after the rotation
    k0, _ = F.window_kv_fp8(bits[:1], bits[:1], np.array([0]), 10000.0)
    assert (k8[:1] != k0).any()

"""Pins of the e4m3 KV-cache oracle (CPU).

The decoder against values fixed by the format (1, 448, 2^-6, 2^-9, NaN,
signed zero) and monotone over the finite codes; the encoder against a
brute-force nearest-value search over every finite code, with ties to the
even code, saturation above 448 and the sign of zero; encode(decode(c)) = c;
the quantisation error bound of 3 mantissa bits; quantise-on-commit writes
exactly the quantised rows and nothing else.
"""
import math

import numpy as np
import pytest

import oracle.fp8_oracle as f8
import oracle.verify_oracle as vo


def test_decode_fixed_values():
    assert f8.e4m3_decode(0x00) == 0.0 and math.copysign(1.0, f8.e4m3_decode(0x80)) < 0
    assert f8.e4m3_decode(0x38) == 1.0 and f8.e4m3_decode(0xB8) == -1.0
    assert f8.e4m3_decode(0x7E) == 448.0 and f8.e4m3_decode(0xFE) == -448.0
    assert f8.e4m3_decode(0x08) == 2.0 ** -6 and f8.e4m3_decode(0x01) == 2.0 ** -9
    assert f8.e4m3_decode(0x07) == 7 * 2.0 ** -9 and f8.e4m3_decode(0x39) == 1.125
    assert math.isnan(f8.e4m3_decode(0x7F)) and math.isnan(f8.e4m3_decode(0xFF))
    vals = [f8.e4m3_decode(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(vals, vals[1:])), "codes 0..126 increase"


def _nearest(x):
    """Brute force: the finite code nearest to x; ties to the even code; beyond 448 -> 448."""
    best, err = None, None
    for c in range(256):
        v = f8.e4m3_decode(c)
        if math.isnan(v) or (v == 0.0 and (c & 0x80) != (0x80 if math.copysign(1.0, x) < 0 else 0)):
            continue
        if (v < 0) != (x < 0) and v != 0.0:
            continue
        d = abs(v - x)
        if best is None or d < err or (d == err and c % 2 == 0 and best % 2 == 1):
            best, err = c, d
    if abs(x) > 448.0:
        best = 0xFE if x < 0 else 0x7E
    return best


def test_encode_matches_brute_force_nearest():
    rng = np.random.default_rng(0)
    xs = list(rng.normal(0, 1, 400)) + list(rng.normal(0, 100, 200)) + list(rng.normal(0, 0.01, 200))
    xs += [0.0, -0.0, 1.0625, 1.1875, 1.5 * 2.0 ** -9, 2.5 * 2.0 ** -9, 448.0, 456.0, 464.0, 1e6, -1e6, -460.0]
    for x in xs:
        assert f8.e4m3_encode(x) == _nearest(float(x)), x


def test_ties_go_to_the_even_code_and_overflow_saturates():
    assert f8.e4m3_encode(1.0625) == 0x38          # halfway 1.0 / 1.125 -> even 0x38
    assert f8.e4m3_encode(1.1875) == 0x3A          # halfway 1.125 / 1.25 -> even 0x3A
    assert f8.e4m3_encode(1.5 * 2.0 ** -9) == 0x02
    assert f8.e4m3_encode(500.0) == 0x7E and f8.e4m3_encode(-1e30) == 0xFE
    assert f8.e4m3_encode(-0.0) == 0x80 and f8.e4m3_encode(float("nan")) == 0x7F


def test_round_trip_of_every_finite_code():
    for c in range(256):
        v = f8.e4m3_decode(c)
        if not math.isnan(v):
            assert f8.e4m3_encode(v) == c


def test_quantisation_error_bound():
    rng = np.random.default_rng(1)
    x = rng.normal(0, 1.0, size=4000).astype(np.float32)
    scale = 0.02
    back = f8.dequantise(f8.quantise(x, scale), scale)
    normal = np.abs(x) / scale >= 2.0 ** -6
    rel = np.abs(back - x)[normal] / np.abs(x)[normal]
    assert rel.max() <= 2.0 ** -4 * (1 + 1e-6)       # half an ulp of a 3-bit mantissa


def test_commit_writes_exactly_the_quantised_rows():
    rng = np.random.default_rng(2)
    pool, L, n = 6, 21, 5
    kc = [rng.integers(0, 126, size=(pool, 4, 16, 256)).astype(np.uint8)]
    vc = [rng.integers(0, 126, size=(pool, 4, 16, 256)).astype(np.uint8)]
    kn = [rng.normal(0, 0.3, size=(n, 4, 256)).astype(np.float32)]
    vn = [rng.normal(0, 0.3, size=(n, 4, 256)).astype(np.float32)]
    table = np.array([[3, 0, 5, 1]])
    path = [[0, 2, 4]]
    ks, vs, ctx = f8.kv_commit_fp8(kc, vc, [0.01], [0.02], kn, vn, table, [L], [0, n], [3], path)
    assert ctx[0] == L + 3
    for i, node in enumerate(path[0]):
        pos = L + i
        page, slot = table[0, pos // 16], pos % 16
        np.testing.assert_array_equal(ks[0][page, :, slot], f8.quantise(kn[0][node], 0.01))
        np.testing.assert_array_equal(vs[0][page, :, slot], f8.quantise(vn[0][node], 0.02))
        ks[0][page, :, slot] = kc[0][page, :, slot]
        vs[0][page, :, slot] = vc[0][page, :, slot]
    np.testing.assert_array_equal(ks[0], kc[0])
    np.testing.assert_array_equal(vs[0], vc[0])

"""Pins of the oracle's number codecs against things other than itself.

* E4M3 decode: the format's defining values and torch's float8_e4m3fn cast.
* E4M3 encode: brute-force nearest-of-all-finite-codes search (ties to the
  even code), torch's float8_e4m3fn cast (|y| <= 448), exact round trips.
* bf16 / fp16 decode: numpy's and torch's casts over all 65536 patterns.
"""
import math

import numpy as np
import pytest
import torch

import oracle

FINITE_POS = np.arange(0, 0x7F)  # codes 0x00..0x7E (non-negative finite)


@pytest.fixture(scope="module")
def table():
    return oracle.e4m3_decode_all()


def test_decode_defining_values(table):
    # OCP E4M3: bias 7, 3 mantissa bits, S.1111.111 = NaN, no infinities.
    assert table[0x00] == 0.0 and math.copysign(1, table[0x80]) == -1.0
    assert table[0x01] == 2.0 ** -9  # smallest subnormal
    assert table[0x07] == 7 * 2.0 ** -9  # largest subnormal
    assert table[0x08] == 2.0 ** -6  # smallest normal
    assert table[0x38] == 1.0
    assert table[0x7E] == 448.0  # largest finite
    assert math.isnan(table[0x7F]) and math.isnan(table[0xFF])
    pos = table[FINITE_POS]
    assert np.all(np.diff(pos) > 0), "non-negative codes must increase with the code"
    np.testing.assert_array_equal(table[0x80:0xFF], -table[0x00:0x7F])


def test_decode_matches_torch_float8(table):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(np.isnan(ref), np.isnan(table))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(ref[ok], table[ok])


def brute_force_encode(y: np.ndarray, table) -> np.ndarray:
    """Nearest finite E4M3 value by exhaustive search; ties go to the code
    with an even mantissa (the even code, since codes are ordered)."""
    pos = table[FINITE_POS]
    a = np.abs(y.astype(np.float64))
    d = np.abs(a[:, None] - pos[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    # among (at most two) tied candidates prefer the even code
    even = (FINITE_POS % 2 == 0)[None, :]
    pick = np.where(cand & even, 1, 0) + np.where(cand, 1, 0)
    code = np.argmax(pick, axis=1).astype(np.uint8)
    sign = np.signbit(y).astype(np.uint8) << 7
    return code | sign


def oracle_encode_many(y):
    return np.array([oracle.e4m3_encode(float(v)) for v in y], dtype=np.uint8)


def all_bf16_in_range():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = (bits.astype(np.uint32) << 16).view(np.float32)
    keep = np.isfinite(vals) & (np.abs(vals) <= 448.0)
    return vals[keep]


def test_encode_brute_force_all_bf16(table):
    y = all_bf16_in_range()
    np.testing.assert_array_equal(oracle_encode_many(y), brute_force_encode(y, table))


def test_encode_brute_force_midpoints_and_neighbours(table):
    pos = table[FINITE_POS]
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)  # exact in fp32
    assert np.all(mids.astype(np.float64) == (pos[:-1] + pos[1:]) / 2)
    up = np.nextafter(mids, np.float32(np.inf))
    dn = np.nextafter(mids, np.float32(0))
    y = np.concatenate([mids, up, dn, -mids, -up, -dn])
    y = y[np.abs(y) <= 448]
    np.testing.assert_array_equal(oracle_encode_many(y), brute_force_encode(y, table))


def test_encode_brute_force_random_fp32(table):
    rng = np.random.default_rng(1234)
    # log-uniform magnitudes over the whole e4m3 range and below it
    mag = np.exp2(rng.uniform(-14, math.log2(448), size=40000)).astype(np.float32)
    y = np.where(rng.integers(0, 2, size=mag.size) == 0, -mag, mag).astype(np.float32)
    np.testing.assert_array_equal(oracle_encode_many(y), brute_force_encode(y, table))


def test_encode_matches_torch_float8():
    rng = np.random.default_rng(99)
    y = np.concatenate([all_bf16_in_range(),
                        rng.uniform(-448, 448, size=20000).astype(np.float32)])
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle_encode_many(y), ref)


def test_encode_round_trip(table):
    for c in list(range(0x00, 0x7F)) + list(range(0x80, 0xFF)):
        assert oracle.e4m3_encode(table[c]) == c


def test_bf16_decode_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32)
    ref = (bits << 16).view(np.float32)
    got = np.array([oracle.bf16_to_f32(int(b)) for b in bits], dtype=np.float32)
    np.testing.assert_array_equal(got.view(np.uint32)[np.isfinite(ref)],
                                  ref.view(np.uint32)[np.isfinite(ref)])
    # torch's bf16 cast agrees too (finite patterns)
    tb = torch.from_numpy(bits.astype(np.int32)).to(torch.int16).view(torch.bfloat16)
    tref = tb.to(torch.float32).numpy()
    fin = np.isfinite(tref)
    np.testing.assert_array_equal(got[fin], tref[fin])


def test_f16_decode_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle.f16_to_f32(int(b)) for b in bits], dtype=np.float32)
    fin = np.isfinite(ref)
    np.testing.assert_array_equal(got[fin], ref[fin])
    assert np.all(np.isinf(got[np.isinf(ref)]))
    assert np.all(np.isnan(got[np.isnan(ref)]))

"""Pins for the oracle's E4M3 encoder and decoder (OCP E4M3 format).

Expected values come from the hand-written golden table, torch's float8
dtype, and a brute-force nearest-code search -- never from the oracle.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.e4m3_ref import brute_force_encode, code_table, golden_codes


def test_decode_matches_golden_table():
    for c, v in golden_codes():
        got = oracle.e4m3_decode(c)
        if math.isnan(v):
            assert math.isnan(got), hex(c)
        else:
            assert got == v and math.copysign(1, got) == math.copysign(1, v), hex(c)


def test_decode_matches_library_dtype_for_all_codes():
    t = code_table()
    for c in range(256):
        got = oracle.e4m3_decode(c)
        if math.isnan(t[c]):
            assert math.isnan(got)
        else:
            assert got == t[c], hex(c)


def test_library_table_matches_golden():
    t = code_table()
    for c, v in golden_codes():
        assert (math.isnan(v) and math.isnan(t[c])) or t[c] == v


def test_encode_every_finite_code_round_trips():
    t = code_table()
    vals = np.array([t[c] for c in range(256) if not math.isnan(t[c])], np.float32)
    codes = np.array([c for c in range(256) if not math.isnan(t[c])], np.uint8)
    assert np.array_equal(oracle.e4m3_encode_array(vals), codes)


def test_encode_all_bf16_patterns_brute_force():
    bits = np.arange(65536, dtype=np.uint32)
    v = (bits << 16).view(np.float32)
    v = v[np.isfinite(v)]
    assert np.array_equal(oracle.e4m3_encode_array(v), brute_force_encode(v))


def test_encode_midpoints_and_neighbours():
    t = code_table()[:0x7F]
    mids = ((t[:-1] + t[1:]) / 2).astype(np.float32)   # 5 significant bits: exact in binary32
    assert np.array_equal(mids.astype(np.float64), (t[:-1] + t[1:]) / 2)
    up = np.nextafter(mids, np.float32(np.inf))
    dn = np.nextafter(mids, np.float32(0))
    above = np.array([448.0, 460.0, 463.99997, 464.0, 464.00003, 480.0, 1e4, 3.0e38], np.float32)
    v = np.concatenate([mids, up, dn, above])
    v = np.concatenate([v, -v])
    assert np.array_equal(oracle.e4m3_encode_array(v), brute_force_encode(v))


def test_encode_random_binary32_brute_force():
    rng = np.random.default_rng(1234)
    n = 200_000
    mag = np.exp2(rng.uniform(-24, 10, n)).astype(np.float32)
    sub = rng.uniform(0, 2.0 ** -5, n // 4).astype(np.float32)
    den = (rng.integers(1, 2 ** 23, n // 8, dtype=np.uint32)).view(np.float32)  # binary32 subnormals
    v = np.concatenate([mag, sub, den])
    v = v * np.where(rng.random(v.size) < 0.5, -1, 1).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode_array(v), brute_force_encode(v))


def test_encode_matches_library_cast_below_448():
    rng = np.random.default_rng(7)
    v = (rng.standard_normal(300_000) * np.exp2(rng.uniform(-12, 8, 300_000))).astype(np.float32)
    v = v[np.abs(v) < 448]
    lib = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode_array(v), lib)


@pytest.mark.parametrize("v,code", [(448.0, 0x7E), (1e30, 0x7E), (-1e30, 0xFE), (464.0, 0x7E),
                                    (-0.0, 0x80), (0.0, 0x00), (2.0 ** -10, 0x00),
                                    (2.0 ** -10 + 2.0 ** -30, 0x01), (-(2.0 ** -9), 0x81)])
def test_encode_special_values(v, code):
    assert oracle.e4m3_encode(v) == code

"""Pins for the oracle's number-format emulation (CPU only).

E4M3 / E2M1 / BF16 are checked against their format definitions (closed-form
code tables), against every rounding midpoint, and against two independent
implementations (torch dtype casts, and ml_dtypes where installed).
"""
import numpy as np
import pytest
import torch

from oracle import codecs as C


def test_e4m3_code_table_closed_form():
    vals = C.e4m3_decode_code(np.arange(256))
    assert vals[0x00] == 0.0
    assert vals[0x01] == 2.0 ** -9          # smallest subnormal
    assert vals[0x07] == 7 * 2.0 ** -9      # largest subnormal
    assert vals[0x08] == 2.0 ** -6          # smallest normal
    assert vals[0x38] == 1.0
    assert vals[0x39] == 1.125
    assert vals[0x7E] == 448.0              # largest finite
    assert np.isnan(vals[0x7F]) and np.isnan(vals[0xFF])
    assert vals[0xB8] == -1.0
    finite = vals[~np.isnan(vals)]
    assert len(finite) == 254
    assert np.max(finite) == 448.0 and np.min(finite) == -448.0


def test_e4m3_decode_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = C.e4m3_decode_code(np.arange(256))
    np.testing.assert_array_equal(np.isnan(ref), np.isnan(ours))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(ref[ok], ours[ok])


def test_e4m3_roundtrip_all_codes():
    codes = np.arange(256)
    vals = C.e4m3_decode_code(codes)
    ok = ~np.isnan(vals) & (codes != 0x80)
    np.testing.assert_array_equal(C.e4m3_encode_code(vals[ok]), codes[ok].astype(np.uint8))
    np.testing.assert_array_equal(C.e4m3(vals[ok]), vals[ok])


def _positive_grid(decode, ncodes):
    v = decode(np.arange(ncodes))
    v = v[~np.isnan(v)]
    return np.unique(v[v >= 0])


def test_e4m3_midpoints_ties_to_even():
    grid = _positive_grid(C.e4m3_decode_code, 128)
    lo, hi = grid[:-1], grid[1:]
    mid = (lo + hi) / 2
    got = C.e4m3(mid)
    lo_codes = C.e4m3_encode_code(lo).astype(np.int64)
    expect = np.where(lo_codes % 2 == 0, lo, hi)     # even mantissa LSB wins
    np.testing.assert_array_equal(got, expect)
    # just off the midpoint rounds to the nearer neighbour
    eps = (hi - lo) * 1e-6
    np.testing.assert_array_equal(C.e4m3(mid - eps), lo)
    np.testing.assert_array_equal(C.e4m3(mid + eps), hi)
    np.testing.assert_array_equal(C.e4m3(-mid), -expect)


def test_e4m3_saturates():
    x = np.array([448.0, 449.0, 463.9, 464.0, 470.0, 500.0, 1e6, -1e6, np.inf, -np.inf])
    np.testing.assert_array_equal(C.e4m3(x), [448, 448, 448, 448, 448, 448, 448, -448, 448, -448])
    assert np.isnan(C.e4m3(np.nan))


def test_e4m3_random_vs_torch_and_ml_dtypes():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-12, 6, 200000))).astype(np.float32)
    x = x[np.abs(x) < 440]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(C.e4m3(x.astype(np.float64)), ref)
    ml = pytest.importorskip("ml_dtypes")
    ref2 = x.astype(ml.float8_e4m3fn).astype(np.float64)
    np.testing.assert_array_equal(C.e4m3(x.astype(np.float64)), ref2)


def test_bf16_vs_torch():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-30, 30, 200000))).astype(np.float32)
    # include exact midpoints between bf16 neighbours
    bits = rng.integers(0, 2 ** 31, 5000, dtype=np.uint32) & 0x7FFF0000 | 0x8000
    mids = bits.view(np.float32)
    mids = mids[np.isfinite(mids)]
    x = np.concatenate([x, mids, -mids])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(C.bf16(x.astype(np.float64)), ref)


def test_e2m1_code_table_and_rounding():
    vals = C.e2m1_decode_code(np.arange(16))
    np.testing.assert_array_equal(vals[:8], [0, 0.5, 1, 1.5, 2, 3, 4, 6])
    np.testing.assert_array_equal(vals[8:], -np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6]))
    np.testing.assert_array_equal(C.e2m1_encode_code(vals[:8]), np.arange(8))
    # midpoints: ties to even (even = mantissa bit 0)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    np.testing.assert_array_equal(C.e2m1(mids), [0, 1, 1, 2, 2, 4, 4])
    np.testing.assert_array_equal(C.e2m1(np.array([6.0, 7.0, 100.0, -9.0])), [6, 6, 6, -6])


def test_e2m1_vs_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(100000) * 3).astype(np.float32)
    x = x[np.abs(x) < 6]
    ref = x.astype(ml.float4_e2m1fn).astype(np.float64)
    np.testing.assert_array_equal(C.e2m1(x.astype(np.float64)), ref)


def test_fp32_rounding():
    x = np.array([0.1, 1 / 3, 2.0 ** -140, 1e30])
    np.testing.assert_array_equal(C.fp32(x), x.astype(np.float32).astype(np.float64))

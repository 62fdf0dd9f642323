"""Pins for oracle/formats.py: printed value sets, library casts, closed forms."""

import numpy as np
import pytest
import torch

from oracle import formats
from tests.conftest import read_golden


def test_e2m1_value_set_matches_page():
    fx = read_golden("e2m1_values.txt")
    page = sorted(float(v) for v in fx["positive"])
    vals = formats.e2m1_decode(np.arange(16))
    mags = sorted(set(np.abs(vals).tolist()) - {0.0})
    assert mags == page
    # 16 states: 8 non-negative codes, each with a sign bit
    assert len(vals) == int(fx["states"][0])
    assert np.all(vals[:8] >= 0)
    # the sign bit negates (code 8 is negative zero)
    np.testing.assert_array_equal(vals[8:], -vals[:8])
    assert np.signbit(vals[8]) and vals[8] == 0.0
    # codes are ordered by magnitude (monotone grid)
    assert np.all(np.diff(vals[:8]) > 0)


def test_e2m1_encode_roundtrip_and_ties():
    codes = np.arange(16, dtype=np.uint8)
    enc = formats.e2m1_encode(formats.e2m1_decode(codes))
    # every code maps back to itself, except -0 which becomes +0
    expect = codes.copy()
    expect[8] = 0
    np.testing.assert_array_equal(enc, expect)
    fx = read_golden("e2m1_rne_ties.txt")
    for x, v in fx["_rows"]:
        got = formats.e2m1_decode(formats.e2m1_encode(np.float64(x)))
        assert got == float(v), (x, got, v)


def test_e2m1_encode_is_nearest_on_sweep():
    y = np.linspace(-8, 8, 64001)
    grid = np.unique(formats.e2m1_decode(np.arange(16)))
    q = formats.e2m1_decode(formats.e2m1_encode(y))
    best = np.min(np.abs(y[:, None] - grid[None, :]), axis=1)
    np.testing.assert_allclose(np.abs(y - q), best, rtol=0, atol=0)
    # tie points pick the even-mantissa code
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    c = formats.e2m1_encode(ties)
    assert np.all((c & 1) == 0)


def test_e4m3_decode_matches_torch_all_codes():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = formats.e4m3_decode(codes.numpy())
    nan = np.isnan(ref)
    np.testing.assert_array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    # closed forms: max 448, smallest subnormal 2^-9, NaN codes
    assert formats.e4m3_decode(0x7E) == 448.0
    assert formats.e4m3_decode(0x01) == 2.0 ** -9
    assert formats.e4m3_decode(0x08) == 2.0 ** -6


def test_e4m3_encode_matches_torch_cast():
    rng = np.random.default_rng(0)
    dense = np.concatenate([
        np.linspace(0, 448, 200001),
        np.exp(rng.uniform(np.log(1e-4), np.log(448), 200000)),
        formats.e4m3_decode(np.arange(127)),                      # exact points
        (formats.e4m3_decode(np.arange(126)) + formats.e4m3_decode(np.arange(1, 127))) / 2,  # ties
    ]).astype(np.float32)
    ref = torch.from_numpy(dense).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = formats.e4m3_encode(dense)
    np.testing.assert_array_equal(got, ref)
    # negative values: sign bit set
    np.testing.assert_array_equal(formats.e4m3_encode(-dense[1:1000]),
                                  ref[1:1000] | np.where(ref[1:1000] != 0, 0x80, 0))
    # saturation (satfinite): beyond 448 stays 448
    assert formats.e4m3_encode(np.float32(1e6)) == 0x7E
    assert formats.e4m3_encode(np.float32(470.0)) == 0x7E


def test_e8m0_and_ceil_log2():
    c = np.arange(255)
    np.testing.assert_array_equal(formats.e8m0_decode(c), np.ldexp(1.0, c - 127))
    assert np.isnan(formats.e8m0_decode(255))
    rng = np.random.default_rng(1)
    y = np.exp(rng.uniform(-60, 60, 100000)).astype(np.float32)
    e = formats.ceil_log2(y)
    y64 = y.astype(np.float64)
    assert np.all(np.ldexp(1.0, e - 1) < y64) and np.all(y64 <= np.ldexp(1.0, e))
    p = np.ldexp(np.float32(1.0), np.arange(-100, 100)).astype(np.float32)
    np.testing.assert_array_equal(formats.ceil_log2(p), np.arange(-100, 100))


def test_bf16_rne_matches_torch():
    rng = np.random.default_rng(2)
    x = rng.standard_normal(200000).astype(np.float32) * np.float32(3.0)
    # exact ties: 16 low bits == 0x8000, both parities of the kept lsb
    t = (rng.integers(0, 64, 2000, dtype=np.uint32) << 17) | np.uint32(0x3F008000)
    t2 = t | 0x10000
    x = np.concatenate([x, t.view(np.float32), t2.astype(np.uint32).view(np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(formats.bf16_bits(x), ref)
    np.testing.assert_array_equal(formats.bf16_value(ref),
                                  torch.from_numpy(x).to(torch.bfloat16).float().numpy())


@pytest.mark.parametrize("bad", [0.0])
def test_bf16_zero(bad):
    assert formats.bf16_bits(np.float32(bad)) == 0
    assert formats.bf16_bits(np.float32(-0.0)) == 0x8000

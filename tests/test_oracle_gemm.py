"""Pins for oracle/gemm.py: exact rational brute force and special cases."""

from fractions import Fraction

import numpy as np
import pytest

from oracle import formats, gemm, quantize


def _brute(a, codes, sc, fmt, g):
    """C[i, j] = g * sum_k A[i, k] * value(code[j, k]) * scale[j, k // G], exact."""
    group = 16 if fmt == "nvfp4" else 32
    m, k = a.shape
    n = codes.shape[0]
    dec_scale = formats.e4m3_decode if fmt == "nvfp4" else formats.e8m0_decode
    out = np.empty((m, n))
    for i in range(m):
        for j in range(n):
            acc = Fraction(0)
            for kk in range(k):
                w = Fraction(float(formats.e2m1_decode(codes[j, kk]))) * \
                    Fraction(float(dec_scale(sc[j, kk // group])))
                acc += Fraction(float(a[i, kk])) * w
            out[i, j] = float(Fraction(float(g)) * acc)
    return out


@pytest.mark.parametrize("fmt,m,n,k,g", [
    ("nvfp4", 3, 4, 64, 1.0),
    ("nvfp4", 1, 3, 48, 0.0123),
    ("mxfp4", 4, 2, 64, 1.0),
    ("mxfp4", 2, 3, 32, 1.0),
])
def test_gemm_matches_exact_rational(fmt, m, n, k, g):
    rng = np.random.default_rng(m * 100 + n * 10 + k)
    a = formats.bf16_round(rng.standard_normal((m, k)).astype(np.float32))
    w = formats.bf16_round((rng.standard_normal((n, k)) * 0.02).astype(np.float32))
    if fmt == "nvfp4":
        codes, sc = quantize.nvfp4_quantize(w, g)
    else:
        codes, sc = quantize.mxfp4_quantize(w)
    wq = gemm.dequantize(codes, sc, fmt)
    got = gemm.gemm(a, wq, g)
    exact = _brute(a, codes, sc, fmt, g)
    assert got.shape == (m, n)
    np.testing.assert_allclose(got, exact, rtol=1e-12, atol=1e-300)


def test_gemm_special_cases():
    rng = np.random.default_rng(7)
    n, k = 24, 128
    w = formats.bf16_round((rng.standard_normal((n, k)) * 0.02).astype(np.float32))
    codes, sc = quantize.nvfp4_quantize(w, 1.0)
    wq = gemm.dequantize(codes, sc, "nvfp4")
    # one-hot rows select weight columns exactly
    cols = np.array([0, 5, 77, 127])
    a = np.zeros((4, k), dtype=np.float32)
    a[np.arange(4), cols] = 1.0
    np.testing.assert_array_equal(gemm.gemm(a, wq, 1.0), wq[:, cols].T)
    # zero activations give zero
    assert np.all(gemm.gemm(np.zeros((3, k), np.float32), wq, 1.0) == 0)
    # all-ones activations give row sums
    np.testing.assert_allclose(gemm.gemm(np.ones((1, k), np.float32), wq, 2.0)[0], 2.0 * wq.sum(1), rtol=1e-15)
    # gemm_rows selects the same output columns as the full product
    a = formats.bf16_round(rng.standard_normal((5, k)).astype(np.float32))
    rows = np.array([3, 11, 23])
    np.testing.assert_array_equal(gemm.gemm_rows(a, codes, sc, "nvfp4", 1.0, rows),
                                  gemm.gemm(a, wq, 1.0)[:, rows])


def test_f16_dequant_bits_exact_and_pinned():
    """Every E2M1 code times every positive finite E4M3 scale is exact in
    binary16; spot values checked against their hand-computed bit patterns."""
    codes = np.tile(np.arange(16, dtype=np.uint8), 126 * 16)[: 126 * 16 * 16].reshape(126 * 16, 16)
    scales = np.repeat(np.arange(1, 127, dtype=np.uint8), 16).reshape(126 * 16, 1)
    bits = gemm.dequantize_f16_bits(codes, scales)
    wq = gemm.dequantize(codes, scales, "nvfp4")
    np.testing.assert_array_equal(bits.view(np.float16).astype(np.float64), wq)
    # code 0x1 (0.5) x scale 0x01 (2^-9) = 2^-10 -> binary16 0x1400;
    # code 0xF (-6) x scale 0x7E (448) = -2688 -> 0xE940; code 0x8 (-0) -> 0x8000
    c = np.array([[0x1, 0xF, 0x8] + [0] * 13], dtype=np.uint8)
    for sc, idx, want in [(0x01, 0, 0x1400), (0x7E, 1, 0xE940), (0x30, 2, 0x8000)]:
        b = gemm.dequantize_f16_bits(c, np.array([[sc]], dtype=np.uint8))
        assert int(b[0, idx]) == want, (sc, idx, hex(int(b[0, idx])))

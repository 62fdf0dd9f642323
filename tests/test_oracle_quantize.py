"""Pins for oracle/quantize.py: hand-worked blocks, invariants, special cases.

Extreme inputs (all-zero, huge and very skewed blocks) follow the testing
advice of "FP4 GEMM on Rubin/Blackwell with CUTLASS", section 7.
"""

import numpy as np
import pytest

from oracle import formats, gemm, quantize
from tests.conftest import read_golden

# largest distance from a grid point to the midpoint of its neighbours
_HALF_GAP = {0.0: 0.25, 0.5: 0.25, 1.0: 0.25, 1.5: 0.25, 2.0: 0.5, 3.0: 0.5, 4.0: 1.0, 6.0: 1.0}


def _f32(v):
    return np.array([float(x) for x in v], dtype=np.float32)


def test_nvfp4_hand_worked_block():
    fx = read_golden("nvfp4_block_example.txt")
    x = _f32(fx["x"])[None, :]
    codes, sc = quantize.nvfp4_quantize(x, 1.0)
    assert sc.tolist() == [[int(fx["scale"][0], 16)]]
    assert codes[0].tolist() == [int(c) for c in fx["codes"]]
    packed = quantize.pack_codes(codes)
    assert packed[0].tolist() == [int(b, 16) for b in fx["packed"]]
    np.testing.assert_array_equal(quantize.unpack_codes(packed), codes)
    wq = gemm.dequantize(codes, sc, "nvfp4")
    np.testing.assert_array_equal(wq[0], _f32(fx["wq"]).astype(np.float64))
    # with g = 0.5: t = 1.5 / (6 * 0.5) = 0.5 -> E4M3 0x30, d = 0.5 * 0.5 = 0.25,
    # so the codes are the same and the block scale doubles
    codes2, sc2 = quantize.nvfp4_quantize(x, 0.5)
    assert sc2.tolist() == [[0x30]]
    np.testing.assert_array_equal(codes2, codes)


def test_mxfp4_hand_worked_blocks():
    fx = read_golden("mxfp4_block_example.txt")
    x = np.stack([_f32(fx["a_x"]), _f32(fx["b_x"])])
    codes, sc = quantize.mxfp4_quantize(x)
    assert sc[:, 0].tolist() == [int(fx["a_scale"][0]), int(fx["b_scale"][0])]
    assert codes[0].tolist() == [int(c) for c in fx["a_codes"]]
    assert codes[1].tolist() == [int(c) for c in fx["b_codes"]]


def _weights(n, k, seed=0):
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((n, k)) * 0.02).astype(np.float32)
    w[0, :] = 0.0                                              # all-zero row
    w[1, :] = formats.bf16_round(rng.standard_normal(k).astype(np.float32) * 3e4)  # huge
    w[2, :] = 1e-6                                             # tiny
    w[2, ::16] = 5.0                                           # very skewed blocks
    w[3, :] = -0.0
    return formats.bf16_round(w)


@pytest.mark.parametrize("g", [1.0, "amax"])
def test_nvfp4_invariants(g):
    w = _weights(40, 512)
    if g == "amax":
        g = quantize.nvfp4_global_scale(w)
    g = np.float32(g)
    codes, sc = quantize.nvfp4_quantize(w, g)
    assert codes.shape == w.shape and sc.shape == (40, 512 // 16)
    # positive finite scales, no negative-zero codes
    assert np.all(sc != 0) and np.all(sc & 0x80 == 0) and np.all(sc != 0x7F)
    assert not np.any(codes == 0x8) and np.all(codes < 16)
    d = formats.e4m3_decode(sc).astype(np.float32) * g
    y = w.reshape(40, -1, 16) / d[..., None]
    q = formats.e2m1_decode(codes).reshape(y.shape)
    mag = np.abs(q)
    half = np.vectorize(_HALF_GAP.get)(mag)
    inside = np.abs(y) <= 6.0
    assert np.all(np.abs(y - q)[inside] <= half[inside])
    assert np.all(mag[~inside] == 6.0)
    assert np.all((np.sign(q) == np.sign(y)) | (q == 0))
    # scale tightness: value(sc) * g * 6 is amax to within half an E4M3 step
    amax = np.abs(w.reshape(40, -1, 16)).max(-1).astype(np.float64)
    t = amax / (6.0 * float(g))
    normal = (t >= 2.0 ** -6) & (t <= 448.0)
    rel = formats.e4m3_decode(sc)[normal] / t[normal]
    assert np.all(np.abs(rel - 1.0) <= 2.0 ** -4 + 1e-6)
    # idempotence: the dequantised weights re-encode to the same codes
    wq = gemm.dequantize(codes, sc, "nvfp4").astype(np.float32) * g
    re = formats.e2m1_encode(wq.reshape(y.shape) / d[..., None]).reshape(codes.shape)
    np.testing.assert_array_equal(re, codes)
    # special cases: an all-zero block gets codes 0 and the smallest scale
    assert np.all(codes[0] == 0) and np.all(sc[0] == 0x01)
    assert np.all(codes[3] == 0)


def test_nvfp4_global_scale_hand_worked():
    """Values worked by hand in tests/golden/nvfp4_global_scale.txt."""
    rows = read_golden("nvfp4_global_scale.txt")["_rows"]
    assert len(rows) >= 5
    for amax_txt, bits_txt in rows:
        amax = float(amax_txt)
        # a small row whose largest magnitude is |amax| (the entry keeps its sign)
        w = np.array([[amax, 0.25 * amax, -0.5 * abs(amax), 0.0]], dtype=np.float32)
        g = quantize.nvfp4_global_scale(w)
        assert isinstance(g, np.float32), type(g)
        assert int(np.asarray(g).view(np.uint32)) == int(bits_txt, 16), (amax, hex(int(np.asarray(g).view(np.uint32))))


def test_nvfp4_exact_grid_block_and_saturation():
    s = 2.0 ** -3
    x = np.array([[6 * s, -6 * s] + [s * v for v in (0.5, 1, 1.5, 2, 3, 4, -0.5, -1, -1.5, -2, -3, -4, 0, 6)]],
                 dtype=np.float32)
    codes, sc = quantize.nvfp4_quantize(x, 1.0)
    assert sc[0, 0] == formats.e4m3_encode(np.float32(s))
    np.testing.assert_array_equal(formats.e2m1_decode(codes[0]) * s, x[0])
    assert codes[0, 0] == 7 and codes[0, 1] == 15
    # scale saturation: t above 448 clamps the scale, codes saturate at 6
    big = np.full((1, 16), 3.0e4, dtype=np.float32)
    codes, sc = quantize.nvfp4_quantize(big, 1.0)
    assert sc[0, 0] == 0x7E and np.all(codes == 7)


def test_mxfp4_invariants():
    w = _weights(40, 512, seed=3)
    codes, sc = quantize.mxfp4_quantize(w)
    assert sc.shape == (40, 512 // 32)
    assert not np.any(codes == 0x8)
    blocks = w.reshape(40, -1, 32).astype(np.float64)
    amax = np.abs(blocks).max(-1)
    scale = formats.e8m0_decode(sc)
    live = amax >= 1e-8
    ratio = amax[live] / scale[live]
    eps = 2.0 ** -22
    assert np.all(ratio > 3 * (1 - eps)) and np.all(ratio <= 6 * (1 + eps))
    # x / 2^e is exact; codes are its nearest grid points (ties even)
    y = blocks / scale[..., None]
    q = formats.e2m1_decode(codes).reshape(y.shape)
    half = np.vectorize(_HALF_GAP.get)(np.abs(q))
    assert np.all(np.abs(y - q) <= half)
    wq = gemm.dequantize(codes, sc, "mxfp4")
    np.testing.assert_array_equal(formats.e2m1_encode(wq.reshape(y.shape) / scale[..., None]).reshape(codes.shape),
                                  codes)
    # all-zero block: codes 0, scale 2^ceil(log2(1e-8/6)) = 2^-29
    assert np.all(codes[0] == 0) and np.all(sc[0] == 127 - 29)


def test_dequant_exact_in_bf16():
    w = _weights(16, 256, seed=5)
    for fmt, q in (("nvfp4", lambda x: quantize.nvfp4_quantize(x, 1.0)),
                   ("mxfp4", quantize.mxfp4_quantize)):
        codes, sc = q(w)
        bits = gemm.dequantize_bf16_bits(codes, sc, fmt)   # raises if inexact
        back = formats.bf16_value(bits).astype(np.float64)
        np.testing.assert_array_equal(back, gemm.dequantize(codes, sc, fmt))


def test_pack_layout():
    codes = np.array([[1, 2, 0xF, 0x0, 7, 8]], dtype=np.uint8)
    assert quantize.pack_codes(codes).tolist() == [[0x21, 0x0F, 0x87]]
    rng = np.random.default_rng(9)
    c = rng.integers(0, 16, (7, 64)).astype(np.uint8)
    np.testing.assert_array_equal(quantize.unpack_codes(quantize.pack_codes(c)), c)

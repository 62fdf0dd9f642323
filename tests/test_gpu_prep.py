"""GPU quantiser, repack and dequant hook vs the oracle (bit-exact)."""

import numpy as np
import pytest
import torch

from fp4_weight_only_gb300 import synth
from oracle import formats, gemm, quantize
from tests.gpu_util import bf16_bits, oracle_quantize, to_device_packed

pytestmark = pytest.mark.gpu


def _extreme_weights(n, k, seed):
    w = synth.weights(n, k, seed=seed)
    w[0] = 0.0                                   # all-zero row
    w[1] = (torch.randn(k) * 3e4).to(torch.bfloat16)  # huge values
    w[2] = 1e-6
    w[2, ::16] = 5.0                             # very skewed blocks
    w[3, 5] = -0.0
    return w


@pytest.mark.parametrize("fmt,g", [("nvfp4", 1.0), ("nvfp4", "amax"), ("mxfp4", 1.0)])
@pytest.mark.parametrize("n,k", [(128, 128), (384, 1024), (77, 96)])
def test_quantize_matches_oracle(cuda_lib, fmt, g, n, k):
    if fmt == "mxfp4" and k % 32:
        pytest.skip("k % 32")
    w = _extreme_weights(n, k, seed=n + k)
    wd = w.cuda()
    if g == "amax":
        amax = cuda_lib.absmax(wd).item()
        assert amax == float(np.abs(w.float().numpy()).max())
        g = cuda_lib.nvfp4_global_scale(amax)
        assert np.float32(g) == quantize.nvfp4_global_scale(w.float().numpy())
    wp, sp = cuda_lib.quantize(wd, fmt, g)
    codes, scales = oracle_quantize(w, fmt, g)
    np.testing.assert_array_equal(sp.cpu().numpy(), scales)
    np.testing.assert_array_equal(wp.cpu().numpy(), quantize.pack_codes(codes))


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("n,k", [(128, 128), (256, 512), (1024, 1024)])
def test_repack_dequant_bitexact(cuda_lib, fmt, n, k):
    w = _extreme_weights(n, k, seed=3 * n + k)
    codes, scales = oracle_quantize(w, fmt, 1.0)
    # also exercise every code value, including negative zero (decodes to -0.0)
    codes[5, :16] = np.arange(16)
    wp, sp = to_device_packed(codes, scales)
    rep = cuda_lib.repack(wp, sp, fmt)
    nchunks = (n // 128) * (k // 128)
    flag_bytes = 16 if fmt == "mxfp4" else 0      # MXFP4: per-chunk flag field
    assert rep.numel() == n * k // 2 + scales.size + nchunks * flag_bytes
    # the repack permutes bits inside 32-bit code words and moves scale bytes:
    # the number of set bits and the multiset of scale bytes are kept
    sbytes = 1024 if fmt == "nvfp4" else 512
    r = rep.cpu().numpy().reshape(nchunks, 8192 + sbytes + flag_bytes)
    packed = quantize.pack_codes(codes)
    popcount = lambda x: int(np.unpackbits(np.ascontiguousarray(x).view(np.uint8)).sum())
    assert popcount(r[:, : 8192 + sbytes]) == popcount(packed) + popcount(scales)
    scale_part = r[:, 8192 : 8192 + sbytes]
    assert sorted(scale_part.reshape(-1).tolist()) == sorted(scales.reshape(-1).tolist())
    if fmt == "mxfp4":
        # flag byte 0: every E8M0 code of the (128-row tile, 128-k stage)
        # chunk is <= 128; bytes 1..15 zero.  Chunks are tile-major.
        blocks = scales.reshape(n // 128, 128, k // 128, 4)
        expect_flag = (blocks <= 128).all(axis=(1, 3)).reshape(-1).astype(np.uint8)
        np.testing.assert_array_equal(r[:, 8192 + sbytes], expect_flag)
        assert not r[:, 8192 + sbytes + 1 :].any()
        if n >= 256:   # row 1's huge values make the first tile take the two-multiply decode
            assert expect_flag.any() and not expect_flag.all()
    out = cuda_lib.dequant(rep, n, k, fmt)
    torch.cuda.synchronize()
    expect = gemm.dequantize_bf16_bits(codes, scales, fmt)
    got = bf16_bits(out)
    bad = np.argwhere(got != expect)
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:4].tolist()}"


def test_dequant_all_e4m3_scales(cuda_lib):
    """Every positive finite E4M3 scale (subnormals included) with every code."""
    n, k = 128, 128 * 16
    rng = np.random.default_rng(11)
    codes = rng.integers(0, 16, (n, k)).astype(np.uint8)
    scales = np.tile(np.arange(1, 127, dtype=np.uint8), (n * k // 16) // 126 + 1)[: n * k // 16]
    scales = scales.reshape(n, k // 16)
    wp, sp = to_device_packed(codes, scales)
    rep = cuda_lib.repack(wp, sp, "nvfp4")
    got = bf16_bits(cuda_lib.dequant(rep, n, k, "nvfp4"))
    np.testing.assert_array_equal(got, gemm.dequantize_bf16_bits(codes, scales, "nvfp4"))


def test_dequant_mx_scale_range(cuda_lib):
    """E8M0 codes 7..247 (scales 2^-120..2^120) with every FP4 code."""
    n, k = 128, 128 * 8
    rng = np.random.default_rng(12)
    codes = rng.integers(0, 16, (n, k)).astype(np.uint8)
    scales = rng.integers(7, 248, (n, k // 32)).astype(np.uint8)
    wp, sp = to_device_packed(codes, scales)
    rep = cuda_lib.repack(wp, sp, "mxfp4")
    got = bf16_bits(cuda_lib.dequant(rep, n, k, "mxfp4"))
    np.testing.assert_array_equal(got, gemm.dequantize_bf16_bits(codes, scales, "mxfp4"))


def test_dequant_mx_fast_path_scale_range(cuda_lib):
    """E8M0 codes 0..128 (every chunk takes the one-multiply decode), with
    the boundary codes 0 (2^-127) and 128 (2^1) in every chunk."""
    n, k = 256, 128 * 8
    rng = np.random.default_rng(13)
    codes = rng.integers(0, 16, (n, k)).astype(np.uint8)
    scales = rng.integers(0, 129, (n, k // 32)).astype(np.uint8)
    scales[::7, ::4] = 0
    scales[3::7, 1::4] = 128
    wp, sp = to_device_packed(codes, scales)
    rep = cuda_lib.repack(wp, sp, "mxfp4")
    r = rep.cpu().numpy().reshape(-1, 8192 + 512 + 16)
    assert r[:, 8192 + 512].all()
    got = bf16_bits(cuda_lib.dequant(rep, n, k, "mxfp4"))
    np.testing.assert_array_equal(got, gemm.dequantize_bf16_bits(codes, scales, "mxfp4"))

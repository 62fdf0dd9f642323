"""NVFP4 / MXFP4 weight quantisers and the two-per-byte packing.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The quantiser is not part of the GEMM, but the GEMM consumes its codes, so it
is fixed here.  Its steps follow the pages:

* block scaling by the block's largest magnitude ("max-abs scaling"), the
  article "FP4 GEMM on Rubin/Blackwell with CUTLASS", section 2.2;
* a floor on the block maximum, ``max(amax, 1e-8)``, so that all-zero (for
  instance padding) blocks do not get a zero scale -- same article, section
  5.2;
* positive scales and no negative-zero codes, the precondition of Petit's
  offline weight transform -- Petit PyPI page, "Known limitations";
* NVFP4 groups of 16 elements with one FP8 scale (Petit blog, "Detailed
  performance analysis"), plus a per-tensor FP32 global scale ``g``;
* MXFP4 groups of 32 elements with an E8M0 power-of-two scale
  ``2^ceil(log2(amax/6))`` and round-to-nearest-even codes.

Precision: the pages do not say in which precision the scale and the division
are computed.  Because these floating-point steps decide integer codes, they
are taken in IEEE binary32 (numpy float32 operations, each correctly
rounded), the precision of the CUDA quantiser; the comparisons that pick the
codes are then exact.
"""

import numpy as np

from . import formats

NVFP4_GROUP = 16
MXFP4_GROUP = 32
_AMAX_FLOOR = np.float32(1e-8)


def nvfp4_global_scale(w):
    """Per-tensor FP32 global scale ``amax(|W|) / (6 * 448)`` (binary32)."""
    amax = np.float32(np.abs(np.asarray(w, dtype=np.float32)).max())
    return np.float32(amax / np.float32(6.0 * 448.0))


def nvfp4_quantize(w, global_scale=1.0):
    """Quantise ``w`` [n, k] (BF16 values) to NVFP4.

    Per row and 16-element block j:
      amax = max |x|
      t    = max(amax, 1e-8) / (6 * g)                  (binary32)
      sc   = E4M3(t), round-to-nearest-even, saturating; a zero code becomes
             0x01 (2^-9) so every scale is positive
      d    = value(sc) * g                              (binary32)
      code = E2M1(x / d), nearest grid point, ties to even, saturating at 6
    Returns (codes uint8 [n, k] with values 0..15, scales uint8 [n, k/16]).
    """
    w = np.asarray(w, dtype=np.float32)
    n, k = w.shape
    if k % NVFP4_GROUP:
        raise ValueError("k must be a multiple of 16")
    blocks = w.reshape(n, k // NVFP4_GROUP, NVFP4_GROUP)
    g = np.float32(global_scale)
    amax = np.abs(blocks).max(axis=-1)
    t = np.maximum(amax, _AMAX_FLOOR) / (np.float32(6.0) * g)
    sc = formats.e4m3_encode(t)
    sc = np.where(sc == 0, np.uint8(1), sc).astype(np.uint8)
    d = formats.e4m3_decode(sc).astype(np.float32) * g
    y = blocks / d[..., None]
    codes = formats.e2m1_encode(y)
    return codes.reshape(n, k), sc


def mxfp4_quantize(w):
    """Quantise ``w`` [n, k] (BF16 values) to MXFP4.

    Per row and 32-element block j:
      y    = max(amax, 1e-8) / 6                        (binary32)
      e    = ceil(log2 y), exact, clamped so that c = e + 127 is in [0, 254]
      code = E2M1(x / 2^e), nearest grid point, ties to even
    Returns (codes uint8 [n, k], scales uint8 [n, k/32] holding c).
    """
    w = np.asarray(w, dtype=np.float32)
    n, k = w.shape
    if k % MXFP4_GROUP:
        raise ValueError("k must be a multiple of 32")
    blocks = w.reshape(n, k // MXFP4_GROUP, MXFP4_GROUP)
    amax = np.abs(blocks).max(axis=-1)
    y = np.maximum(amax, _AMAX_FLOOR) / np.float32(6.0)
    e = formats.ceil_log2(y)
    c = np.clip(e + 127, 0, 254)
    e = c - 127
    q = np.ldexp(blocks, (-e)[..., None].astype(np.int32)).astype(np.float32)
    codes = formats.e2m1_encode(q)
    return codes.reshape(n, k), c.astype(np.uint8)


def pack_codes(codes):
    """Two codes per byte: element 2j in the low nibble, 2j+1 in the high."""
    codes = np.asarray(codes, dtype=np.uint8)
    if codes.shape[-1] % 2:
        raise ValueError("k must be even")
    return (codes[..., 0::2] & 0xF) | ((codes[..., 1::2] & 0xF) << 4)


def unpack_codes(packed):
    """Inverse of :func:`pack_codes`."""
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out

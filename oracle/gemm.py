"""Exact dequantisation and the FP64 reference product.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The method (Petit blog, "Efficient dequantization via preprocessing"; Petit
PyPI page, "Features") multiplies BF16 activations by FP4 weights that are
turned back into BF16 before they meet the matrix unit.  A dequantised weight
is ``code * block_scale``: an E2M1 value (at most 2 significant bits) times an
E4M3 (4 bits) or E8M0 (1 bit) scale, so it has at most 5 significant bits and
is exactly a BF16 number for every E4M3 scale and for E8M0 exponents within
+-120.  The NVFP4 global scale is applied to the product, not to the weights.

The reference product is the plain definition

    C[i, j] = g * sum_k A[i, k] * Wq[j, k]        (W stored [n, k], k-major)

evaluated in float64 with a library matrix product.  Each term is exact in
float64 (8 + 5 significant bits); only the summation rounds.
"""

import numpy as np

from . import formats

_GROUP = {"nvfp4": 16, "mxfp4": 32}


def scale_values(scales, fmt):
    """Decoded block scales (float64)."""
    if fmt == "nvfp4":
        return formats.e4m3_decode(scales)
    if fmt == "mxfp4":
        return formats.e8m0_decode(scales)
    raise ValueError(fmt)


def dequantize(codes, scales, fmt):
    """Wq[n, k] = value(code[n, k]) * scale[n, k // group], float64, exact."""
    codes = np.asarray(codes)
    vals = formats.e2m1_decode(codes)
    s = scale_values(scales, fmt)
    return vals * np.repeat(s, _GROUP[fmt], axis=-1)


def dequantize_bf16_bits(codes, scales, fmt):
    """BF16 bit patterns of :func:`dequantize`; raises if any is inexact."""
    wq = dequantize(codes, scales, fmt)
    f32 = wq.astype(np.float32)
    bits = formats.bf16_bits(f32)
    back = formats.bf16_value(bits).astype(np.float64)
    same = (back == wq) | (np.isnan(back) & np.isnan(wq))
    if not np.all(same):
        raise ArithmeticError("dequantised weight not exactly representable in BF16")
    # keep the sign of zero (a negative-zero code decodes to -0.0)
    return bits


def dequantize_f16_bits(codes, scales):
    """IEEE binary16 bit patterns of the NVFP4 :func:`dequantize` (the FP16-
    activation variant's operand, Petit blog "Introduction": FP16/BF16
    activations); raises if any value is inexact in binary16."""
    wq = dequantize(codes, scales, "nvfp4")
    h = wq.astype(np.float16)
    if not np.all(h.astype(np.float64) == wq):
        raise ArithmeticError("dequantised weight not exactly representable in FP16")
    return h.view(np.uint16)


def gemm(a, wq, global_scale=1.0):
    """C = g * A . Wq^T in float64.  ``a`` [m, k], ``wq`` [n, k]."""
    a64 = np.asarray(a, dtype=np.float64)
    w64 = np.asarray(wq, dtype=np.float64)
    return float(global_scale) * (a64 @ w64.T)


def gemm_rows(a, codes, scales, fmt, global_scale=1.0, rows=None):
    """Reference output columns C[:, rows] computed from those weight rows only.

    Used to check sampled outputs of full-size problems without
    dequantising the whole weight matrix.
    """
    codes = np.asarray(codes)
    scales = np.asarray(scales)
    if rows is not None:
        codes = codes[rows]
        scales = scales[rows]
    return gemm(a, dequantize(codes, scales, fmt), global_scale)

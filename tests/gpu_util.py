"""Helpers shared by the GPU tests: oracle-side preparation and comparison.

Expected values always come from ``oracle/`` on the CPU; the CUDA path only
ever receives the oracle's codes/scales (or is checked to reproduce them).
"""

import numpy as np
import torch

from oracle import formats, gemm, quantize

# GEMM parity bounds: max|C - ref| <= 1e-2 max|ref| and rel-L2 <= 4e-3 (the BF16 output
# rounding alone gives about 1e-3 rel-L2)
MAX_ABS_REL = 1e-2
REL_L2 = 4e-3


def oracle_quantize(w_bf16, fmt, g=1.0):
    """(codes [n,k], scales) from the oracle, for BF16 weights (torch CPU)."""
    w = w_bf16.float().numpy()
    if fmt == "nvfp4":
        return quantize.nvfp4_quantize(w, g)
    return quantize.mxfp4_quantize(w)


def to_device_packed(codes, scales, device="cuda"):
    wp = torch.from_numpy(np.ascontiguousarray(quantize.pack_codes(codes))).to(device)
    sp = torch.from_numpy(np.ascontiguousarray(scales)).to(device)
    return wp, sp


def oracle_reference(a_bf16, codes, scales, fmt, g=1.0, rows=None):
    a = a_bf16.float().numpy()
    return gemm.gemm_rows(a, codes, scales, fmt, g, rows)


def compare(c_gpu, ref):
    """Returns (max_abs_err / max|ref|, rel_l2) of a BF16 result vs FP64 ref."""
    c = c_gpu.float().cpu().numpy().astype(np.float64)
    assert c.shape == ref.shape, (c.shape, ref.shape)
    assert np.all(np.isfinite(c))
    err = c - ref
    denom = max(np.abs(ref).max(), 1e-300)
    l2 = np.linalg.norm(ref)
    rel_l2 = np.linalg.norm(err) / l2 if l2 > 0 else np.linalg.norm(err)
    return np.abs(err).max() / denom, rel_l2


def assert_parity(c_gpu, ref, what=""):
    mx, l2 = compare(c_gpu, ref)
    assert mx <= MAX_ABS_REL and l2 <= REL_L2, f"{what}: max-abs/max|ref| {mx:.3e}, rel-L2 {l2:.3e}"
    return mx, l2


def bf16_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)

"""Number formats of the FP4 weight-only GEMM, written from their definitions.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

* E2M1 ("FP4"): 1 sign bit, 2 exponent bits, 1 mantissa bit.  The article
  "FP4 GEMM on Rubin/Blackwell with CUTLASS" (mhpq.cn), section 2.1, lists the
  non-zero positive values 0.5, 1, 1.5, 2, 3, 4, 6 and says a value is mapped
  to the nearest grid point; with the sign and zero the format has 16 states.
  The bit encoding below (exponent bias 1, exponent field 0 = subnormal) is the
  one that reproduces exactly that value set.  Ties between two grid points go
  to the point whose mantissa bit is 0 (round-half-to-even); magnitudes above
  6 saturate to 6.
* E4M3FN: the FP8 block-scale type of NVFP4 (the Petit blog says "16 elements
  share one FP8 scale", section "Detailed performance analysis"; E4M3 with a
  448 maximum is the reading).  Bias 7, no infinities, 0x7F/0xFF are NaN,
  subnormal step 2^-9, max 448.  Encoding is round-to-nearest-even with
  saturation to +-448.
* E8M0: the MXFP4 block scale, an unsigned biased exponent 2^(c-127); 0xFF is
  NaN.
* BF16: the top 16 bits of an IEEE binary32; conversion from binary32 is
  round-to-nearest-even on the bit pattern.
"""

import numpy as np

E2M1_CODES = np.arange(16, dtype=np.uint8)


# ---------------------------------------------------------------- E2M1 (FP4)
def e2m1_decode(code):
    """Value of each 4-bit E2M1 code (float64).  Code 0x8 decodes to -0.0."""
    code = np.asarray(code).astype(np.int64)
    sign = (code >> 3) & 1
    exp = (code >> 1) & 3
    man = code & 1
    normal = np.ldexp(1.0 + 0.5 * man, exp - 1)      # 2^(e-1) * (1 + m/2)
    subnormal = 0.5 * man                             # e == 0: m * 2^0 * 1/2
    mag = np.where(exp == 0, subnormal, normal).astype(np.float64)
    return np.where(sign == 1, -mag, mag)


def e2m1_encode(y, chunk=1 << 20):
    """Nearest E2M1 code to each value of ``y`` (exact comparison in float64).

    Ties go to the even-mantissa neighbour; magnitudes beyond 6 saturate to
    6 (the nearest grid point).  A result of magnitude zero always gets code
    0x0 (never the negative zero 0x8), as the Petit PyPI page ("Known
    limitations") requires of quantised weights.
    """
    y = np.asarray(y, dtype=np.float64)
    flat = y.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint8)
    grid = e2m1_decode(np.arange(8))                  # 0, .5, 1, 1.5, 2, 3, 4, 6
    even = (np.arange(8) & 1) == 0
    for lo in range(0, flat.size, chunk):
        v = flat[lo:lo + chunk]
        # saturate first: beyond 6 the nearest point is 6, and clamping keeps
        # the distances below from losing all precision for huge inputs
        mag = np.minimum(np.abs(v), 6.0)
        dist = np.abs(mag[:, None] - grid[None, :])
        best = dist.min(axis=1)
        cand = dist == best[:, None]
        # adjacent grid points have opposite mantissa parity, so at most one
        # even candidate exists; prefer it, else take the single candidate.
        pick_even = np.argmax(cand & even[None, :], axis=1)
        has_even = (cand & even[None, :]).any(axis=1)
        pick_any = np.argmax(cand, axis=1)
        idx = np.where(has_even, pick_even, pick_any).astype(np.uint8)
        neg = (v < 0) & (idx != 0)
        out[lo:lo + chunk] = idx | (neg.astype(np.uint8) << 3)
    return out.reshape(y.shape)


# ------------------------------------------------------------------- E4M3FN
def e4m3_decode(code):
    """Value of each E4M3FN byte (float64); 0x7F / 0xFF give NaN."""
    code = np.asarray(code).astype(np.int64)
    sign = (code >> 7) & 1
    exp = (code >> 3) & 15
    man = code & 7
    normal = np.ldexp(1.0 + man / 8.0, exp - 7)
    subnormal = np.ldexp(man / 8.0, -6)
    mag = np.where(exp == 0, subnormal, normal).astype(np.float64)
    mag = np.where((exp == 15) & (man == 7), np.nan, mag)
    return np.where(sign == 1, -mag, mag)


_E4M3_POS = e4m3_decode(np.arange(127))            # codes 0x00..0x7E, ascending


def e4m3_encode(t):
    """Round-to-nearest-even E4M3FN code of each value, saturating at +-448."""
    t = np.asarray(t, dtype=np.float64)
    mag = np.abs(t)
    hi = np.searchsorted(_E4M3_POS, mag, side="left")   # vals[hi-1] < mag <= vals[hi]
    hi = np.clip(hi, 0, 126)
    lo = np.clip(hi - 1, 0, 126)
    d_lo = np.abs(mag - _E4M3_POS[lo])
    d_hi = np.abs(_E4M3_POS[hi] - mag)
    pick = np.where(d_lo < d_hi, lo, hi)
    tie = d_lo == d_hi
    pick = np.where(tie, np.where(lo % 2 == 0, lo, hi), pick)
    pick = np.where(mag >= 448.0, 126, pick)            # satfinite
    code = pick.astype(np.uint8)
    neg = (t < 0) & (code != 0)
    return code | (neg.astype(np.uint8) << 7)


# --------------------------------------------------------------------- E8M0
def e8m0_decode(code):
    """2^(c-127) for each E8M0 byte (float64); 0xFF gives NaN."""
    code = np.asarray(code).astype(np.int64)
    val = np.ldexp(1.0, code - 127)
    return np.where(code == 255, np.nan, val)


def ceil_log2(y):
    """Exact ceil(log2(y)) for positive finite ``y`` via frexp.

    frexp gives y = f * 2^E with f in [0.5, 1); y is a power of two exactly
    when f == 0.5, and then log2(y) = E - 1; otherwise ceil(log2(y)) = E.
    """
    f, e = np.frexp(np.asarray(y))
    return np.where(f == 0.5, e - 1, e).astype(np.int64)


# --------------------------------------------------------------------- BF16
def bf16_bits(x):
    """Round-to-nearest-even BF16 bit pattern of float32 values (no NaNs)."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> 16) & 1
    return ((b + 0x7FFF + lsb) >> 16).astype(np.uint16)


def bf16_value(bits):
    """float32 value of BF16 bit patterns."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def bf16_round(x):
    """float32 values rounded to the nearest BF16 (ties to even)."""
    return bf16_value(bf16_bits(x))

"""FP8 E4M3 ("fn" variant) and E8M0 codecs, written from the OCP 8-bit floating point
and OCP Microscaling (MX) v1.0 format definitions.  Test infrastructure only.

The pages name the formats without defining them: "Kimi K3.1 Pro Inference Acceleration:
Day0 Optimization on Heterogeneous AI Hardware", sections "Full MXFP8 Quantization with
Per-Group Dynamic Scaling for LI" and "FP8 KVCache with Per-Token-Head-Tile Quantization
for SFA".  The element type of both is E4M3 (the MX element type of MXFP8, and the FP8
KV type of the workloads); the MX shared scale is E8M0.

E4M3 "fn": 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, no infinities,
NaN = S.1111.111, largest finite 448 = 1.75 * 2^8, subnormals m * 2^-9 (m = 1..7).
E8M0: an unsigned biased exponent, value 2^(code - 127), code 255 = NaN.

Pinned in tests/test_oracle_codecs.py: exhaustive decode of all 256 codes against the
ml_dtypes and torch float8_e4m3fn types, encode of every midpoint and of random values
against the libraries' round-to-nearest-even cast, and the saturation rule.
"""

import numpy as np

E4M3_MAX = 448.0
# Quantum of the subnormal range and of the lowest normal binade: 2^-6 * 2^-3.
_E4M3_MIN_EXP = -6


def e4m3_decode(codes):
    """Decode E4M3 codes (uint8 array) to float64 values, exactly."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = c >> 7
    exp = (c >> 3) & 0xF
    man = c & 0x7
    # normal: (1 + m/8) * 2^(exp-7) = (8 + m) * 2^(exp-10); subnormal: m * 2^-9
    mag = np.where(exp == 0, man * 2.0 ** -9, (8 + man) * np.ldexp(1.0, exp - 10))
    mag = np.where((exp == 0xF) & (man == 0x7), np.nan, mag)
    return np.where(sign == 1, -mag, mag)


def e4m3_encode(x):
    """Encode float64 values to E4M3 codes with round-to-nearest-even and saturation.

    Finite values beyond +-448 saturate to +-448 (the "satfinite" reading: the format has
    no infinity, and a quantiser that picks its own scale never wants NaN); the sign of
    zero is kept (-0.0 and negative values that round to zero give 0x80); NaN gives 0x7F.
    """
    x = np.asarray(x, dtype=np.float64)
    nan = np.isnan(x)
    neg = np.signbit(x)
    a = np.where(nan, 0.0, np.abs(x))
    a = np.minimum(a, E4M3_MAX)
    # floor(log2 a) for a > 0: frexp gives a = f * 2^E with f in [0.5, 1).
    _, E = np.frexp(a)
    e = np.where(a > 0, E - 1, _E4M3_MIN_EXP)
    e = np.maximum(e, _E4M3_MIN_EXP)
    quantum = np.ldexp(1.0, e - 3)           # spacing of 3-mantissa-bit values in binade e
    val = np.rint(a / quantum) * quantum      # exact scaling; rint rounds half to even
    # val is a grid point in [0, 448]; turn it into bits.
    sub = val < 2.0 ** _E4M3_MIN_EXP
    man_sub = np.rint(val / 2.0 ** -9).astype(np.int64)
    f, E2 = np.frexp(np.where(sub, 1.0, val))
    exp_field = (E2 - 1) + 7
    man = np.rint((2.0 * f - 1.0) * 8.0).astype(np.int64)
    code = np.where(sub, man_sub, (exp_field << 3) | man)
    code = code | (neg.astype(np.int64) << 7)
    code = np.where(nan, 0x7F, code)
    return code.astype(np.uint8)


def e8m0_decode(codes):
    """Decode E8M0 scale codes to float64 powers of two (code 255 is NaN)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    v = np.ldexp(1.0, c - 127)
    return np.where(c == 255, np.nan, v)

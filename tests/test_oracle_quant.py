"""Pins of the oracle's MXFP8 and FP8-tile quantisers: hand cases of the E8M0 rule,
closed-form round-trip bounds, idempotence, a library route for the element rounding and
exact rational arithmetic for the FP8 quotient."""

from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle.codecs import e4m3_decode
from oracle.quant import (mxfp8_quantize, mxfp8_dequantize, fp8_tile_quantize,
                          fp8_tile_dequantize, fp8_tile_bounds)

ml_dtypes = pytest.importorskip("ml_dtypes")


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("amax,exp", [
    (1.0, -8), (1.5, -8), (255.0, -1), (256.0, 0), (447.0, 0), (448.0, 0), (449.0, 0),
    (2.0 ** -130, -127), (2.0 ** -119, -127), (2.0 ** -118, -126), (3.0e38, 119),
])
def test_e8m0_rule_hand_cases(amax, exp):
    # OCP MX: shared exponent = floor(log2(amax)) - 8, clamped to [-127, 127]
    x = np.zeros(32)
    x[5] = amax
    x[6] = -amax / 4
    _, sc = mxfp8_quantize(x)
    assert int(sc[0]) == exp + 127


def test_zero_group():
    codes, sc = mxfp8_quantize(np.zeros(64))
    assert sc.tolist() == [127, 127] and not codes.any()
    codes, sc = fp8_tile_quantize(np.zeros(576))
    assert not sc.any() and not codes.any()


def _mx_data(seed=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((257, 128)).astype(np.float32)
    x[:, 7] *= 8          # outlier channel
    x[3] *= 1e-30         # subnormal-ish group scales
    x[4] *= 1e30
    x[5, :32] = 0.0       # a zero group
    return _bf16(x)


def test_mxfp8_roundtrip_bound():
    x = _mx_data()
    codes, sc = mxfp8_quantize(x)
    xh = mxfp8_dequantize(codes, sc)
    s = np.repeat(np.ldexp(1.0, sc.astype(np.int64) - 127), 32, axis=-1)
    sat = np.abs(x) > 448 * s
    err = np.abs(x - xh)
    bound = np.maximum(2.0 ** -4 * np.abs(x), 2.0 ** -10 * s)
    assert np.all(err[~sat] <= bound[~sat])
    assert np.all(np.abs(xh[sat]) == 448 * s[sat])
    # the group maximum always lands in [256, 448] * 2^e
    g = np.abs(xh).reshape(-1, 4, 32).max(-1)
    gs = s.reshape(-1, 4, 32)[..., 0]
    nz = g > 0
    assert np.all((g[nz] >= 256 * gs[nz]) & (g[nz] <= 448 * gs[nz]))


def test_mxfp8_idempotent():
    x = _mx_data(1)
    c1, s1 = mxfp8_quantize(x)
    c2, s2 = mxfp8_quantize(mxfp8_dequantize(c1, s1))
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2)


def test_mxfp8_elements_vs_library_cast():
    # The element rounding is a plain E4M3 cast of x * 2^-e (saturated): library route.
    x = _mx_data(2)
    codes, sc = mxfp8_quantize(x)
    s = np.repeat(np.ldexp(1.0, -(sc.astype(np.int64) - 127)), 32, axis=-1)
    y = np.clip(x * s, -448, 448).astype(np.float32)
    ref = y.astype(ml_dtypes.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(codes, ref)


def test_fp8_tile_bounds_576():
    assert fp8_tile_bounds(576) == [(0, 128), (128, 256), (256, 384), (384, 512), (512, 576)]


def _tile_data(seed=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((300, 576)).astype(np.float32)
    x[1] *= 1e-35
    x[2] *= 1e35
    x[3, 512:] = 0.0
    return _bf16(x)


def test_fp8_tile_scale_is_float32_division():
    x = _tile_data()
    _, sc = fp8_tile_quantize(x)
    for t, (lo, hi) in enumerate(fp8_tile_bounds(576)):
        amax = np.abs(x[:, lo:hi]).max(-1).astype(np.float32)
        assert np.array_equal(sc[:, t], amax / np.float32(448.0))


def _exact_rne_e4m3(q):
    """Correct round-to-nearest-even of an exact rational to E4M3 (saturating), by
    comparison against the exact grid -- independent of the oracle's encoder."""
    grid = sorted(set(Fraction(float(v)) for v in np.abs(e4m3_decode(np.arange(127, dtype=np.uint8)))
                      if not np.isnan(v)))
    a = abs(q)
    if a >= grid[-1]:
        return grid[-1] if q >= 0 else -grid[-1]
    import bisect
    i = bisect.bisect_right(grid, a) - 1
    lo, hi = grid[i], grid[i + 1]
    if a - lo < hi - a:
        r = lo
    elif a - lo > hi - a:
        r = hi
    else:
        # even mantissa: codes are monotone in value, so compare code parity
        r = lo if (i % 2 == 0) else hi
    return r if q >= 0 else -r


def test_fp8_tile_codes_vs_exact_rational():
    x = _tile_data(1)[:40]
    codes, sc = fp8_tile_quantize(x)
    dec = e4m3_decode(codes)
    for r in range(x.shape[0]):
        for t, (lo, hi) in enumerate(fp8_tile_bounds(576)):
            s = Fraction(float(sc[r, t]))
            for d in range(lo, hi, 7):
                if s == 0:
                    assert dec[r, d] == 0
                    continue
                want = _exact_rne_e4m3(Fraction(float(x[r, d])) / s)
                assert Fraction(float(dec[r, d])) == want, (r, d)


def test_fp8_tile_quotient_adversarial_vs_exact_rational():
    # every bf16 mantissa pair (x, amax) at exponent offsets 0..12: the fp64 quotient
    # must round like the exact quotient
    mant = np.arange(128, 256, dtype=np.float64) / 128.0
    rng = np.random.default_rng(5)
    am = rng.choice(mant, 24, replace=False)
    for a in am:
        amax = a * 4.0
        for shift in range(0, 13):
            xs = mant * 4.0 * 2.0 ** -shift
            row = np.zeros(128)
            row[0] = amax
            row[1:] = xs[:127]
            codes, sc = fp8_tile_quantize(row[None])
            s = Fraction(float(sc[0, 0]))
            dec = e4m3_decode(codes[0])
            for d in range(128):
                assert Fraction(float(dec[d])) == _exact_rne_e4m3(Fraction(float(row[d])) / s)


def test_fp8_tile_roundtrip_bound_and_idempotence():
    x = _tile_data(3)
    codes, sc = fp8_tile_quantize(x)
    xh = fp8_tile_dequantize(codes, sc)
    s = np.concatenate([np.repeat(sc[:, t:t + 1].astype(np.float64), hi - lo, axis=1)
                        for t, (lo, hi) in enumerate(fp8_tile_bounds(576))], axis=1)
    bound = np.maximum(2.0 ** -4 * np.abs(x), 2.0 ** -10 * s) * (1 + 2.0 ** -40)
    assert np.all(np.abs(x - xh) <= bound)

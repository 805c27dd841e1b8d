"""Pins of the oracle's FP8 codecs against independent library implementations of the
OCP formats (ml_dtypes and torch float8_e4m3fn / float8_e8m0fnu)."""

import numpy as np
import pytest
import torch

from oracle.codecs import e4m3_decode, e4m3_encode, e8m0_decode

ml_dtypes = pytest.importorskip("ml_dtypes")

ALL = np.arange(256, dtype=np.uint8)


def _same(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.array_equal(np.isnan(a), np.isnan(b)) and np.array_equal(
        np.where(np.isnan(a), 0, a), np.where(np.isnan(b), 0, b)) and np.array_equal(
        np.signbit(np.where(np.isnan(a), 0, a)), np.signbit(np.where(np.isnan(b), 0, b)))


def test_decode_exhaustive_vs_ml_dtypes():
    ref = ALL.view(ml_dtypes.float8_e4m3fn).astype(np.float64)
    assert _same(e4m3_decode(ALL), ref)


def test_decode_exhaustive_vs_torch():
    ref = torch.from_numpy(ALL.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert _same(e4m3_decode(ALL), ref)


def test_decode_known_values():
    assert e4m3_decode(np.uint8(0x7E)) == 448.0
    assert e4m3_decode(np.uint8(0x01)) == 2.0 ** -9
    assert e4m3_decode(np.uint8(0x08)) == 2.0 ** -6
    assert e4m3_decode(np.uint8(0x38)) == 1.0
    assert np.isnan(e4m3_decode(np.uint8(0x7F))) and np.isnan(e4m3_decode(np.uint8(0xFF)))


def test_encode_roundtrips_every_finite_code():
    finite = ALL[~np.isnan(e4m3_decode(ALL))]
    assert np.array_equal(e4m3_encode(e4m3_decode(finite)), finite)


def test_encode_midpoints_and_neighbours_vs_ml_dtypes():
    # The libraries cast through float32, so their inputs here are float32-exact: every
    # midpoint of the E4M3 grid and its float32 neighbours on both sides.
    vals = np.unique(np.abs(e4m3_decode(ALL[~np.isnan(e4m3_decode(ALL))])))
    mids = ((vals[1:] + vals[:-1]) / 2).astype(np.float32)
    eps = np.concatenate([mids, np.nextafter(mids, np.float32(0)),
                          np.nextafter(mids, np.float32(np.inf)), [np.float32(464.0)]])
    xs = np.concatenate([eps, -eps]).astype(np.float64)
    ref = xs.astype(np.float32).astype(ml_dtypes.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(e4m3_encode(xs), ref)


def test_encode_rounds_float64_neighbours_of_midpoints_correctly():
    # Closed form: a value just below (above) a midpoint rounds to the lower (upper)
    # neighbour; exactly on it, to the neighbour with the even mantissa.
    vals = np.unique(np.abs(e4m3_decode(ALL[~np.isnan(e4m3_decode(ALL))])))
    lo, hi = vals[:-1], vals[1:]
    mids = (lo + hi) / 2
    assert np.array_equal(e4m3_decode(e4m3_encode(np.nextafter(mids, 0))), lo)
    assert np.array_equal(e4m3_decode(e4m3_encode(np.nextafter(mids, np.inf))), hi)
    on = e4m3_encode(mids)
    even = np.where((e4m3_encode(lo) & 1) == 0, lo, hi)
    assert np.array_equal(e4m3_decode(on), even)


def test_encode_random_vs_ml_dtypes_and_torch():
    rng = np.random.default_rng(123)
    mag = np.exp2(rng.uniform(-14, np.log2(464.0), 200000))
    xs = (mag * rng.choice([-1.0, 1.0], mag.size)).astype(np.float32).astype(np.float64)
    ours = e4m3_encode(xs)
    assert np.array_equal(ours, xs.astype(ml_dtypes.float8_e4m3fn).view(np.uint8))
    t = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, t)


def test_encode_saturates_and_keeps_sign_of_zero():
    assert e4m3_encode(np.array([470.0, 1e30, -500.0])).tolist() == [0x7E, 0x7E, 0xFE]
    assert e4m3_encode(np.array([0.0, -0.0, -1e-30, 1e-30])).tolist() == [0x00, 0x80, 0x80, 0x00]
    assert e4m3_encode(np.array([np.nan]))[0] == 0x7F


def test_e8m0_decode_vs_ml_dtypes():
    ref = ALL.view(ml_dtypes.float8_e8m0fnu).astype(np.float64)
    assert _same(e8m0_decode(ALL), ref)

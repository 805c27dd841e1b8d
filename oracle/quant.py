"""Cache quantisers of the DSA path, in float64.  Test infrastructure only.

* MXFP8 for the Lightning Indexer (q and k): "Kimi K3.1 Pro Inference Acceleration:
  Day0 Optimization on Heterogeneous AI Hardware", section "Full MXFP8 Quantization with
  Per-Group Dynamic Scaling for LI" -- one scaling factor per group of 32 elements,
  chosen per group from the data.  Also "Deep Dive into Sparse Attention and Engineering
  Optimizations for Efficient Inference in Kimi K3.1 Pro", section 2.2 (every 32
  elements share one scaling factor).
* FP8 KV cache for Sparse Flash Attention: same page, section "FP8 KVCache with
  Per-Token-Head-Tile Quantization for SFA" -- one scaling factor per 128-element tile
  of each token (and head; the MLA latent cache has a single KV head).

Readings adopted where the pages are silent:

* MX scale rule: the OCP MX v1.0 rule, shared exponent e = floor(log2(amax)) - 8
  (8 = the largest exponent of E4M3), clamped to [-127, 127], stored as E8M0 code e+127;
  elements are x * 2^-e rounded to nearest even and saturated to +-448.  A group whose
  amax is 0 stores code 127 and all-zero element codes.
* FP8 tile rule: scale = fp32(amax / 448) rounded to nearest (fp32 division of the bf16
  amax); element codes are the exact quotient x / scale rounded once to E4M3 (nearest
  even, saturating).  A tile whose amax is 0 stores scale 0.0 and all-zero codes.
* The 576-wide MLA latent row (512 "nope" + 64 "rope") is cut into the tiles
  [0,128), [128,256), [256,384), [384,512), [512,576): five tiles, the last 64 wide.
"""

import numpy as np

from .codecs import e4m3_decode, e4m3_encode, E4M3_MAX

MX_GROUP = 32
FP8_TILE = 128
_E4M3_EMAX = 8


def mxfp8_quantize(x):
    """MXFP8 (E4M3 elements, E8M0 scale per 32 along the last axis).

    x: float array (..., D) with D a multiple of 32 (the bf16 values, exactly in fp64).
    Returns (codes uint8 (..., D), scale_codes uint8 (..., D // 32)).
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    assert d % MX_GROUP == 0
    g = x.reshape(x.shape[:-1] + (d // MX_GROUP, MX_GROUP))
    amax = np.abs(g).max(axis=-1)
    _, E = np.frexp(amax)                       # amax = f * 2^E, f in [0.5, 1)
    e = np.where(amax > 0, (E - 1) - _E4M3_EMAX, 0)
    e = np.clip(e, -127, 127)
    scale_codes = (e + 127).astype(np.uint8)
    scaled = g * np.ldexp(1.0, -e)[..., None]   # exact: multiplication by a power of two
    codes = e4m3_encode(scaled)
    codes = np.where((amax > 0)[..., None], codes, np.uint8(0))
    return codes.reshape(x.shape).astype(np.uint8), scale_codes


def mxfp8_dequantize(codes, scale_codes):
    """Inverse of mxfp8_quantize: e4m3(code) * 2^(scale_code - 127), exact in fp64."""
    codes = np.asarray(codes, dtype=np.uint8)
    d = codes.shape[-1]
    v = e4m3_decode(codes).reshape(codes.shape[:-1] + (d // MX_GROUP, MX_GROUP))
    s = np.ldexp(1.0, np.asarray(scale_codes).astype(np.int64) - 127)
    return (v * s[..., None]).reshape(codes.shape)


def fp8_tile_bounds(d):
    """Tile boundaries along a row of width d: 128-wide tiles, the last one partial."""
    starts = list(range(0, d, FP8_TILE))
    return [(s, min(s + FP8_TILE, d)) for s in starts]


def fp8_tile_quantize(x):
    """FP8 E4M3 with one fp32 scale per 128-element tile along the last axis.

    x: float array (..., D) (the bf16 values).  Returns (codes uint8 (..., D),
    scales float32 (..., ceil(D / 128))).
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    tiles = fp8_tile_bounds(d)
    codes = np.zeros(x.shape, dtype=np.uint8)
    scales = np.zeros(x.shape[:-1] + (len(tiles),), dtype=np.float32)
    for t, (lo, hi) in enumerate(tiles):
        xt = x[..., lo:hi]
        amax = np.abs(xt).max(axis=-1)
        # fp32 division of two fp32 numbers == fp64 division rounded to fp32
        # (53 >= 2*24 + 2, so the double rounding is innocuous).
        scale = (amax / E4M3_MAX).astype(np.float32)
        s64 = scale.astype(np.float64)
        nz = s64 > 0
        safe = np.where(nz, s64, 1.0)
        # The fp64 quotient of a bf16 value by an fp32 scale is the exact quotient
        # whenever it sits on an e4m3 rounding boundary (see the pin in the tests), so
        # rounding it once more to E4M3 is the correctly rounded code.
        q = xt / safe[..., None]
        ct = e4m3_encode(q)
        codes[..., lo:hi] = np.where(nz[..., None], ct, np.uint8(0))
        scales[..., t] = scale
    return codes, scales


def fp8_tile_dequantize(codes, scales):
    """Inverse of fp8_tile_quantize: e4m3(code) * scale[tile], in fp64."""
    codes = np.asarray(codes, dtype=np.uint8)
    d = codes.shape[-1]
    out = e4m3_decode(codes)
    scales = np.asarray(scales, dtype=np.float32).astype(np.float64)
    for t, (lo, hi) in enumerate(fp8_tile_bounds(d)):
        out[..., lo:hi] *= scales[..., t:t + 1]
    return out

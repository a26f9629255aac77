"""e2m1 (FP4) and e4m3 (FP8) codecs, written out from the format definitions.

Source passage: page "GPU kernel porting with AI agents", section "Sage
Attention 3" -- values are FP4 e2m1 (15 representable values), quantised in
1x16 groups (NVFP4), with scale factors in FP8 e4m3.  The bit layouts are the
public format definitions (1 sign bit, then exponent, then mantissa):

* e2m1: bias 1, no inf/NaN.  Magnitude codes 0..7 decode to
  0, 0.5, 1, 1.5, 2, 3, 4, 6; bit 3 is the sign.  +0 and -0 both exist, so the
  16 codes carry 15 distinct values.
* e4m3 ("fn" flavour): bias 7, no infinities, 0x7F/0xFF are NaN, largest
  finite magnitude 448, subnormal step 2**-9.

Encoders round to nearest with ties to the even code and saturate to the
largest finite magnitude (the readings "FP4 rounding" and "scale rule" of the
design notes).  The sign is kept, so a negative value that rounds to zero
becomes the negative-zero code.  Everything here is computed in float64 from
exact float32 inputs, so comparisons against grid points and midpoints are
exact.
"""

import numpy as np

# ---------------------------------------------------------------- e2m1 -----

#: magnitudes of e2m1 codes 0..7 (exponent bias 1; code 1 is the subnormal 0.5)
E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)
E2M1_MAX = 6.0


def _e2m1_magnitude_from_bits(code):
    """Decode the 3 magnitude bits from the exponent/mantissa fields."""
    e = (code >> 1) & 0x3
    m = code & 0x1
    # e == 0: subnormal m * 2**(1 - bias) * 0.5 ; else (1 + m/2) * 2**(e - bias)
    sub = m * 0.5
    norm = (1.0 + 0.5 * m) * np.exp2(e.astype(np.float64) - 1.0)
    return np.where(e == 0, sub, norm)


def e2m1_decode(codes):
    """Nibble codes (any int array, values 0..15) -> float64 values."""
    c = np.asarray(codes).astype(np.int64) & 0xF
    mag = _e2m1_magnitude_from_bits(c & 0x7)
    return np.where((c & 0x8) != 0, -mag, mag)


def _nearest_even(mag, grid):
    """Index of the grid point nearest to ``mag`` (float64 arrays), ties to the
    even index.  ``grid`` is sorted ascending and index parity equals code
    parity (the mantissa LSB) for both formats here.  Values beyond the last
    grid point map to the last index (saturation)."""
    mag = np.asarray(mag, dtype=np.float64)
    hi = np.searchsorted(grid, mag, side="left")          # grid[hi-1] < mag <= grid[hi]
    hi = np.clip(hi, 0, len(grid) - 1)
    lo = np.clip(hi - 1, 0, len(grid) - 1)
    d_lo = mag - grid[lo]
    d_hi = grid[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    idx = np.where(pick_hi, hi, lo)
    idx = np.where(mag >= grid[-1], len(grid) - 1, idx)   # saturate
    idx = np.where(mag <= grid[0], 0, idx)
    return idx


def e2m1_encode(x):
    """float array -> uint8 nibble codes; RNE ties-to-even, saturating at 6,
    sign kept (so -0.0 and small negatives give 0x8)."""
    x = np.asarray(x, dtype=np.float64)
    idx = _nearest_even(np.abs(x), E2M1_MAGNITUDES)
    sign = np.signbit(x).astype(np.int64) << 3
    return (idx | sign).astype(np.uint8)


# ---------------------------------------------------------------- e4m3 -----

E4M3_MAX = 448.0


def e4m3_decode(codes):
    """Byte codes (uint8) -> float64 values; 0x7F / 0xFF decode to NaN."""
    c = np.asarray(codes).astype(np.int64) & 0xFF
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0,
                   m * 2.0 ** -9,                                   # subnormal: m/8 * 2**(1-7)
                   (8 + m) * np.exp2(e.astype(np.float64) - 10.0))  # (1 + m/8) * 2**(e-7)
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return np.where((c & 0x80) != 0, -mag, mag)


#: all finite non-negative e4m3 values, index == code (0x00 .. 0x7E)
E4M3_GRID = e4m3_decode(np.arange(0x7F, dtype=np.uint8))


def e4m3_encode(x):
    """float array -> uint8 codes; RNE ties-to-even, saturating at +-448
    ("satfinite"), never producing the NaN codes."""
    x = np.asarray(x, dtype=np.float64)
    idx = _nearest_even(np.abs(x), E4M3_GRID)
    sign = np.signbit(x).astype(np.int64) << 7
    return (idx | sign).astype(np.uint8)

"""Number formats of the NVFP4 layer, written from their published definitions.

* E2M1 (FP4): 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit. Exponent
  field 0 is subnormal (m * 0.5). Magnitudes of codes 0..7:
  0, 0.5, 1, 1.5, 2, 3, 4, 6. Code = sign * 8 + (exponent << 1 | mantissa).
  No inf, no NaN.
* E4M3 (OCP FP8 E4M3, "e4m3fn"): 1 sign, 4 exponent bits (bias 7), 3 mantissa
  bits; exponent 0 is subnormal (m * 2^-9); S.1111.111 is NaN; no inf; the
  largest finite value is 1.75 * 2^8 = 448.
* BF16: the upper 16 bits of an IEEE binary32.

Encoders round to nearest, ties to the code with an even mantissa (RNE), and
saturate finite values beyond the largest magnitude to it ("satfinite"). The
sign is kept, so a negative value that rounds to zero encodes as -0.

NVFP4 packing (bloomery issue #565, §4, #489: "U8-packed E2M1 pairs"):
element 2i sits in the low nibble of byte i, element 2i+1 in the high nibble.
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------- E2M1

def e2m1_magnitude(code3: np.ndarray) -> np.ndarray:
    """Magnitude of a 3-bit E2M1 code (exponent, mantissa) as float64."""
    code3 = np.asarray(code3, dtype=np.int64)
    e = code3 >> 1
    m = code3 & 1
    sub = m * 0.5                              # exponent field 0: 0.m * 2^(1-1)
    nrm = (1.0 + 0.5 * m) * np.exp2(e - 1.0)   # 1.m * 2^(e-1)
    return np.where(e == 0, sub, nrm)


E2M1_GRID = e2m1_magnitude(np.arange(8))  # 0, .5, 1, 1.5, 2, 3, 4, 6


def e2m1_decode(code: np.ndarray) -> np.ndarray:
    """4-bit code -> float64 value (sign bit 3)."""
    code = np.asarray(code, dtype=np.int64)
    mag = E2M1_GRID[code & 7]
    return np.where(code & 8, -mag, mag)


def _rne_on_grid(mag: np.ndarray, grid: np.ndarray) -> np.ndarray:
    """Index of the nearest grid value to each magnitude (grid ascending, index
    parity = mantissa parity); ties go to the even index; values above the top
    saturate to it."""
    mag = np.asarray(mag, dtype=np.float64)
    top = len(grid) - 1
    hi = np.searchsorted(grid, mag, side="left")          # grid[hi-1] < mag <= grid[hi]
    hi = np.clip(hi, 0, top)
    lo = np.clip(hi - 1, 0, top)
    d_lo = mag - grid[lo]
    d_hi = grid[hi] - mag
    pick = np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi, np.where(lo % 2 == 0, lo, hi)))
    pick = np.where(mag >= grid[top], top, pick)
    pick = np.where(mag <= 0.0, 0, pick)
    return pick


def e2m1_encode(v: np.ndarray) -> np.ndarray:
    """float (no NaN) -> 4-bit code, RNE, satfinite, sign kept."""
    v = np.asarray(v, dtype=np.float64)
    if np.isnan(v).any():
        raise ValueError("E2M1 encode: NaN input")
    idx = _rne_on_grid(np.abs(v), E2M1_GRID)
    return (idx + 8 * np.signbit(v)).astype(np.uint8)


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """[..., 2n] 4-bit codes -> [..., n] bytes, element 2i in the low nibble."""
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = packed & 0x0F
    out[..., 1::2] = packed >> 4
    return out

# ---------------------------------------------------------------- E4M3

def e4m3_magnitude(code7: np.ndarray) -> np.ndarray:
    """Magnitude of a 7-bit E4M3 code (exponent, mantissa) as float64; 127 is NaN."""
    code7 = np.asarray(code7, dtype=np.int64)
    e = code7 >> 3
    m = code7 & 7
    sub = m * 2.0 ** -9                        # 0.mmm * 2^(1-7)
    nrm = (1.0 + m / 8.0) * np.exp2(e - 7.0)
    val = np.where(e == 0, sub, nrm)
    return np.where(code7 == 127, np.nan, val)


E4M3_GRID = e4m3_magnitude(np.arange(127))   # the 127 finite magnitudes, 0 .. 448
E4M3_MAX = 448.0


def e4m3_decode(code: np.ndarray) -> np.ndarray:
    code = np.asarray(code, dtype=np.int64)
    mag = e4m3_magnitude(code & 0x7F)
    return np.where(code & 0x80, -mag, mag)


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """float (no NaN) -> E4M3 byte, RNE, satfinite, sign kept."""
    v = np.asarray(v, dtype=np.float64)
    if np.isnan(v).any():
        raise ValueError("E4M3 encode: NaN input")
    idx = _rne_on_grid(np.abs(v), E4M3_GRID)
    return (idx + 128 * np.signbit(v)).astype(np.uint8)

# ---------------------------------------------------------------- BF16

def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    bits = np.asarray(bits, dtype=np.uint16).astype(np.uint32)
    return (bits << 16).view(np.float32)


def f32_to_bf16(v: np.ndarray) -> np.ndarray:
    """float32 -> BF16 bits, round to nearest even (finite inputs; overflow to inf)."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    bits = v.view(np.uint32)
    lo_bits = bits & np.uint32(0xFFFF0000)                   # truncate the magnitude
    hi_bits = lo_bits + np.uint32(0x10000)                   # next BF16 magnitude up
    alo = np.abs(lo_bits.view(np.float32).astype(np.float64))
    ahi = np.abs(hi_bits.view(np.float32).astype(np.float64))
    ahi = np.where(np.isinf(ahi), 2.0 ** 128, ahi)           # one step past the largest finite
    a = np.abs(v.astype(np.float64))
    d_lo = a - alo
    d_hi = ahi - a
    odd = (lo_bits >> 16) & 1
    up = (d_hi < d_lo) | ((d_hi == d_lo) & (odd == 1))
    return ((lo_bits >> 16) + up.astype(np.uint32)).astype(np.uint16)


def round_bf16(v: np.ndarray) -> np.ndarray:
    """Value of v (float64 or float32) after rounding to FP32 then BF16."""
    return bf16_to_f32(f32_to_bf16(np.asarray(v, dtype=np.float64).astype(np.float32))).astype(np.float64)

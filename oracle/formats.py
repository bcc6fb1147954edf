"""Number formats, written out from their bit-field definitions.

* E2M1 (FP4): 1 sign, 2 exponent, 1 mantissa bit.  Its non-negative values are
  0, 0.5, 1, 1.5, 2, 3, 4, 6 ("Quantization in deployment", "Fake
  quantization", the E2M1 value list; "Quantization chains", "MXFP4 against
  NVFP4 scales").
* E4M3 (FP8, the ``fn`` variant): 1 sign, 4 exponent (bias 7), 3 mantissa
  bits, no infinities, S.1111.111 is NaN; largest finite 448, smallest normal
  2^-6, smallest subnormal 2^-9 ("Quantization chains", "E4M3 against E5M2").
* E8M0: an unsigned biased exponent, value 2^(byte - 127) (the OCP MX scale;
  "Quantization in deployment", format cheat sheet: "one power-of-2 scale per
  32 numbers (E8M0)").
* FP16: IEEE binary16; numpy's float32 -> float16 cast rounds to nearest even.
"""
from __future__ import annotations

import numpy as np

# Non-negative E2M1 values, indexed by the 3-bit code (exponent bits, mantissa bit).
E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)
E2M1_MAX = 6.0
E4M3_MAX = 448.0
# The float32 value of the 1e-12 clamp used by the pages' amax / scale clamps.
F32_1E_12 = np.float32(1e-12)


def e2m1_decode(code) -> np.ndarray:
    """Value of 4-bit E2M1 codes (bit 3 is the sign) as float64."""
    c = np.asarray(code, dtype=np.int64)
    mag = E2M1_MAGNITUDES[c & 7]
    return np.where((c & 8) != 0, -mag, mag)


def e2m1_nearest(mag, ties: str = "smaller") -> np.ndarray:
    """Index (0..7) of the E2M1 magnitude nearest to each ``mag`` in [0, 6].

    "Quantization in deployment", "Fake quantization", ``fp4``: the value is
    the one at the smallest absolute distance, and when two are equally near
    the first one in the table (the smaller magnitude) is taken.  The distances
    are formed in float64, where they are exact for float32 inputs.

    ``ties="even"`` is the IEEE alternative (round half to even, the rounding
    of the hardware E2M1 convert): of two equally near values the one with the
    even code, i.e. mantissa bit 0, is taken.
    """
    m = np.asarray(mag, dtype=np.float64)
    dist = np.abs(m[..., None] - E2M1_MAGNITUDES)
    first = np.argmin(dist, axis=-1)
    if ties == "smaller":
        return first.astype(np.uint8)
    if ties != "even":
        raise ValueError(ties)
    nxt = np.minimum(first + 1, 7)
    tie = np.take_along_axis(dist, nxt[..., None], -1)[..., 0] == np.take_along_axis(
        dist, first[..., None], -1)[..., 0]
    return np.where(tie & (first % 2 == 1), nxt, first).astype(np.uint8)


def e4m3_decode(byte) -> np.ndarray:
    """Value of E4M3 bytes as float64 (NaN for the two NaN codes)."""
    b = np.asarray(byte, dtype=np.int64)
    sign = np.where((b >> 7) & 1, -1.0, 1.0)
    exp = (b >> 3) & 0xF
    man = (b & 7).astype(np.float64)
    sub = man / 8.0 * 2.0 ** -6
    nor = (1.0 + man / 8.0) * np.exp2(exp.astype(np.float64) - 7.0)
    val = np.where(exp == 0, sub, nor)
    val = np.where((exp == 15) & ((b & 7) == 7), np.nan, val)
    return sign * val


# Finite non-negative E4M3 values in code order 0x00..0x7E (increasing).
_E4M3_POS = e4m3_decode(np.arange(0x7F))


def e4m3_encode(t) -> np.ndarray:
    """Round non-negative finite values to E4M3 bytes: nearest value, ties to
    the even code (round to nearest even), values above 448 saturate to 448.

    Consecutive codes hold consecutive values, so the even code of a tied pair
    is the one with a zero mantissa LSB.
    """
    x = np.asarray(t, dtype=np.float64)
    if np.any(~(x >= 0)):
        raise ValueError("e4m3_encode expects finite non-negative values")
    hi = np.searchsorted(_E4M3_POS, x, side="left")  # first value >= x
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_lo = np.abs(x - _E4M3_POS[lo])
    d_hi = np.abs(_E4M3_POS[hi] - x)
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(x >= E4M3_MAX, 0x7E, code)
    return code.astype(np.uint8)


def e8m0_decode(byte) -> np.ndarray:
    return np.exp2(np.asarray(byte, dtype=np.float64) - 127.0)


def fp16_encode(s) -> np.ndarray:
    """float32 -> IEEE binary16 bits (round to nearest even)."""
    with np.errstate(over="ignore"):
        return np.asarray(s, dtype=np.float32).astype(np.float16).view(np.uint16)


def fp16_decode(bits) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def floor_log2(a) -> np.ndarray:
    """Exact floor(log2(a)) for positive finite float32 ``a``:
    a = f * 2**e with f in [0.5, 1) gives floor(log2 a) = e - 1."""
    _, e = np.frexp(np.asarray(a, dtype=np.float32))
    return e.astype(np.int64) - 1

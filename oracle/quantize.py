"""Quantizers and dequantizers: NVFP4, MXFP4 and INT4 g128.

Every quantizer takes a float32 array [rows, K] (bf16 inputs are widened to
float32 exactly before they get here) and returns packed codes [rows, K/2]
(uint8, element 2j in the low nibble) plus its scales in plain row-major
[rows, K/block] order.  The arithmetic on the way to a code is float32 with
IEEE rounding, step by step as the pages write it; dequantization is float64,
where every product below is exact.
"""
from __future__ import annotations

import numpy as np

from .formats import (
    E2M1_MAX, E4M3_MAX, F32_1E_12, e2m1_decode, e2m1_nearest, e4m3_decode,
    e4m3_encode, e8m0_decode, floor_log2, fp16_decode, fp16_encode,
)

F32 = np.float32
_CHUNK_ELEMS = 1 << 22  # rows are processed in chunks of about this many elements


def _rows_chunks(rows: int, K: int):
    step = max(1, _CHUNK_ELEMS // max(K, 1))
    for r0 in range(0, rows, step):
        yield r0, min(rows, r0 + step)


def _as_f32_2d(x) -> np.ndarray:
    a = np.asarray(x, dtype=np.float32)
    if a.ndim != 2:
        raise ValueError("expected a 2-D [rows, K] array")
    return a


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """[rows, K] 4-bit codes -> [rows, K/2] bytes; element 2j -> low nibble."""
    c = np.asarray(codes, dtype=np.uint8) & 0xF
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty((p.shape[0], p.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = p & 0xF
    out[:, 1::2] = p >> 4
    return out


def _ties(rounding: str) -> str:
    """The E2M1 tie rule of a rounding mode: the pages' (ties to the smaller
    magnitude) or IEEE round half to even."""
    if rounding == "pages":
        return "smaller"
    if rounding == "rne":
        return "even"
    raise ValueError(rounding)


def _e2m1_codes(x: np.ndarray, S: np.ndarray, ties: str = "smaller") -> np.ndarray:
    """E2M1 codes of x / S ("Quantization in deployment", "Fake quantization",
    ``fp4``): y = clamp(x / S, -6, 6) in float32, the nearest E2M1 magnitude
    (ties to the smaller one, or to the even code with ``ties="even"``), and
    the sign of x in bit 3."""
    y = np.clip(x / S, F32(-E2M1_MAX), F32(E2M1_MAX))
    idx = e2m1_nearest(np.abs(y), ties)
    return idx | ((x < 0).astype(np.uint8) << 3)


# ---------------------------------------------------------------------------
# NVFP4: E2M1 codes, one E4M3 scale per 16, one FP32 scale per tensor
# ---------------------------------------------------------------------------

def nvfp4_tensor_scale(x) -> np.float32:
    """Per-tensor scale g = max(amax, 1e-12) / (448 * 6), in float32
    ("Quantization in deployment", "Fake quantization", ``nvfp4``: the global
    scale; "Quantization chains", "Bits per weight": one FP32 scale per tensor)."""
    a = _as_f32_2d(x)
    amax = F32(np.max(np.abs(a))) if a.size else F32(0.0)
    return F32(max(amax, F32_1E_12) / F32(E4M3_MAX * E2M1_MAX))


def quantize_nvfp4(x, g=None, rows=None, rounding="pages"):
    """NVFP4 quantization ("Quantization in deployment", "Fake quantization",
    ``nvfp4`` then ``fp4``), per block of 16 along K:

    1. amax_b = max |x| over the block;
    2. t = (amax_b / 6) / g, two float32 divisions in that order;
    3. the block scale is t rounded to E4M3 (nearest even) -> byte bs;
    4. S = max(e4m3(bs), 1e-12) * g in float32;
    5. each element is rounded to E2M1 at x / S, clamped to +-6.

    A block whose scale byte is 0 stores all-zero codes (reading 4).
    ``g`` defaults to :func:`nvfp4_tensor_scale` of the whole ``x``; ``rows``
    optionally selects the rows to quantize (g still covers the whole x).
    ``rounding="rne"`` rounds step 5 half to even instead of to the smaller
    magnitude (everything else is unchanged).
    Returns (codes [r, K/2] u8, scales [r, K/16] u8, g float32).
    """
    a = _as_f32_2d(x)
    K = a.shape[1]
    if K % 16:
        raise ValueError("K must be a multiple of 16")
    g = nvfp4_tensor_scale(a) if g is None else F32(g)
    src = a if rows is None else a[np.asarray(rows)]
    R = src.shape[0]
    codes = np.empty((R, K // 2), dtype=np.uint8)
    scales = np.empty((R, K // 16), dtype=np.uint8)
    for r0, r1 in _rows_chunks(R, K):
        blk = src[r0:r1].reshape(r1 - r0, K // 16, 16)
        amax_b = np.max(np.abs(blk), axis=-1)
        t = (amax_b / F32(6.0)) / g
        bs = e4m3_encode(t)
        S = (np.maximum(e4m3_decode(bs).astype(np.float32), F32_1E_12) * g).astype(np.float32)
        c = _e2m1_codes(blk, S[..., None], _ties(rounding))
        c = np.where((bs == 0)[..., None], np.uint8(0), c)
        codes[r0:r1] = pack_nibbles(c.reshape(r1 - r0, K))
        scales[r0:r1] = bs
    return codes, scales, g


def dequantize_nvfp4(codes, scales, g) -> np.ndarray:
    """x_hat = e2m1(code) * e4m3(scale) * g, in float64 (exact)."""
    c = unpack_nibbles(codes)
    R, K = c.shape
    v = e2m1_decode(c).reshape(R, K // 16, 16)
    s = e4m3_decode(np.asarray(scales)) * np.float64(g)
    return (v * s[..., None]).reshape(R, K)


# ---------------------------------------------------------------------------
# MXFP4: E2M1 codes, one E8M0 (power of two) scale per 32
# ---------------------------------------------------------------------------

def quantize_mxfp4(x, rows=None, rounding="pages"):
    """MXFP4 quantization ("Quantization in deployment", "Fake quantization",
    ``mxfp4``), per block of 32 along K:

    1. amax_b = max(max |x|, 1e-12);
    2. e = floor(log2 amax_b) - 2 (the largest E2M1 exponent is 2), taken
       exactly from the float32 bits (reading 2), so that the block maximum
       lands in [4, 8) times the scale ("Quantization chains", "MXFP4 against
       NVFP4 scales");
    3. scale S = 2^e, stored as the E8M0 byte e + 127;
    4. each element is rounded to E2M1 at x / S, clamped to +-6 (ties to the
       smaller magnitude, or half to even with ``rounding="rne"``).

    Returns (codes [r, K/2] u8, scales [r, K/32] u8).
    """
    a = _as_f32_2d(x)
    K = a.shape[1]
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    src = a if rows is None else a[np.asarray(rows)]
    R = src.shape[0]
    codes = np.empty((R, K // 2), dtype=np.uint8)
    scales = np.empty((R, K // 32), dtype=np.uint8)
    for r0, r1 in _rows_chunks(R, K):
        blk = src[r0:r1].reshape(r1 - r0, K // 32, 32)
        amax_b = np.maximum(np.max(np.abs(blk), axis=-1), F32_1E_12)
        e = floor_log2(amax_b) - 2
        S = np.ldexp(F32(1.0), e.astype(np.int32)).astype(np.float32)
        c = _e2m1_codes(blk, S[..., None], _ties(rounding))
        codes[r0:r1] = pack_nibbles(c.reshape(r1 - r0, K))
        scales[r0:r1] = (e + 127).astype(np.uint8)
    return codes, scales


def dequantize_mxfp4(codes, scales) -> np.ndarray:
    c = unpack_nibbles(codes)
    R, K = c.shape
    v = e2m1_decode(c).reshape(R, K // 32, 32)
    return (v * e8m0_decode(scales)[..., None]).reshape(R, K)


# ---------------------------------------------------------------------------
# INT4 g128: symmetric integers in [-8, 7], one FP16 scale per 128
# ---------------------------------------------------------------------------

def quantize_int4_g128(x, rows=None):
    """Symmetric INT4 group quantization ("Low-bit inference for very large
    MoE", "Why quantization-aware training", ``fake_int4``, with groups of 128
    and an FP16 scale as in "Quantization chains", "Bits per weight"):

    1. s = amax_g / 7 in float32, stored as FP16 (nearest even) -> s16;
    2. q = round-half-even(x / s16), clamped to [-8, 7] (reading 3: the
       division is by the stored FP16 scale, so x_hat = q * s16);
    3. a zero FP16 scale gives q = 0.

    Returns (codes [r, K/2] u8 two's complement nibbles, scales [r, K/128] u16
    FP16 bits).
    """
    a = _as_f32_2d(x)
    K = a.shape[1]
    if K % 128:
        raise ValueError("K must be a multiple of 128")
    src = a if rows is None else a[np.asarray(rows)]
    R = src.shape[0]
    codes = np.empty((R, K // 2), dtype=np.uint8)
    scales = np.empty((R, K // 128), dtype=np.uint16)
    for r0, r1 in _rows_chunks(R, K):
        blk = src[r0:r1].reshape(r1 - r0, K // 128, 128)
        amax_g = np.max(np.abs(blk), axis=-1)
        s16 = fp16_encode(amax_g / F32(7.0))
        sf = fp16_decode(s16).astype(np.float32)[..., None]
        with np.errstate(divide="ignore", invalid="ignore"):
            q = np.rint(blk / sf)
        q = np.where(sf == 0, F32(0.0), np.clip(q, F32(-8.0), F32(7.0)))
        codes[r0:r1] = pack_nibbles((q.astype(np.int8).astype(np.uint8) & 0xF).reshape(r1 - r0, K))
        scales[r0:r1] = s16
    return codes, scales


def int4_values(codes) -> np.ndarray:
    """Signed integers of packed two's complement nibbles, [rows, K] int8."""
    c = unpack_nibbles(codes).astype(np.int8)
    return np.where(c >= 8, c - 16, c).astype(np.int8)


def dequantize_int4_g128(codes, scales) -> np.ndarray:
    q = int4_values(codes).astype(np.float64)
    R, K = q.shape
    s = fp16_decode(scales)
    return (q.reshape(R, K // 128, 128) * s[..., None]).reshape(R, K)

"""FP8 (E4M3) blockwise quantization and the block-promoted FP8 GEMM.

TEST INFRASTRUCTURE ONLY (see the package docstring): a plain restatement of
the pages' definitions, never called by the product path.

* Quantization ("Quantization in deployment", "Fake quantization",
  ``fp8_blockwise`` and ``fp8``): weights get one scale per 128 x 128 block,
  activations one per (1, 128) block, i.e. per token and per 128 channels.
  For each block: amax = max |x| over the block, s = max(amax, 1e-12) / 448,
  and every element becomes the E4M3 value of clamp(x / s, -448, 448), the
  cast rounding to nearest even.  The block height is min(block rows, rows),
  and the shape must divide into whole blocks (the page reshapes into them).
* GEMM ("Quantization in deployment", exercise 2, the cost of block FP8): the
  tensor cores multiply and accumulate the FP8 codes within one 128-wide K
  block, that block's sum is multiplied by its activation and weight scales,
  and the results of the K blocks are summed:
      C[m, n] = sum_kb  sa[m, kb] * sb[n // 128, kb] * sum_{k in kb} qa[m, k] qb[n, k].
* W4A8 ("Low-bit inference for very large MoE", "Kernels on different
  hardware", the W4A8 row: INT4 weights dequantized to FP8, activations
  quantized to FP8, the product on FP8 tensor cores).  The INT4 values -8..7
  are exact E4M3 values, so the weight codes enter the FP8 product unchanged
  and their FP16 group scale (one per 128 along K, aligned with the 128-wide
  K blocks) joins the activation scale in the per-block promotion:
      C[m, n] = sum_kb  sa[m, kb] * s16[n, kb] * sum_{k in kb} qa[m, k] q[n, k].

Arithmetic: the quantizer steps are float32 with IEEE rounding, as the page's
float32 tensors compute them.  The GEMM is float64: the block sums of E4M3
products are exact there (each product has at most 8 significant bits and a
block adds 128 of them), and only the scaling and the sum over blocks round.
"""
from __future__ import annotations

import numpy as np

from .formats import E4M3_MAX, F32_1E_12, e4m3_decode, e4m3_encode, fp16_decode
from .quantize import int4_values

F32 = np.float32
FP8_BLOCK_K = 128


def e4m3_encode_signed(y) -> np.ndarray:
    """E4M3 bytes of float32 values: the magnitude clamped to 448 and rounded
    to nearest even (``e4m3_encode``), the sign bit from the sign of ``y``
    (an IEEE cast keeps the sign of a value that rounds to zero, and of -0)."""
    v = np.asarray(y, dtype=np.float32)
    if not np.all(np.isfinite(v)):
        raise ValueError("e4m3_encode_signed expects finite values")
    mag = e4m3_encode(np.minimum(np.abs(v).astype(np.float64), E4M3_MAX))
    return np.where(np.signbit(v), mag | np.uint8(0x80), mag).astype(np.uint8)


def _block_rows(rows: int, block_rows: int) -> int:
    return min(block_rows, rows)


def quantize_fp8_blockwise(x, block=(128, 128)):
    """Blockwise E4M3 quantization of a float32 [rows, K] array.

    block = (128, 128) for weights, (1, 128) for activations.  Returns
    (codes [rows, K] u8, scales float32 [rows / br, K / bc]) with br =
    min(block[0], rows), bc = block[1].
    """
    a = np.asarray(x, dtype=np.float32)
    if a.ndim != 2:
        raise ValueError("expected a 2-D [rows, K] array")
    rows, K = a.shape
    br, bc = _block_rows(rows, block[0]), block[1]
    if br == 0 or rows % br or K % bc:
        raise ValueError("the shape must divide into whole blocks")
    g = a.reshape(rows // br, br, K // bc, bc)
    amax = np.max(np.abs(g), axis=(1, 3))                     # [rows/br, K/bc]
    s = (np.maximum(amax, F32_1E_12) / F32(E4M3_MAX)).astype(np.float32)
    y = (g / s[:, None, :, None]).astype(np.float32)          # one IEEE division each
    y = np.clip(y, F32(-E4M3_MAX), F32(E4M3_MAX))
    codes = e4m3_encode_signed(y).reshape(rows, K)
    return codes, s


def dequantize_fp8_blockwise(codes, scales, block=(128, 128)) -> np.ndarray:
    """x_hat = e4m3(code) * s of the element's block, in float64 (exact)."""
    c = np.asarray(codes)
    rows, K = c.shape
    br, bc = _block_rows(rows, block[0]), block[1]
    v = e4m3_decode(c).reshape(rows // br, br, K // bc, bc)
    s = np.asarray(scales, dtype=np.float64)
    return (v * s[:, None, :, None]).reshape(rows, K)


def gemm_fp8_blockwise(qa, sa, qb, sb) -> np.ndarray:
    """Block-promoted FP8 product, float64 [M, N].

    qa: E4M3 [M, K] with sa float32 [M, K/128] (activation blocks (1, 128));
    qb: E4M3 [N, K] with sb float32 [N/128, K/128] (weight blocks 128 x 128,
    or one block row when N < 128).
    """
    A = e4m3_decode(np.asarray(qa))
    B = e4m3_decode(np.asarray(qb))
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K or K % FP8_BLOCK_K:
        raise ValueError("K must match and be a multiple of 128")
    br = _block_rows(N, 128)
    sa = np.asarray(sa, dtype=np.float64)
    sb = np.asarray(sb, dtype=np.float64)
    C = np.zeros((M, N), dtype=np.float64)
    for kb in range(K // FP8_BLOCK_K):
        ks = slice(kb * FP8_BLOCK_K, (kb + 1) * FP8_BLOCK_K)
        P = A[:, ks] @ B[:, ks].T                              # exact block sums
        wscale = np.repeat(sb[:, kb], br)                      # per output column
        C += P * sa[:, kb][:, None] * wscale[None, :]
    return C


def int4_to_e4m3(q) -> np.ndarray:
    """E4M3 bytes of INT4 values (exact: every integer in -8..7 is an E4M3
    value), the weight conversion of W4A8."""
    return e4m3_encode_signed(np.asarray(q, dtype=np.float32))


def gemm_w4a8(qa, sa, w_codes, w_scales) -> np.ndarray:
    """W4A8 product, float64 [M, N]: FP8 activations qa [M, K] with (1, 128)
    block scales sa float32 [M, K/128]; INT4 g128 weights (packed codes
    [N, K/2], FP16 scale bits [N, K/128]) converted to E4M3 and promoted per
    128-wide K block with sa[m, kb] * s16[n, kb]."""
    A = e4m3_decode(np.asarray(qa))
    B = e4m3_decode(int4_to_e4m3(int4_values(w_codes)))
    M, K = A.shape
    if B.shape[1] != K or K % FP8_BLOCK_K:
        raise ValueError("K must match and be a multiple of 128")
    sa = np.asarray(sa, dtype=np.float64)
    sw = fp16_decode(np.asarray(w_scales))                    # [N, K/128] float64
    C = np.zeros((M, B.shape[0]), dtype=np.float64)
    for kb in range(K // FP8_BLOCK_K):
        ks = slice(kb * FP8_BLOCK_K, (kb + 1) * FP8_BLOCK_K)
        P = A[:, ks] @ B[:, ks].T                              # exact block sums
        C += P * sa[:, kb][:, None] * sw[:, kb][None, :]
    return C

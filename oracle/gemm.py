"""FP64 reference products of the dequantized operands.

C = A_hat . B_hat^T with B stored [N, K] (the weight layout).  The products of
dequantized 4-bit values are exact in float64 and the sums are float64; the
matrix product is numpy's float64 matmul, used as a library step.

* W4A4 ("Low-bit inference for very large MoE", "Kernels on different
  hardware": activations quantized to FP4 too, both operands enter the FP4
  tensor cores): C = dequant(A) . dequant(B)^T.
* W4A16 (same section, W4A16 row, which lists INT4 and FP4 weights with
  16-bit activations): C = A_bf16 . dequant(W)^T, W in INT4 g128, NVFP4 or
  MXFP4.
* Grouped MoE (same section, "MoE's grouped GEMM must support low bits too":
  one low-bit weight matrix per expert, grouped by routing): for every expert
  e, C[rows of e] = A_hat[tokens routed to e] . W_hat_e^T, where the tokens are
  quantized once as a whole tensor and their rows gathered (reading 7).
"""
from __future__ import annotations

import numpy as np

from .quantize import (
    dequantize_int4_g128, dequantize_mxfp4, dequantize_nvfp4, quantize_mxfp4,
    quantize_nvfp4,
)


def gemm_fp64(a_hat: np.ndarray, b_hat: np.ndarray) -> np.ndarray:
    """float64 C = a_hat . b_hat^T (b_hat is [N, K])."""
    return np.asarray(a_hat, np.float64) @ np.asarray(b_hat, np.float64).T


def gemm_w4a4_nvfp4(a_codes, a_scales, a_g, b_codes, b_scales, b_g) -> np.ndarray:
    return gemm_fp64(dequantize_nvfp4(a_codes, a_scales, a_g),
                     dequantize_nvfp4(b_codes, b_scales, b_g))


def gemm_w4a4_mxfp4(a_codes, a_scales, b_codes, b_scales) -> np.ndarray:
    return gemm_fp64(dequantize_mxfp4(a_codes, a_scales), dequantize_mxfp4(b_codes, b_scales))


def gemm_w4a16_int4(a, w_codes, w_scales) -> np.ndarray:
    """C = a . dequant(W)^T with ``a`` the (bf16-valued) activations."""
    return gemm_fp64(np.asarray(a, np.float64), dequantize_int4_g128(w_codes, w_scales))


def gemm_w4a16_nvfp4(a, w_codes, w_scales, w_g) -> np.ndarray:
    """C = a . dequant(W)^T, W NVFP4 (row-major E4M3 scales, tensor scale w_g)."""
    return gemm_fp64(np.asarray(a, np.float64), dequantize_nvfp4(w_codes, w_scales, w_g))


def gemm_w4a16_mxfp4(a, w_codes, w_scales) -> np.ndarray:
    """C = a . dequant(W)^T, W MXFP4 (row-major E8M0 scales)."""
    return gemm_fp64(np.asarray(a, np.float64), dequantize_mxfp4(w_codes, w_scales))


def grouped_gemm_moe(tokens, expert_offsets, row_token, experts_q):
    """Routed NVFP4 MoE product.

    tokens: float32 [T, K] (bf16 values); expert_offsets: [E+1]; row_token:
    [R] token id of each routed row, rows grouped by expert; experts_q: list of
    (codes, scales, g) per expert.  Returns float64 C [R, N].
    """
    a_codes, a_scales, a_g = quantize_nvfp4(tokens)
    a_hat = dequantize_nvfp4(a_codes, a_scales, a_g)
    E = len(expert_offsets) - 1
    R = int(expert_offsets[-1])
    N = experts_q[0][0].shape[0] if E else 0
    out = np.zeros((R, N), dtype=np.float64)
    for e in range(E):
        r0, r1 = int(expert_offsets[e]), int(expert_offsets[e + 1])
        if r1 == r0:
            continue
        w_hat = dequantize_nvfp4(*experts_q[e])
        out[r0:r1] = gemm_fp64(a_hat[row_token[r0:r1]], w_hat)
    return out


def mxfp4_operands(a, b):
    """Quantize both operands of an MXFP4 W4A4 product."""
    return quantize_mxfp4(a), quantize_mxfp4(b)

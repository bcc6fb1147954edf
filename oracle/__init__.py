"""CPU oracle for block-scaled 4-bit quantization and the GEMMs that consume it.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product path (``int4_gemm_gb300``) never calls it and shares no code with it:
it is a plain, slow restatement of what the method computes, written from the
pages' definitions, so that the CUDA kernels can be checked against something
that does not share their mistakes.

Sources (web pages, cited by title and section):

* "Quantization in deployment" (anrans.github.io AI-infra handbook, serving /
  perf), section "Fake quantization": the E2M1 value set, round-to-nearest
  E2M1 (``fp4``), MXFP4 (one power-of-two scale per 32) and NVFP4 (one E4M3
  scale per 16 plus an FP32 per-tensor scale), and the E4M3 cast.
* "Low-bit inference for very large MoE: INT4, FP4 and quantization-aware
  training" (same handbook, frontier), section "Why quantization-aware
  training": symmetric INT4 group quantization ``fake_int4``.
* "Quantization chains: bits with scales, where INT4 loses, and what rounds to
  zero" (inferenceinterviews.com): E4M3 limits, bits per weight, the MXFP4 vs
  NVFP4 example, the per-tensor vs per-block E4M3 example.
* "LLM quantization" (drpranayjha.com, part 18): the eight-weight worked
  example and the outlier example.
* "Quantization in deployment", "Fake quantization" (``fp8``,
  ``fp8_blockwise``) and exercise 2 (block FP8's per-block promotion in the
  GEMM): FP8 blockwise quantization and GEMM (``oracle.fp8``).

Readings taken where the pages are silent or disagree (each one is also listed
with its reason in the design notes of this repository):

1. E2M1 ties go to the smaller magnitude (the ``argmin`` in ``fp4`` returns the
   first minimum).
2. MXFP4's exponent is the exact ``floor(log2(amax))`` of the FP32 amax.
3. INT4 g128 stores its scale as FP16 (round to nearest even) and divides by
   the stored FP16 value; a zero FP16 scale gives all-zero codes.
4. An NVFP4 block whose E4M3 scale encodes to zero stores scale byte 0 and
   all-zero codes.
5. A code's sign bit is ``x < 0``.
6. Element 2j of a row goes to the low nibble of byte j, element 2j+1 to the
   high nibble; INT4 codes are 4-bit two's complement.
7. The NVFP4 per-tensor scale covers the whole operand passed in.
8. FP8 blockwise: an E4M3 byte keeps the sign of x / s, also when it rounds to
   zero (an IEEE cast; x = -0 gives 0x80).

Parity pins: every quantizer and the E2M1 / E4M3 / E8M0 / FP16 encoders are
pinned by tests against values printed on the pages, closed forms and brute
force.  The FP64 GEMMs are pinned by brute-force summation on tiny shapes and
by special cases (identity operand, equal blocks); no page prints a GEMM
output, so beyond that their parity rests on the FP64 definition.
"""

from . import formats, quantize, gemm, fp8  # noqa: F401
from .quantize import (  # noqa: F401
    nvfp4_tensor_scale, quantize_nvfp4, quantize_mxfp4, quantize_int4_g128,
    dequantize_nvfp4, dequantize_mxfp4, dequantize_int4_g128,
    pack_nibbles, unpack_nibbles,
)
from .gemm import (  # noqa: F401
    gemm_fp64, gemm_w4a4_nvfp4, gemm_w4a4_mxfp4, gemm_w4a16_int4, gemm_w4a16_nvfp4,
    gemm_w4a16_mxfp4, grouped_gemm_moe,
)
from .fp8 import (  # noqa: F401
    e4m3_encode_signed, quantize_fp8_blockwise, dequantize_fp8_blockwise, gemm_fp8_blockwise,
    int4_to_e4m3, gemm_w4a8,
)

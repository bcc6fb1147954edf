"""The C-ABI library without a GPU: it builds, loads, exports every function the
public header declares, and rejects bad arguments on the host before any
launch (these calls return before touching the device)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q4gemm.h")


@pytest.fixture(scope="module")
def clib():
    from int4_gemm_gb300 import build
    import int4_gemm_gb300 as q4
    build.build()
    return q4.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("defined",)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ["quantize_nvfp4", "quantize_mxfp4", "quantize_int4_g128", "gemm_w4a4_nvfp4",
                 "gemm_w4a4_mxfp4", "gemm_w4a4_mxfp4_fused", "gemm_w4a16_int4", "gemm_w4a16_nvfp4", "gemm_w4a16_mxfp4",
                 "grouped_gemm_moe", "q4_sync_status", "quantize_fp8_blockwise", "gemm_fp8_blockwise", "gemm_w4a8", "w4a8_weight_scales",
                 "q4_workspace_size", "q4_scales_to_mma"]:
        assert want in names


def test_library_exports_every_declared_symbol(clib):
    for name in declared_functions():
        assert hasattr(clib, name), name


def test_host_argument_checks(clib):
    P = ctypes.c_void_p
    fake = 0x10000  # never dereferenced: every call below fails validation first
    # K not a multiple of the block
    assert clib.quantize_mxfp4(fake, 1, 4, 48, fake, fake, 0, None) == -2
    assert clib.quantize_int4_g128(fake, 1, 4, 64, fake, fake, None) == -2
    assert clib.gemm_w4a16_int4(fake, fake, fake, 4, 4, 100, fake, None, 0, None) == -2
    # bad dtype, negative sizes, null pointers, misalignment
    assert clib.quantize_mxfp4(fake, 7, 4, 64, fake, fake, 0, None) == -1
    assert clib.quantize_int4_g128(fake, 1, -1, 128, fake, fake, None) == -1
    assert clib.gemm_w4a16_int4(None, fake, fake, 4, 4, 128, fake, None, 0, None) == -1
    assert clib.gemm_w4a16_int4(fake + 2, fake, fake, 4, 4, 128, fake, None, 0, None) == -1
    # NVFP4 quantize needs its workspace
    assert clib.quantize_nvfp4(fake, 1, 4, 64, fake, fake, 0, fake, None, 0, None) == -6
    # FP4-weight W4A16: K % 128, a missing tensor scale, misaligned NVFP4 scales
    assert clib.gemm_w4a16_nvfp4(fake, fake, fake, fake, 4, 4, 100, fake, None, 0, None) == -2
    assert clib.gemm_w4a16_mxfp4(fake, fake, fake, 4, 4, 64, fake, None, 0, None) == -2
    assert clib.gemm_w4a16_nvfp4(fake, fake, fake, None, 4, 4, 128, fake, None, 0, None) == -1
    # FP8 blockwise: K % 128, N % 128, rows % 128 for weight blocks, bad block height,
    # bad output dtype, misaligned operands
    assert clib.quantize_fp8_blockwise(fake, 1, 4, 100, 1, fake, fake, None) == -2
    assert clib.quantize_fp8_blockwise(fake, 1, 100, 128, 128, fake, fake, None) == -2
    assert clib.quantize_fp8_blockwise(fake, 1, 4, 128, 2, fake, fake, None) == -1
    assert clib.quantize_fp8_blockwise(fake + 8, 1, 4, 128, 1, fake, fake, None) == -1
    assert clib.gemm_fp8_blockwise(fake, fake, fake, fake, 4, 128, 100, fake, 1, None, 0, None) == -2
    assert clib.gemm_fp8_blockwise(fake, fake, fake, fake, 4, 100, 128, fake, 1, None, 0, None) == -2
    assert clib.gemm_fp8_blockwise(fake, fake, fake, fake, 4, 128, 128, fake, 2, None, 0, None) == -1
    assert clib.gemm_fp8_blockwise(fake + 4, fake, fake, fake, 4, 128, 128, fake, 1, None, 0, None) == -1
    assert clib.gemm_fp8_blockwise(None, fake, fake, fake, 0, 128, 128, fake, 1, None, 0, None) == 0
    # W4A8: K % 128, N % 128, misaligned weight scales or output, bad output dtype
    assert clib.gemm_w4a8(fake, fake, fake, fake, 4, 128, 100, fake, 1, None, 0, None) == -2
    assert clib.gemm_w4a8(fake, fake, fake, fake, 4, 100, 128, fake, 1, None, 0, None) == -2
    assert clib.gemm_w4a8(fake, fake, fake, fake + 4, 4, 128, 128, fake, 1, None, 0, None) == -1
    assert clib.gemm_w4a8(fake, fake, fake, fake, 4, 128, 128, fake + 8, 1, None, 0, None) == -1
    assert clib.gemm_w4a8(fake, fake, fake, fake, 4, 128, 128, fake, 2, None, 0, None) == -1
    assert clib.w4a8_weight_scales(fake, 4, 100, fake, None) == -2
    assert clib.w4a8_weight_scales(fake + 1, 4, 128, fake, None) == -1
    assert clib.gemm_w4a16_nvfp4(fake, fake, fake + 1, fake, 4, 4, 128, fake, None, 0, None) == -1
    assert clib.gemm_w4a16_mxfp4(None, fake, fake, 4, 4, 128, fake, None, 0, None) == -1
    # fused MXFP4 GEMM: K % 256, a bad activation or output dtype (all checked before B)
    assert clib.gemm_w4a4_mxfp4_fused(fake, 1, None, 4, 4, 128, fake, 1, fake, 1 << 20, None) == -2
    assert clib.gemm_w4a4_mxfp4_fused(fake, 5, None, 4, 4, 256, fake, 1, fake, 1 << 20, None) == -1
    assert clib.gemm_w4a4_mxfp4_fused(fake, 1, None, 4, 4, 256, fake, 2, fake, 1 << 20, None) == -1
    # grouped MoE: the weights operand must be given, quantized, with a known scale layout
    import int4_gemm_gb300 as q4
    args = (fake, 8, 256, fake, fake, 16, 2)
    assert clib.grouped_gemm_moe(*args, None, 256, fake, fake, 1 << 30, None) == -1
    raw = q4._Operand(fake, 1, fake, fake, 1, fake)
    assert clib.grouped_gemm_moe(*args, ctypes.byref(raw), 256, fake, fake, 1 << 30, None) == -1
    bad = q4._Operand(None, 0, fake, fake, 7, fake)
    assert clib.grouped_gemm_moe(*args, ctypes.byref(bad), 256, fake, fake, 1 << 30, None) == -1
    # an unknown rounding mode
    assert clib.quantize_mxfp4_ex(fake, 1, 4, 64, fake, fake, 0, 2, None) == -1
    assert clib.quantize_nvfp4_ex(fake, 1, 4, 64, fake, fake, 0, -1, fake, fake, 256, None) == -1
    # the read probe: 16-byte aligned source, whole 16-byte words, a sink
    assert clib.q4_read_probe(None, 16, fake, None) == -1
    assert clib.q4_read_probe(fake + 1, 16, fake, None) == -1
    assert clib.q4_read_probe(fake, 17, fake, None) == -1
    assert clib.q4_read_probe(fake, 16, None, None) == -1
    assert clib.q4_read_probe(fake, 0, None, None) == 0
    # empty problems are no-ops
    assert clib.quantize_int4_g128(None, 1, 0, 128, None, None, None) == 0
    assert clib.gemm_w4a16_int4(None, None, None, 0, 4, 128, None, None, 0, None) == 0
    assert clib.gemm_w4a16_mxfp4(None, None, None, 0, 4, 128, None, None, 0, None) == 0


def test_workspace_sizes(clib):
    for op in (3, 5, 6, 7, 8):  # W4A16 (INT4, NVFP4, MXFP4), FP8 blockwise, W4A8: none
        assert clib.q4_workspace_size(op, 16, 8192, 8192) == 0
    n = clib.q4_workspace_size(1, 8192, 28672, 8192)
    assert n >= 8192 * 4096 + 28672 * 4096  # room for both operands' codes
    assert clib.q4_mma_scales_bytes(130, 5) == 256 * 8
    # the fused MXFP4 GEMM: the gate's 256 bytes, then what the two-launch call uses
    assert clib.q4_workspace_size(9, 256, 2048, 7168) == 256 + clib.q4_workspace_size(2, 256, 2048, 7168)
    assert clib.q4_workspace_size_moe(4096, 2048, 7168, 64, 32768) > 4096 * 3584


def test_status_strings(clib):
    for s in (0, -1, -2, -3, -4, -5, -6):
        assert clib.q4_status_string(s)

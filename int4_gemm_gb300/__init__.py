"""Python binding of the q4gemm C ABI (``include/q4gemm.h``).

Argument marshalling only: tensors are passed by ``data_ptr()`` together with
torch's current CUDA stream, and every step runs in the library's kernels.
PyTorch provides device memory (outputs and workspaces are torch tensors
allocated here, on the caller's side of the ABI) and streams.  There is no
fallback: if ``libq4gemm.so`` is missing or a call fails, an exception is
raised.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Union

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libq4gemm.so")

Q4_OK = 0
F32, BF16, F16 = 0, 1, 2
ROWMAJOR, MMA = 0, 1
OP_QUANTIZE_NVFP4, OP_GEMM_W4A4_NVFP4, OP_GEMM_W4A4_MXFP4, OP_GEMM_W4A16_INT4 = 0, 1, 2, 3
OP_GROUPED_GEMM_MOE, OP_GEMM_W4A16_NVFP4, OP_GEMM_W4A16_MXFP4 = 4, 5, 6
OP_GEMM_FP8_BLOCKWISE, OP_GEMM_W4A8 = 7, 8
OP_GEMM_W4A4_MXFP4_FUSED = 9

_DTYPE = {torch.float32: F32, torch.bfloat16: BF16, torch.float16: F16}
_LAYOUT = {"rowmajor": ROWMAJOR, "mma": MMA}
_ROUNDING = {"pages": 0, "rne": 1}  # q4_rounding: E2M1 ties to the smaller magnitude / to even

_lib: Optional[ctypes.CDLL] = None


class Q4Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = _lib.q4_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{fn} failed: {msg} ({status})")
        self.status = status


class _Operand(ctypes.Structure):
    _fields_ = [("raw", ctypes.c_void_p), ("raw_dtype", ctypes.c_int),
                ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("scale_layout", ctypes.c_int), ("tensor_scale", ctypes.c_void_p)]


def _sig(lib, name, restype, *argtypes):
    f = getattr(lib, name)
    f.restype = restype
    f.argtypes = list(argtypes)


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library (built by ``__graft_entry__.build()`` or
    ``python -m int4_gemm_gb300.build``).  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m int4_gemm_gb300.build`")
    lib = ctypes.CDLL(path)
    P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    _sig(lib, "q4_workspace_size", SZ, I, I64, I64, I64)
    _sig(lib, "q4_workspace_size_moe", SZ, I64, I64, I64, I, I64)
    _sig(lib, "q4_mma_scales_bytes", SZ, I64, I64)
    _sig(lib, "quantize_nvfp4", I, P, I, I64, I64, P, P, I, P, P, SZ, P)
    _sig(lib, "quantize_mxfp4", I, P, I, I64, I64, P, P, I, P)
    _sig(lib, "quantize_nvfp4_ex", I, P, I, I64, I64, P, P, I, I, P, P, SZ, P)
    _sig(lib, "quantize_mxfp4_ex", I, P, I, I64, I64, P, P, I, I, P)
    _sig(lib, "quantize_int4_g128", I, P, I, I64, I64, P, P, P)
    _sig(lib, "q4_scales_to_mma", I, P, I64, I64, P, P)
    op = ctypes.POINTER(_Operand)
    _sig(lib, "gemm_w4a4_nvfp4", I, op, op, I64, I64, I64, P, I, P, SZ, P)
    _sig(lib, "gemm_w4a4_mxfp4", I, op, op, I64, I64, I64, P, I, P, SZ, P)
    _sig(lib, "gemm_w4a4_mxfp4_fused", I, P, I, op, I64, I64, I64, P, I, P, SZ, P)
    _sig(lib, "gemm_w4a16_int4", I, P, P, P, I64, I64, I64, P, P, SZ, P)
    _sig(lib, "gemm_w4a16_nvfp4", I, P, P, P, P, I64, I64, I64, P, P, SZ, P)
    _sig(lib, "gemm_w4a16_mxfp4", I, P, P, P, I64, I64, I64, P, P, SZ, P)
    _sig(lib, "grouped_gemm_moe", I, P, I64, I64, P, P, I64, I, op, I64, P, P, SZ, P)
    _sig(lib, "quantize_fp8_blockwise", I, P, I, I64, I64, I, P, P, P)
    _sig(lib, "gemm_fp8_blockwise", I, P, P, P, P, I64, I64, I64, P, I, P, SZ, P)
    _sig(lib, "w4a8_weight_scales", I, P, I64, I64, P, P)
    _sig(lib, "gemm_w4a8", I, P, P, P, P, I64, I64, I64, P, I, P, SZ, P)
    _sig(lib, "q4_sync_status", I, P)
    _sig(lib, "q4_status_string", ctypes.c_char_p, I)
    _sig(lib, "q4_set_wait_timeout_ms", I, I)
    _sig(lib, "q4_selftest_wait_timeout", I, P)
    _sig(lib, "q4_read_probe_sink_words", SZ)
    _sig(lib, "q4_read_probe", I, P, SZ, P, P)
    _sig(lib, "gemm_w4a4_nvfp4_noalloc", I, P, I, op, I64, I64, I64, P, I, P)
    _sig(lib, "q4_noalloc_scratch_bytes", SZ)
    _sig(lib, "q4_noalloc_required_bytes", SZ, I64, I64)
    _lib = lib
    return lib


def lib() -> ctypes.CDLL:
    return load()


def _check(fn: str, status: int):
    if status != Q4_OK:
        raise Q4Error(fn, status)


# The current stream's handle without building a Stream object (a few us per
# call otherwise); the public route where this build of torch lacks it.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream=None) -> int:
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _cuda2d(x: torch.Tensor, name: str) -> torch.Tensor:
    if not x.is_cuda or x.dim() != 2 or not x.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 2-D CUDA tensor")
    return x


def _out(out: Optional[torch.Tensor], M: int, N: int, dtype: torch.dtype, device) -> torch.Tensor:
    """A new [M, N] output, or the caller's, checked against the call."""
    if out is None:
        return torch.empty((M, N), dtype=dtype, device=device)
    if (tuple(out.shape) != (M, N) or out.dtype != dtype or out.device != torch.device(device)
            or not out.is_contiguous()):
        raise ValueError(f"out must be a contiguous {dtype} tensor of shape ({M}, {N}) on {device}")
    return out


def _empty(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 0), dtype=torch.uint8, device=device)


def workspace(op: int, M: int, N: int, K: int, device) -> torch.Tensor:
    n = lib().q4_workspace_size(op, M, N, K)
    ws = _empty(max(n, 256), device)
    if op == OP_GEMM_W4A4_MXFP4_FUSED:
        ws[:256].zero_()  # the grid gate's counters start at zero
    return ws


def mma_scales_bytes(rows: int, nsf: int) -> int:
    return int(lib().q4_mma_scales_bytes(rows, nsf))


# --------------------------------------------------------------------------- quantizers

def quantize_nvfp4(x: torch.Tensor, scale_layout: str = "rowmajor", rounding: str = "pages",
                   stream=None):
    """-> (codes u8 [rows, K/2], scales u8, tensor_scale f32 [1]).
    rounding: "pages" (E2M1 ties to the smaller magnitude) or "rne"."""
    _cuda2d(x, "x")
    rows, K = x.shape
    dev = x.device
    codes = torch.empty((rows, K // 2), dtype=torch.uint8, device=dev)
    lay = _LAYOUT[scale_layout]
    if lay == ROWMAJOR:
        scales = torch.empty((rows, K // 16), dtype=torch.uint8, device=dev)
    else:
        scales = _empty(mma_scales_bytes(rows, K // 16), dev)
    ts = torch.empty(1, dtype=torch.float32, device=dev)
    ws = workspace(OP_QUANTIZE_NVFP4, rows, 0, K, dev)
    _check("quantize_nvfp4", lib().quantize_nvfp4_ex(
        x.data_ptr(), _DTYPE[x.dtype], rows, K, codes.data_ptr(), scales.data_ptr(), lay,
        _ROUNDING[rounding], ts.data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream)))
    return codes, scales, ts


def quantize_mxfp4(x: torch.Tensor, scale_layout: str = "rowmajor", rounding: str = "pages",
                   stream=None):
    """-> (codes u8 [rows, K/2], scales u8).
    rounding: "pages" (E2M1 ties to the smaller magnitude) or "rne"."""
    _cuda2d(x, "x")
    rows, K = x.shape
    dev = x.device
    codes = torch.empty((rows, K // 2), dtype=torch.uint8, device=dev)
    lay = _LAYOUT[scale_layout]
    if lay == ROWMAJOR:
        scales = torch.empty((rows, K // 32), dtype=torch.uint8, device=dev)
    else:
        scales = _empty(mma_scales_bytes(rows, K // 32), dev)
    _check("quantize_mxfp4", lib().quantize_mxfp4_ex(
        x.data_ptr(), _DTYPE[x.dtype], rows, K, codes.data_ptr(), scales.data_ptr(), lay,
        _ROUNDING[rounding], _stream(stream)))
    return codes, scales


def quantize_int4_g128(x: torch.Tensor, stream=None):
    """-> (codes u8 [rows, K/2], scales int16 [rows, K/128] holding FP16 bits)."""
    _cuda2d(x, "x")
    rows, K = x.shape
    codes = torch.empty((rows, K // 2), dtype=torch.uint8, device=x.device)
    scales = torch.empty((rows, K // 128), dtype=torch.int16, device=x.device)
    _check("quantize_int4_g128", lib().quantize_int4_g128(
        x.data_ptr(), _DTYPE[x.dtype], rows, K, codes.data_ptr(), scales.data_ptr(),
        _stream(stream)))
    return codes, scales


def scales_to_mma(src: torch.Tensor, stream=None) -> torch.Tensor:
    _cuda2d(src, "src")
    rows, nsf = src.shape
    dst = _empty(mma_scales_bytes(rows, nsf), src.device)
    _check("q4_scales_to_mma", lib().q4_scales_to_mma(src.data_ptr(), rows, nsf, dst.data_ptr(),
                                                      _stream(stream)))
    return dst


# --------------------------------------------------------------------------- GEMMs

@dataclass
class Fp4Operand:
    """A quantized FP4 operand as returned by quantize_nvfp4 / quantize_mxfp4."""
    codes: torch.Tensor
    scales: torch.Tensor
    scale_layout: str = "rowmajor"
    tensor_scale: Optional[torch.Tensor] = None


def _operand(x: Union[torch.Tensor, Fp4Operand], K: int) -> tuple[_Operand, int]:
    if isinstance(x, Fp4Operand):
        _cuda2d(x.codes, "operand codes")
        if x.codes.shape[1] * 2 != K:
            raise ValueError(f"operand codes hold K = {x.codes.shape[1] * 2}, not {K}")
        return _Operand(None, 0, x.codes.data_ptr(), x.scales.data_ptr(), _LAYOUT[x.scale_layout],
                        _ptr(x.tensor_scale)), x.codes.shape[0]
    _cuda2d(x, "operand")
    if x.shape[1] != K:
        raise ValueError(f"operand has K = {x.shape[1]}, not {K}")
    return _Operand(x.data_ptr(), _DTYPE[x.dtype], None, None, 0, None), x.shape[0]


def _gemm_fp4(fn: str, op: int, A, B, K: int, out_dtype: torch.dtype, stream=None, ws=None,
              out=None) -> torch.Tensor:
    a, M = _operand(A, K)
    b, N = _operand(B, K)
    dev = (A.codes if isinstance(A, Fp4Operand) else A).device
    C = _out(out, M, N, out_dtype, dev)
    if ws is None:
        ws = workspace(op, M, N, K, dev)
    _check(fn, getattr(lib(), fn)(ctypes.byref(a), ctypes.byref(b), M, N, K, C.data_ptr(),
                                  _DTYPE[out_dtype], ws.data_ptr(), ws.numel(), _stream(stream)))
    return C


def gemm_w4a4_nvfp4(A, B, K: int, out_dtype=torch.bfloat16, stream=None, ws=None,
                    out=None) -> torch.Tensor:
    """C = A_hat . B_hat^T; A and B are raw tensors (quantized on the fly) or
    Fp4Operand.  ``ws`` (from :func:`workspace`) and ``out`` may be given to
    keep allocations out of a CUDA-graph capture."""
    return _gemm_fp4("gemm_w4a4_nvfp4", OP_GEMM_W4A4_NVFP4, A, B, K, out_dtype, stream, ws, out)


def gemm_w4a4_mxfp4(A, B, K: int, out_dtype=torch.bfloat16, stream=None, ws=None,
                    out=None) -> torch.Tensor:
    return _gemm_fp4("gemm_w4a4_mxfp4", OP_GEMM_W4A4_MXFP4, A, B, K, out_dtype, stream, ws, out)


def gemm_w4a4_mxfp4_fused(A: torch.Tensor, B, K: int, out_dtype=torch.bfloat16, stream=None,
                          ws=None, out=None) -> torch.Tensor:
    """gemm_w4a4_mxfp4 of a raw A in one launch: the GEMM quantizes A in its
    prologue.  ``ws`` must come from ``workspace(OP_GEMM_W4A4_MXFP4_FUSED,
    ...)`` (its first 256 bytes are the gate's counters, zero before the first
    call; each call leaves them zero)."""
    _cuda2d(A, "A")
    if A.shape[1] != K:
        raise ValueError(f"A has K = {A.shape[1]}, not {K}")
    b, N = _operand(B, K)
    M = A.shape[0]
    C = _out(out, M, N, out_dtype, A.device)
    if ws is None:
        ws = workspace(OP_GEMM_W4A4_MXFP4_FUSED, M, N, K, A.device)
    _check("gemm_w4a4_mxfp4_fused",
           lib().gemm_w4a4_mxfp4_fused(A.data_ptr(), _DTYPE[A.dtype], ctypes.byref(b), M, N, K,
                                       C.data_ptr(), _DTYPE[out_dtype], ws.data_ptr(), ws.numel(),
                                       _stream(stream)))
    return C


def gemm_w4a4_nvfp4_noalloc(A: torch.Tensor, B: Fp4Operand, K: int, out_dtype=torch.bfloat16,
                            out=None, stream=None) -> torch.Tensor:
    """gemm_w4a4_nvfp4 with raw activations for callers that cannot provide a
    workspace: the quantized activations go to the library's fixed 16 MiB
    per-GPU scratch array (see include/q4gemm.h).  B must carry MMA-layout
    scales.  Calls that overlap on the GPU share that scratch and race."""
    if not isinstance(A, torch.Tensor):
        raise ValueError("A must be the raw activation tensor")
    _, M = _operand(A, K)
    b, N = _operand(B, K)
    C = _out(out, M, N, out_dtype, A.device)
    _check("gemm_w4a4_nvfp4_noalloc", lib().gemm_w4a4_nvfp4_noalloc(
        A.data_ptr(), _DTYPE[A.dtype], ctypes.byref(b), M, N, K, C.data_ptr(), _DTYPE[out_dtype],
        _stream(stream)))
    return C


def gemm_w4a16_int4(A: torch.Tensor, Wq: torch.Tensor, Ws: torch.Tensor, out=None,
                    stream=None, ws=None) -> torch.Tensor:
    """C [M, N] bf16 = A [M, K] bf16 . dequant(Wq, Ws)^T.  ``ws``: optional
    workspace (q4_workspace_size gives 0 for this call today)."""
    _cuda2d(A, "A")
    M, K = A.shape
    N = Wq.shape[0]
    C = _out(out, M, N, torch.bfloat16, A.device)
    _check("gemm_w4a16_int4", lib().gemm_w4a16_int4(A.data_ptr(), Wq.data_ptr(), Ws.data_ptr(), M,
                                                     N, K, C.data_ptr(), _ptr(ws), 0 if ws is None else ws.numel(),
                                                     _stream(stream)))
    return C


def gemm_w4a16_nvfp4(A: torch.Tensor, Wq: torch.Tensor, Ws: torch.Tensor, Wg: torch.Tensor,
                     out=None, stream=None, ws=None) -> torch.Tensor:
    """C [M, N] bf16 = A [M, K] bf16 . dequant(W)^T, W NVFP4: codes [N, K/2],
    row-major E4M3 scales [N, K/16], tensor scale Wg (one float32)."""
    _cuda2d(A, "A")
    M, K = A.shape
    N = Wq.shape[0]
    C = _out(out, M, N, torch.bfloat16, A.device)
    _check("gemm_w4a16_nvfp4", lib().gemm_w4a16_nvfp4(A.data_ptr(), Wq.data_ptr(), Ws.data_ptr(),
                                                       Wg.data_ptr(), M, N, K, C.data_ptr(),
                                                       _ptr(ws), 0 if ws is None else ws.numel(),
                                                       _stream(stream)))
    return C


def gemm_w4a16_mxfp4(A: torch.Tensor, Wq: torch.Tensor, Ws: torch.Tensor, out=None,
                     stream=None, ws=None) -> torch.Tensor:
    """C [M, N] bf16 = A [M, K] bf16 . dequant(W)^T, W MXFP4: codes [N, K/2],
    row-major E8M0 scales [N, K/32]."""
    _cuda2d(A, "A")
    M, K = A.shape
    N = Wq.shape[0]
    C = _out(out, M, N, torch.bfloat16, A.device)
    _check("gemm_w4a16_mxfp4", lib().gemm_w4a16_mxfp4(A.data_ptr(), Wq.data_ptr(), Ws.data_ptr(),
                                                       M, N, K, C.data_ptr(), _ptr(ws),
                                                       0 if ws is None else ws.numel(),
                                                       _stream(stream)))
    return C


def quantize_fp8_blockwise(x: torch.Tensor, block_rows: int, codes=None, scales=None,
                           stream=None):
    """FP8 (E4M3) blockwise quantization of x [rows, K] (f32 / bf16 / f16):
    block_rows 128 for weights (128 x 128 blocks), 1 for activations (1 x 128).
    -> (codes u8 [rows, K], scales float32 [rows / block_rows, K / 128])."""
    _cuda2d(x, "x")
    rows, K = x.shape
    if codes is None:
        codes = torch.empty((rows, K), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((rows // max(block_rows, 1), K // 128), dtype=torch.float32,
                             device=x.device)
    _check("quantize_fp8_blockwise", lib().quantize_fp8_blockwise(
        x.data_ptr(), _DTYPE[x.dtype], rows, K, block_rows, codes.data_ptr(), scales.data_ptr(),
        _stream(stream)))
    return codes, scales


def gemm_fp8_blockwise(qa: torch.Tensor, sa: torch.Tensor, qb: torch.Tensor, sb: torch.Tensor,
                       out_dtype=torch.bfloat16, out=None, stream=None) -> torch.Tensor:
    """C [M, N] = sum over 128-wide K blocks of sa * sb * (qa . qb^T): qa E4M3
    [M, K] with sa [M, K/128], qb E4M3 [N, K] with sb [N/128, K/128]."""
    _cuda2d(qa, "qa")
    M, K = qa.shape
    N = qb.shape[0]
    C = _out(out, M, N, out_dtype if out is None else out.dtype, qa.device)
    _check("gemm_fp8_blockwise", lib().gemm_fp8_blockwise(
        qa.data_ptr(), sa.data_ptr(), qb.data_ptr(), sb.data_ptr(), M, N, K, C.data_ptr(),
        _DTYPE[C.dtype], None, 0, _stream(stream)))
    return C


def w4a8_weight_scales(w_scales: torch.Tensor, stream=None) -> torch.Tensor:
    """FP16 INT4 group scales [N, K/128] (as quantize_int4_g128 returns them,
    int16 bits) -> float32 [K/128, N], the layout gemm_w4a8 reads."""
    _cuda2d(w_scales, "w_scales")
    N, KB = w_scales.shape
    out = torch.empty((KB, N), dtype=torch.float32, device=w_scales.device)
    _check("w4a8_weight_scales", lib().w4a8_weight_scales(
        w_scales.data_ptr(), N, KB * 128, out.data_ptr(), _stream(stream)))
    return out


def gemm_w4a8(qa: torch.Tensor, sa: torch.Tensor, w_codes: torch.Tensor, w_scales_kn: torch.Tensor,
              out_dtype=torch.bfloat16, out=None, stream=None) -> torch.Tensor:
    """C [M, N] = sum over 128-wide K blocks of sa * s16 * (qa . q^T): qa E4M3
    [M, K] with sa [M, K/128]; INT4 codes [N, K/2] with w4a8_weight_scales'
    float32 [K/128, N]."""
    _cuda2d(qa, "qa")
    M, K = qa.shape
    N = w_codes.shape[0]
    C = _out(out, M, N, out_dtype if out is None else out.dtype, qa.device)
    _check("gemm_w4a8", lib().gemm_w4a8(
        qa.data_ptr(), sa.data_ptr(), w_codes.data_ptr(), w_scales_kn.data_ptr(), M, N, K,
        C.data_ptr(), _DTYPE[C.dtype], None, 0, _stream(stream)))
    return C


def moe_workspace(T: int, N: int, K: int, E: int, R: int, device,
                  w_scale_layout: str = "mma") -> torch.Tensor:
    n = int(lib().q4_workspace_size_moe(T, N, K, E, R))
    if w_scale_layout == "rowmajor":  # room for the weight scales in the tensor-core layout
        n += E * mma_scales_bytes(N, K // 16)
    return _empty(max(n, 256), device)


def grouped_gemm_moe(tokens: torch.Tensor, expert_offsets: torch.Tensor, row_token: torch.Tensor,
                     w_codes: torch.Tensor, w_scales: torch.Tensor, w_tensor_scales: torch.Tensor,
                     N: int, ws: Optional[torch.Tensor] = None, out=None, stream=None,
                     w_scale_layout: str = "mma") -> torch.Tensor:
    """C [R, N] bf16: routed rows times their expert's NVFP4 weights.
    w_codes [E, N, K/2]; w_scales: E stacked MMA-layout scale tensors, or
    [E, N, K/16] row-major bytes with ``w_scale_layout="rowmajor"``;
    w_tensor_scales [E] float32; expert_offsets [E+1] / row_token [R] int32."""
    _cuda2d(tokens, "tokens")
    T, K = tokens.shape
    E = expert_offsets.numel() - 1
    R = row_token.numel()
    C = _out(out, R, N, torch.bfloat16, tokens.device)
    if ws is None:
        ws = moe_workspace(T, N, K, E, R, tokens.device, w_scale_layout)
    w = _Operand(None, 0, w_codes.data_ptr(), w_scales.data_ptr(), _LAYOUT[w_scale_layout],
                 w_tensor_scales.data_ptr())
    _check("grouped_gemm_moe", lib().grouped_gemm_moe(
        tokens.data_ptr(), T, K, expert_offsets.data_ptr(), row_token.data_ptr(), R, E,
        ctypes.byref(w), N, C.data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream)))
    return C


def sync_status(stream=None) -> int:
    """Synchronize and return (and clear) the first error latched by a kernel."""
    return int(lib().q4_sync_status(_stream(stream)))


def set_wait_timeout_ms(ms: int) -> int:
    return int(lib().q4_set_wait_timeout_ms(ms))


def read_probe(src: torch.Tensor, sink: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Measurement aid: one bare streaming read of ``src`` (q4_read_probe).
    Returns the sink (int32 words, contents meaningless)."""
    if not src.is_cuda or not src.is_contiguous():
        raise ValueError("src must be a contiguous CUDA tensor")
    if sink is None:
        sink = torch.zeros(int(lib().q4_read_probe_sink_words()), dtype=torch.int32, device=src.device)
    _check("q4_read_probe", lib().q4_read_probe(src.data_ptr(), src.numel() * src.element_size(),
                                                sink.data_ptr(), _stream(stream)))
    return sink

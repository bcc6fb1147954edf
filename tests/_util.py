"""Test helpers: tolerance checks and layout permutations (no method arithmetic)."""
import numpy as np

FRO_TOL = 2e-3   # relative Frobenius error of a GEMM output against the FP64 oracle
ROW_TOL = 1e-2   # max |C - R|_ij relative to the L2 norm of oracle row i


def gemm_errors(C, R):
    C = np.asarray(C, np.float64)
    R = np.asarray(R, np.float64)
    fro = np.linalg.norm(C - R) / max(np.linalg.norm(R), 1e-300)
    rown = np.linalg.norm(R, axis=1, keepdims=True)
    mx = float(np.max(np.abs(C - R) / np.maximum(rown, 1e-300))) if R.size else 0.0
    return float(fro), mx


def assert_gemm_close(C, R, fro_tol=FRO_TOL, row_tol=ROW_TOL):
    fro, mx = gemm_errors(C, R)
    assert np.all(np.isfinite(np.asarray(C, np.float64))), "non-finite output"
    assert fro <= fro_tol and mx <= row_tol, f"relative Frobenius {fro:.3e}, max row-relative {mx:.3e}"
    return fro, mx


def to_mma_layout(rowmajor: np.ndarray) -> np.ndarray:
    """Row-major [rows, nsf] scale bytes -> the tensor-core tile layout
    documented in include/q4gemm.h (rows by 128, scale columns by 4)."""
    rows, nsf = rowmajor.shape
    rp, sp = -(-rows // 128) * 128, -(-nsf // 4) * 4
    padded = np.zeros((rp, sp), np.uint8)
    padded[:rows, :nsf] = rowmajor
    t = padded.reshape(rp // 128, 4, 32, sp // 4, 4)      # [R, r/32, r%32, J, s%4]
    t = t.transpose(0, 3, 2, 1, 4)                        # [R, J, r%32, r/32, s%4]
    return np.ascontiguousarray(t).reshape(-1)


def spread(seed, rows, K, lo=-8, hi=8):
    """float32 N(0,1) rows, each scaled by a random power of two."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, K)).astype(np.float32)
    return x * np.exp2(rng.integers(lo, hi, size=(rows, 1))).astype(np.float32)

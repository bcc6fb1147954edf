"""The no-allocation variant of the NVFP4 W4A4 GEMM.

Some callers cannot give the library a workspace (a plugin interface that
passes only inputs and outputs, an engine whose memory pool is fully
reserved).  gemm_w4a4_nvfp4_noalloc keeps its
scratch in a fixed per-GPU device array instead.  These checks call it through
the C ABI and compare it with gemm_w4a4_nvfp4 (the workspace entry point) on
two calls in a row -- the second with different activations, so a scratch
left over from the first call would show -- and check the size limit.  This
file is collected last so that a failure here comes after every other test.
"""
import numpy as np
import pytest
import torch

import int4_gemm_gb300 as q4
import oracle
import workloads
from tests._util import assert_gemm_close

pytestmark = pytest.mark.gpu


def _weights(lib, N, K, seed):
    b = workloads.nvfp4_pair(1, N, K, seed)[1]
    c, s, g = lib.quantize_nvfp4(torch.from_numpy(b).cuda(), scale_layout="mma")
    return b, q4.Fp4Operand(c, s, "mma", g)


def test_noalloc_matches_workspace_entry_point_twice(lib):
    M, N, K = 300, 520, 1024
    b, B = _weights(lib, N, K, seed=41)
    for call, seed in enumerate((42, 43)):
        a = workloads.nvfp4_pair(M, 1, K, seed, a_std=1.0, channel_outliers=True)[0]
        if call == 1:
            a *= 3.0  # a different tensor scale than the first call
        A = workloads.to_bf16(a).cuda()
        want = lib.gemm_w4a4_nvfp4(A, B, K, out_dtype=torch.float32)
        got = lib.gemm_w4a4_nvfp4_noalloc(A, B, K, out_dtype=torch.float32)
        assert lib.sync_status() == 0
        assert_gemm_close(got.cpu().numpy(), want.cpu().numpy(), fro_tol=1e-6, row_tol=1e-6)
        R = oracle.gemm_w4a4_nvfp4(*oracle.quantize_nvfp4(A.float().cpu().numpy()),
                                   *oracle.quantize_nvfp4(b))
        assert_gemm_close(got.cpu().numpy(), R)


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    L = lib.lib()
    cap = L.q4_noalloc_scratch_bytes()
    assert cap == 16 << 20
    K = 8192
    M_ok = 3072
    assert L.q4_noalloc_required_bytes(M_ok, K) <= cap
    assert L.q4_noalloc_required_bytes(4096, K) > cap
    _, B = _weights(lib, 256, K, seed=44)
    A = torch.zeros((4096, K), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(q4.Q4Error) as ei:
        lib.gemm_w4a4_nvfp4_noalloc(A, B, K)
    assert ei.value.status == -7
    # a problem just inside the limit runs
    out = lib.gemm_w4a4_nvfp4_noalloc(A[:M_ok].contiguous(), B, K)
    assert out.shape == (M_ok, 256) and lib.sync_status() == 0

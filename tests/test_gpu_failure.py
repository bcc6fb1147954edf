"""Failure detection on the GPU without a fault: a bounded pipeline wait that
runs out latches Q4_ERR_TIMEOUT, the host reads (and clears) it, and the
context keeps working."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._util import assert_gemm_close

pytestmark = pytest.mark.gpu

Q4_ERR_TIMEOUT = -4


def test_bounded_wait_runs_out_and_the_context_survives(lib):
    assert lib.sync_status() == 0
    prev = lib.set_wait_timeout_ms(50)
    try:
        rc = lib.lib().q4_selftest_wait_timeout(torch.cuda.current_stream().cuda_stream)
        assert rc == 0
        assert lib.sync_status() == Q4_ERR_TIMEOUT  # latched by the kernel ...
        assert lib.sync_status() == 0               # ... and cleared by the read
    finally:
        assert lib.set_wait_timeout_ms(prev) == 50
    # the same context still computes correct results
    M, N, K = 130, 300, 768
    a, b = workloads.nvfp4_pair(M, N, K, seed=77, a_std=1.0, channel_outliers=True)
    C = lib.gemm_w4a4_nvfp4(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), K,
                            out_dtype=torch.float32)
    R = oracle.gemm_w4a4_nvfp4(*oracle.quantize_nvfp4(a), *oracle.quantize_nvfp4(b))
    assert_gemm_close(C.cpu().numpy(), R)
    assert lib.sync_status() == 0

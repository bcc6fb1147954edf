"""W4A8 on the GPU against the oracle: the weight-scale conversion bit for bit,
and the product of FP8 activations ((1, 128) blocks) with INT4 g128 weights
converted to E4M3 on the fly, on shapes with ragged M, one and many K blocks,
K-block counts that do not divide the TMEM slots or the scale-buffer ring, more
tiles than SMs and both output types, plus a sampled check at full size."""
import numpy as np
import pytest
import torch

import int4_gemm_gb300 as q4
import oracle
import workloads
from tests._util import assert_gemm_close

pytestmark = pytest.mark.gpu


def _operands(M, N, K, seed):
    a = workloads.normal(workloads.rng_for(seed, 1), (M, K), 1.0)
    workloads.scale_channels(workloads.rng_for(seed, 5), a)
    w = workloads.int4_weights(N, K, seed)
    return a, w


def test_w4a8_weight_scales_conversion(lib):
    w = workloads.int4_weights(384, 1024, 3)
    _, ws = oracle.quantize_int4_g128(w)
    got = lib.w4a8_weight_scales(torch.from_numpy(ws.view(np.int16)).cuda())
    want = oracle.formats.fp16_decode(ws).astype(np.float32).T
    assert np.array_equal(got.cpu().numpy(), want)


# M <= 128: one CTA per 128 x 128 tile; M > 128: CTA pairs on 256 x 256
# tiles, incl. an odd CTA holding one row (257), N a multiple of 128 but not
# of 256 (the pair tile's second half and its weight scales absent: 384, 640,
# 128), one K block (128)
W4A8_SHAPES = [(128, 128, 128), (1, 128, 1024), (200, 256, 512), (130, 384, 896),
               (2048, 1536, 512), (1000, 2048, 2304), (257, 640, 256), (384, 128, 384),
               (129, 256, 128)]


@pytest.mark.parametrize("shape", W4A8_SHAPES)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_w4a8_gemm(lib, shape, out_dtype):
    M, N, K = shape
    a, w = _operands(M, N, K, seed=sum(shape))
    qa, sa = lib.quantize_fp8_blockwise(torch.from_numpy(a).cuda(), 1)
    wc, ws = oracle.quantize_int4_g128(w)
    wsk = lib.w4a8_weight_scales(torch.from_numpy(ws.view(np.int16)).cuda())
    C = lib.gemm_w4a8(qa, sa, torch.from_numpy(wc).cuda(), wsk, out_dtype=out_dtype)
    R = oracle.gemm_w4a8(*oracle.quantize_fp8_blockwise(a, (1, 128)), wc, ws)
    assert_gemm_close(C.float().cpu().numpy(), R)
    assert lib.sync_status() == 0


def test_w4a8_gemm_repeatable_and_empty(lib):
    M, N, K = 300, 1024, 768
    a, w = _operands(M, N, K, 7)
    qa, sa = lib.quantize_fp8_blockwise(torch.from_numpy(a).cuda(), 1)
    wc, ws = oracle.quantize_int4_g128(w)
    wq = torch.from_numpy(wc).cuda()
    wsk = lib.w4a8_weight_scales(torch.from_numpy(ws.view(np.int16)).cuda())
    C1 = lib.gemm_w4a8(qa, sa, wq, wsk, out_dtype=torch.float32)
    C2 = lib.gemm_w4a8(qa, sa, wq, wsk, out_dtype=torch.float32)
    assert torch.equal(C1, C2)
    assert lib.gemm_w4a8(qa[:0], sa[:0], wq, wsk, out_dtype=torch.float32).shape == (0, N)
    with pytest.raises(q4.Q4Error):
        lib.gemm_w4a8(qa, sa, wq[:100], wsk, out_dtype=torch.float32)
    assert lib.sync_status() == 0


def test_w4a8_gemm_full_size_sampled(lib):
    """The prefill shape (8192 x 28672 x 8192) with INT4 g128 weights: sampled
    activation rows and weight rows against the oracle on those rows (each
    weight row's groups are quantized on their own)."""
    M, N, K = 8192, 28672, 8192
    a = workloads.prefill_activations(M=M, K=K)
    w = workloads.normal(workloads.rng_for(workloads.SEED_BASE + 4, 2), (N, K), 0.02)
    wc_dev, ws_dev = lib.quantize_int4_g128(torch.from_numpy(w).cuda())
    qa, sa = lib.quantize_fp8_blockwise(a.cuda(), 1)
    C = lib.gemm_w4a8(qa, sa, wc_dev, lib.w4a8_weight_scales(ws_dev))
    rows = np.array([0, 1, 127, 128, 4095, 5000, 8190, 8191])
    cols = np.concatenate([np.arange(0, 128), np.arange(12928, 13056), np.arange(N - 128, N)])
    oa = oracle.quantize_fp8_blockwise(a.float().numpy()[rows], (1, 128))
    wc, ws = oracle.quantize_int4_g128(w[cols])
    assert np.array_equal(wc_dev[cols].cpu().numpy(), wc)
    R = oracle.gemm_w4a8(*oa, wc, ws)
    assert_gemm_close(C[rows][:, cols].float().cpu().numpy(), R)
    assert lib.sync_status() == 0

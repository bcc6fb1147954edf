"""FP8 blockwise path on the GPU against the oracle: quantizer codes and scales
bit for bit (activation (1, 128) blocks and weight 128 x 128 blocks, each input
dtype, outliers, zero blocks, negative zeros), the block-promoted GEMM on
shapes with ragged M, one and many K blocks, K-block counts that do not divide
the four TMEM slots, more tiles than SMs and both output types, and a sampled
check of the full-size workload."""
import numpy as np
import pytest
import torch

import int4_gemm_gb300 as q4
import oracle
import workloads
from tests._util import assert_gemm_close

pytestmark = pytest.mark.gpu


def _acts(M, K, seed):
    """float32 activations with outlier channels, a zero block and -0 entries."""
    a = workloads.normal(workloads.rng_for(seed, 1), (M, K), 1.0)
    workloads.scale_channels(workloads.rng_for(seed, 5), a)
    a[0, :128] = 0.0
    if K >= 256:
        a[0, 128:136] = -0.0
    return a


def _weights(N, K, seed):
    w = workloads.normal(workloads.rng_for(seed, 2), (N, K), 0.02)
    w[:, :128] *= np.float32(8.0)          # one K block column with larger scales
    return w


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("shape", [(3, 256), (257, 1024), (64, 7168)])
def test_fp8_activation_quantizer_bit_exact(lib, dtype, shape):
    M, K = shape
    x = torch.from_numpy(_acts(M, K, seed=M + K)).to(dtype)
    codes, scales = lib.quantize_fp8_blockwise(x.cuda(), 1)
    oc, os_ = oracle.quantize_fp8_blockwise(x.float().numpy(), (1, 128))
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    assert lib.sync_status() == 0


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("shape", [(128, 128), (384, 640)])
def test_fp8_weight_quantizer_bit_exact(lib, dtype, shape):
    N, K = shape
    w = _weights(N, K, seed=N + K)
    w[:128, :128] = 0.0                     # an all-zero 128 x 128 block
    x = torch.from_numpy(w).to(dtype)
    codes, scales = lib.quantize_fp8_blockwise(x.cuda(), 128)
    oc, os_ = oracle.quantize_fp8_blockwise(x.float().numpy(), (128, 128))
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    assert lib.sync_status() == 0


def test_fp8_quantizer_values_next_to_e4m3_midpoints(lib):
    """x / s lands on (and one float32 ulp either side of) every E4M3 midpoint."""
    pos = oracle.formats.e4m3_decode(np.arange(0x7F))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    vals = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))])
    vals = vals[vals <= np.float32(448.0)]
    n = -(-vals.size // 127) * 127
    y = np.resize(vals, n).reshape(-1, 127)
    # a block (1, 128) whose amax is exactly 448 has s = 1: x / s = x
    x = np.concatenate([y, np.full((y.shape[0], 1), 448.0, np.float32)], axis=1)
    x[1::2] *= np.float32(-1.0)
    codes, scales = lib.quantize_fp8_blockwise(torch.from_numpy(x).cuda(), 1)
    oc, os_ = oracle.quantize_fp8_blockwise(x, (1, 128))
    assert np.all(os_ == np.float32(1.0))
    assert np.array_equal(codes.cpu().numpy(), oc)


# M <= 128: one CTA per 128 x 128 tile; M > 128: CTA pairs on 256 x 256 tiles,
# incl. an odd CTA holding one row (257), N a multiple of 128 but not of 256
# (the pair tile's second half absent: 640, 128), one K block (128)
FP8_SHAPES = [(128, 128, 128), (1, 128, 1024), (200, 256, 512), (130, 384, 896),
              (2048, 1536, 512), (1000, 2048, 1280), (257, 640, 256), (384, 128, 384),
              (129, 256, 128)]


@pytest.mark.parametrize("shape", FP8_SHAPES)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_fp8_blockwise_gemm(lib, shape, out_dtype):
    M, N, K = shape
    a, w = _acts(M, K, seed=sum(shape)), _weights(N, K, seed=2 * sum(shape))
    qa, sa = lib.quantize_fp8_blockwise(torch.from_numpy(a).cuda(), 1)
    qb, sb = lib.quantize_fp8_blockwise(torch.from_numpy(w).cuda(), 128)
    C = lib.gemm_fp8_blockwise(qa, sa, qb, sb, out_dtype=out_dtype)
    R = oracle.gemm_fp8_blockwise(*oracle.quantize_fp8_blockwise(a, (1, 128)),
                                  *oracle.quantize_fp8_blockwise(w, (128, 128)))
    assert_gemm_close(C.float().cpu().numpy(), R)
    assert lib.sync_status() == 0


def test_fp8_blockwise_gemm_repeatable_and_empty(lib):
    M, N, K = 300, 1024, 768
    a, w = _acts(M, K, 5), _weights(N, K, 6)
    qa, sa = lib.quantize_fp8_blockwise(torch.from_numpy(a).cuda(), 1)
    qb, sb = lib.quantize_fp8_blockwise(torch.from_numpy(w).cuda(), 128)
    C1 = lib.gemm_fp8_blockwise(qa, sa, qb, sb, out_dtype=torch.float32)
    C2 = lib.gemm_fp8_blockwise(qa, sa, qb, sb, out_dtype=torch.float32)
    assert torch.equal(C1, C2)
    E = lib.gemm_fp8_blockwise(qa[:0], sa[:0], qb, sb, out_dtype=torch.float32)
    assert E.shape == (0, N)
    with pytest.raises(q4.Q4Error):
        lib.gemm_fp8_blockwise(qa, sa, qb[:100], sb, out_dtype=torch.float32)
    assert lib.sync_status() == 0


def test_fp8_blockwise_gemm_full_size_sampled(lib):
    """The bench workload (activations 8192 x 8192 quantized on the device, B
    28672 x 8192): sampled rows and weight block rows against the oracle (each
    128 x 128 weight block is quantized on its own, so a block row of B
    quantizes alone to the same codes and scales)."""
    M, N, K = 8192, 28672, 8192
    a = workloads.prefill_activations(M=M, K=K)
    b = workloads.normal(workloads.rng_for(workloads.SEED_BASE + 4, 2), (N, K), 0.02)
    qa, sa = lib.quantize_fp8_blockwise(a.cuda(), 1)
    qb, sb = lib.quantize_fp8_blockwise(torch.from_numpy(b).cuda(), 128)
    C = lib.gemm_fp8_blockwise(qa, sa, qb, sb)
    rows = np.array([0, 1, 127, 128, 4095, 5000, 8190, 8191])
    nbs = [0, 101, N // 128 - 1]
    cols = np.concatenate([np.arange(nb * 128, nb * 128 + 128) for nb in nbs])
    oa = oracle.quantize_fp8_blockwise(a.float().numpy()[rows], (1, 128))
    ob = oracle.quantize_fp8_blockwise(b[cols], (128, 128))
    assert np.array_equal(qa[rows].cpu().numpy(), oa[0])
    assert np.array_equal(qb[cols].cpu().numpy(), ob[0])
    assert np.array_equal(sb[nbs].cpu().numpy(), ob[1])
    R = oracle.gemm_fp8_blockwise(*oa, *ob)
    assert_gemm_close(C[rows][:, cols].float().cpu().numpy(), R)
    assert lib.sync_status() == 0

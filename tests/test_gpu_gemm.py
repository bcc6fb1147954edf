"""GPU GEMMs against the FP64 oracle on shapes that span several tiles, ragged
M / N tails, single and many K blocks, more tiles than SMs, both operand paths
(raw operands quantized on the fly, pre-quantized operands in either scale
layout) and both output types."""
import ctypes

import numpy as np
import pytest
import torch

import int4_gemm_gb300 as q4
import oracle
import workloads
from tests._util import assert_gemm_close, to_mma_layout

pytestmark = pytest.mark.gpu

W4A4_SHAPES = [(16, 256, 512), (1, 256, 256), (130, 300, 768), (257, 520, 1024),
               (128, 256, 4096), (2048, 4096, 256), (300, 1000, 512), (1000, 2048, 1024)]


def _nv_pair(M, N, K, seed):
    a, b = workloads.nvfp4_pair(M, N, K, seed, a_std=1.0, channel_outliers=True)
    return a, b


@pytest.mark.parametrize("shape", W4A4_SHAPES)
def test_w4a4_nvfp4_raw_operands(lib, shape):
    M, N, K = shape
    a, b = _nv_pair(M, N, K, seed=sum(shape))
    C = lib.gemm_w4a4_nvfp4(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), K,
                            out_dtype=torch.float32)
    R = oracle.gemm_w4a4_nvfp4(*oracle.quantize_nvfp4(a), *oracle.quantize_nvfp4(b))
    assert_gemm_close(C.cpu().numpy(), R)
    assert lib.sync_status() == 0


# More than 76 output tiles of 128 x 256 and M above one tile: CTA pairs
# (2-SM MMA, 256 x 256 tiles).  1100 rows = 9 M tiles (the last pair's second
# CTA lies past M); N = 2350 ends in a tile whose upper 128-row B half lies
# entirely past N, N = 2600 in a partial half.
PAIR_SHAPES = [(1100, 2350, 768), (1024, 2600, 512)]


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("shape", PAIR_SHAPES)
def test_w4a4_cta_pairs(lib, fmt, shape):
    M, N, K = shape
    if fmt == "nvfp4":
        a, b = _nv_pair(M, N, K, seed=M + 7)
        C = lib.gemm_w4a4_nvfp4(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), K,
                                out_dtype=torch.float32)
        R = oracle.gemm_w4a4_nvfp4(*oracle.quantize_nvfp4(a), *oracle.quantize_nvfp4(b))
    else:
        a, b = workloads.mxfp4_pair(M, N, K, seed=M + 9)
        C = lib.gemm_w4a4_mxfp4(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), K,
                                out_dtype=torch.float32)
        R = oracle.gemm_w4a4_mxfp4(*oracle.quantize_mxfp4(a), *oracle.quantize_mxfp4(b))
    assert_gemm_close(C.cpu().numpy(), R)
    assert lib.sync_status() == 0


@pytest.mark.parametrize("layout", ["rowmajor", "mma"])
@pytest.mark.parametrize("shape", [(130, 300, 768), (512, 768, 1024)])
def test_w4a4_nvfp4_prequantized_bf16(lib, layout, shape):
    M, N, K = shape
    a, b = _nv_pair(M, N, K, seed=3 + M)
    ad = workloads.to_bf16(a).cuda()
    qa = q4.Fp4Operand(*_q(lib.quantize_nvfp4(ad, scale_layout=layout), layout))
    qb = q4.Fp4Operand(*_q(lib.quantize_nvfp4(torch.from_numpy(b).cuda(), scale_layout=layout), layout))
    C = lib.gemm_w4a4_nvfp4(qa, qb, K, out_dtype=torch.bfloat16)
    R = oracle.gemm_w4a4_nvfp4(*oracle.quantize_nvfp4(ad.float().cpu().numpy()), *oracle.quantize_nvfp4(b))
    assert_gemm_close(C.float().cpu().numpy(), R)


def _q(t, layout):
    codes, scales, g = t
    return codes, scales, layout, g


@pytest.mark.parametrize("shape", W4A4_SHAPES)
def test_w4a4_mxfp4_raw_operands(lib, shape):
    M, N, K = shape
    a, b = workloads.mxfp4_pair(M, N, K, seed=sum(shape) + 1)
    ad = workloads.to_bf16(a).cuda()
    C = lib.gemm_w4a4_mxfp4(ad, torch.from_numpy(b).cuda(), K, out_dtype=torch.bfloat16)
    R = oracle.gemm_w4a4_mxfp4(*oracle.quantize_mxfp4(ad.float().cpu().numpy()), *oracle.quantize_mxfp4(b))
    assert_gemm_close(C.float().cpu().numpy(), R)


# MXFP4 with raw activations: the GEMM quantizes them itself, in a prologue,
# into the workspace.  Shapes for each launch form: split-K on 128-wide N
# tiles (the MoE shape; a small one), one CTA per 128 x 256 tile (one K
# block, so no split), and CTA pairs.
PROLOGUE_SHAPES = [(256, 2048, 7168), (100, 512, 1024), (64, 20480, 256), (1000, 6144, 512)]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("shape", PROLOGUE_SHAPES)
def test_w4a4_mxfp4_prologue_quantization(lib, dtype, shape):
    """The codes and tensor-core-layout scales the fused call's prologue leaves
    in the workspace are the oracle's bit for bit, the product matches the
    oracle's and the two-launch call's bit for bit, and the gate's counters
    are zero again afterwards."""
    M, N, K = shape
    a, b = workloads.mxfp4_pair(M, N, K, seed=sum(shape) + 3)
    ad = torch.from_numpy(a).to(dtype).cuda()
    cb, sb = lib.quantize_mxfp4(torch.from_numpy(b).cuda(), scale_layout="mma")
    Bq = q4.Fp4Operand(cb, sb, "mma")
    ws = lib.workspace(q4.OP_GEMM_W4A4_MXFP4_FUSED, M, N, K, ad.device)
    C = lib.gemm_w4a4_mxfp4_fused(ad, Bq, K, out_dtype=torch.float32, ws=ws)
    assert lib.sync_status() == 0
    oa = oracle.quantize_mxfp4(ad.float().cpu().numpy())
    wsh = ws.cpu().numpy()
    assert not wsh[:256].any()
    codes0 = 256  # after the gate's 256 bytes
    assert np.array_equal(wsh[codes0:codes0 + M * K // 2].reshape(M, K // 2), oa[0])
    sf0 = codes0 + -(-(M * K // 2) // 256) * 256  # the scales follow the codes, 256-byte aligned
    want = to_mma_layout(oa[1])
    valid = to_mma_layout(np.ones_like(oa[1])) == 1  # rows past M are padding
    assert np.array_equal(wsh[sf0:sf0 + want.size][valid], want[valid])
    R = oracle.gemm_w4a4_mxfp4(*oa, *oracle.quantize_mxfp4(b))
    assert_gemm_close(C.cpu().numpy(), R)
    C2 = lib.gemm_w4a4_mxfp4(ad, Bq, K, out_dtype=torch.float32)
    assert torch.equal(C, C2)


def test_w4a4_mxfp4_fused_gate_reuse(lib):
    """One workspace serves a run of fused calls with different grids (split-K
    clusters, one CTA per tile, pairs) back to back, unsynchronized: each
    call's gate starts from the zero the previous one left, and every product
    equals the two-launch call's."""
    shapes = [(256, 2048, 7168), (1000, 6144, 512), (100, 512, 1024), (64, 20480, 256),
              (256, 2048, 7168)]
    cap = max(q4.lib().q4_workspace_size(q4.OP_GEMM_W4A4_MXFP4_FUSED, *s) for s in shapes)
    ws = torch.zeros(cap, dtype=torch.uint8, device="cuda")
    runs = []
    for i, (M, N, K) in enumerate(shapes * 2):
        a, b = workloads.mxfp4_pair(M, N, K, seed=100 + i)
        ad, bd = torch.from_numpy(a).to(torch.bfloat16).cuda(), torch.from_numpy(b).cuda()
        cb, sb = lib.quantize_mxfp4(bd, scale_layout="mma")
        Bq = q4.Fp4Operand(cb, sb, "mma")
        runs.append((ad, Bq, K, lib.gemm_w4a4_mxfp4_fused(ad, Bq, K, ws=ws)))
    torch.cuda.synchronize()
    assert lib.sync_status() == 0
    assert not ws[:256].any()
    for ad, Bq, K, C in runs:
        assert torch.equal(C, lib.gemm_w4a4_mxfp4(ad, Bq, K))


def test_w4a4_mxfp4_fused_checks(lib):
    """The fused call checks its arguments on the host: K against A, the
    workspace's size, and an empty problem launches nothing."""
    M, N, K = 64, 256, 512
    a, b = workloads.mxfp4_pair(M, N, K, seed=7)
    ad = torch.from_numpy(a).to(torch.bfloat16).cuda()
    cb, sb = lib.quantize_mxfp4(torch.from_numpy(b).cuda(), scale_layout="mma")
    Bq = q4.Fp4Operand(cb, sb, "mma")
    with pytest.raises(ValueError):
        lib.gemm_w4a4_mxfp4_fused(ad, Bq, 2 * K)
    small = torch.zeros(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(RuntimeError):
        lib.gemm_w4a4_mxfp4_fused(ad, Bq, K, ws=small)
    C = lib.gemm_w4a4_mxfp4_fused(ad[:0], Bq, K)
    assert C.shape == (0, N)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("shape", [(256, 2048, 7168), (128, 4096, 8192), (100, 1000, 1024),
                                   (64, 9000, 512)])
def test_w4a4_splitk_reductions_agree(lib, fmt, shape):
    """Few output tiles: split K over a cluster.  With a full workspace the
    ranks' partial sums meet in it (L2); without one (the C call with ws =
    NULL) they meet in distributed shared memory.  Both add them in rank order,
    so the results agree bit for bit."""
    M, N, K = shape
    a, b = (_nv_pair if fmt == "nvfp4" else workloads.mxfp4_pair)(M, N, K, seed=M + K)
    quant = lib.quantize_nvfp4 if fmt == "nvfp4" else lib.quantize_mxfp4
    qa, qb = quant(torch.from_numpy(a).cuda(), scale_layout="mma"), quant(torch.from_numpy(b).cuda(), scale_layout="mma")
    A = q4.Fp4Operand(*qa[:2], "mma", qa[2] if fmt == "nvfp4" else None)
    B = q4.Fp4Operand(*qb[:2], "mma", qb[2] if fmt == "nvfp4" else None)
    f = lib.gemm_w4a4_nvfp4 if fmt == "nvfp4" else lib.gemm_w4a4_mxfp4
    C1 = f(A, B, K, out_dtype=torch.float32)  # full workspace
    C2 = torch.empty_like(C1)
    oa, ob = q4._operand(A, K)[0], q4._operand(B, K)[0]
    fn = lib.lib().gemm_w4a4_nvfp4 if fmt == "nvfp4" else lib.lib().gemm_w4a4_mxfp4
    assert fn(ctypes.byref(oa), ctypes.byref(ob), M, N, K, C2.data_ptr(), q4.F32, None, 0,
              torch.cuda.current_stream().cuda_stream) == 0
    assert torch.equal(C1, C2)
    assert lib.sync_status() == 0


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("shape", [(128, 256, 4096), (256, 2048, 2048), (1000, 2048, 1024),
                                   (1100, 2350, 768)])
def test_w4a4_bitwise_repeatable(lib, fmt, shape):
    """Split-K (few tiles) and persistent (many tiles) launches reduce in a fixed
    order: two runs give the same bits."""
    M, N, K = shape
    a, b = (_nv_pair if fmt == "nvfp4" else workloads.mxfp4_pair)(M, N, K, seed=M + N)
    f = lib.gemm_w4a4_nvfp4 if fmt == "nvfp4" else lib.gemm_w4a4_mxfp4
    ad, bd = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    C1 = f(ad, bd, K, out_dtype=torch.float32)
    C2 = f(ad, bd, K, out_dtype=torch.float32)
    assert torch.equal(C1, C2)
    assert lib.sync_status() == 0


@pytest.mark.parametrize("layout", ["rowmajor", "mma"])
def test_w4a4_mxfp4_prequantized(lib, layout):
    M, N, K = 200, 600, 1280
    a, b = workloads.mxfp4_pair(M, N, K, seed=11)
    ca, sa = lib.quantize_mxfp4(torch.from_numpy(a).cuda(), scale_layout=layout)
    cb, sb = lib.quantize_mxfp4(torch.from_numpy(b).cuda(), scale_layout=layout)
    C = lib.gemm_w4a4_mxfp4(q4.Fp4Operand(ca, sa, layout), q4.Fp4Operand(cb, sb, layout), K,
                            out_dtype=torch.float32)
    R = oracle.gemm_w4a4_mxfp4(*oracle.quantize_mxfp4(a), *oracle.quantize_mxfp4(b))
    assert_gemm_close(C.cpu().numpy(), R)


def test_tiny_workload_fp32(lib):
    """The tiny NVFP4 problem with the eight-weight worked row, fp32 output."""
    a, b = workloads.tiny()
    C = lib.gemm_w4a4_nvfp4(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), 512,
                            out_dtype=torch.float32)
    R = oracle.gemm_w4a4_nvfp4(*oracle.quantize_nvfp4(a), *oracle.quantize_nvfp4(b))
    fro, _ = assert_gemm_close(C.cpu().numpy(), R)
    assert fro < 1e-5  # fp32 output: only the accumulation order differs


def test_identity_operand(lib):
    """B = I (K = 256): C = c * A_hat with c = 6 * 448 * gB."""
    M, K = 96, 256
    a, _ = workloads.nvfp4_pair(M, 8, K, seed=5)
    eye = np.zeros((K, K), np.float32)
    np.fill_diagonal(eye, 1.0)
    C = lib.gemm_w4a4_nvfp4(torch.from_numpy(a).cuda(), torch.from_numpy(eye).cuda(), K,
                            out_dtype=torch.float32).cpu().numpy()
    qa, qb = oracle.quantize_nvfp4(a), oracle.quantize_nvfp4(eye)
    want = oracle.dequantize_nvfp4(*qa) * (6.0 * 448.0 * float(qb[2]))
    assert np.allclose(C, want, rtol=1e-6, atol=0)


# ragged N and M, odd group counts, one group, several blocks of 16 tokens, one
# row block with a long K, many row blocks with a short K
W4A16_SHAPES = [(1, 256, 1024), (4, 520, 2048), (16, 1000, 1152), (5, 128, 128),
                (17, 300, 8192), (33, 256, 512), (16, 2048, 8192), (8, 128, 8192),
                (3, 8192, 256), (2, 130, 384)]


@pytest.mark.parametrize("shape", W4A16_SHAPES)
def test_w4a16_int4(lib, shape):
    M, N, K = shape
    A, W = workloads.decode(M, seed=sum(shape), N=N, K=K)
    wq, ws = lib.quantize_int4_g128(torch.from_numpy(W).cuda())
    owq, ows = oracle.quantize_int4_g128(W)
    assert np.array_equal(wq.cpu().numpy(), owq) and np.array_equal(ws.cpu().numpy().view(np.uint16), ows)
    C = lib.gemm_w4a16_int4(A.cuda(), wq, ws)
    R = oracle.gemm_w4a16_int4(A.float().numpy(), owq, ows)
    assert_gemm_close(C.float().cpu().numpy(), R)
    assert lib.sync_status() == 0


W4A16_FP4_SHAPES = [(1, 256, 1024), (4, 520, 2048), (16, 1000, 1152), (5, 128, 128),
                    (17, 300, 8192), (33, 256, 512), (8, 128, 8192), (3, 8192, 256)]


def _fp4_weights(lib, w, fmt):
    """GPU-quantized FP4 weights (row-major scales), checked bit for bit
    against the oracle's, and the oracle's copy."""
    wt = torch.from_numpy(w).cuda()
    if fmt == "nvfp4":
        c, s, g = lib.quantize_nvfp4(wt)
        oq = oracle.quantize_nvfp4(w)
        assert np.array_equal(c.cpu().numpy(), oq[0]) and np.array_equal(s.cpu().numpy(), oq[1])
        assert g.cpu().numpy()[0] == oq[2]
        return (c, s, g), oq
    c, s = lib.quantize_mxfp4(wt)
    oq = oracle.quantize_mxfp4(w)
    assert np.array_equal(c.cpu().numpy(), oq[0]) and np.array_equal(s.cpu().numpy(), oq[1])
    return (c, s), oq


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("shape", W4A16_FP4_SHAPES)
def test_w4a16_fp4_weights(lib, shape, fmt):
    M, N, K = shape
    A, w = workloads.decode(M, seed=sum(shape) + 3, N=N, K=K)
    q, oq = _fp4_weights(lib, w, fmt)
    if fmt == "nvfp4":
        C = lib.gemm_w4a16_nvfp4(A.cuda(), *q)
        R = oracle.gemm_w4a16_nvfp4(A.float().numpy(), *oq)
    else:
        C = lib.gemm_w4a16_mxfp4(A.cuda(), *q)
        R = oracle.gemm_w4a16_mxfp4(A.float().numpy(), *oq)
    assert_gemm_close(C.float().cpu().numpy(), R)
    assert lib.sync_status() == 0


@pytest.mark.parametrize("c", [1.0, 3.0e-7, 3.0e5])
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_w4a16_fp4_identity_activations_give_the_weights(lib, fmt, c):
    """A = c I (and a tensor scale of 1): every output is one dequantized
    weight, e2m1 x block scale, times c -- at most 14 significant bits, so
    FP32 holds it and the only rounding is the store to bf16.  The output must
    equal the oracle's, bit for bit, for every code (the subnormal 0.5
    included) and scale met, with activations of ordinary size and ones far
    outside the f16 range (3e-7, 3e5)."""
    K, N = 256, 384
    w = workloads.normal(workloads.rng_for(31, 2), (N, K), 0.02)
    w[5, 3:40] *= 300.0  # large blocks next to small ones in the same rows
    w[9, 100:140] *= 1e-3
    q, oq = _fp4_weights(lib, w, fmt)
    cb = torch.tensor(c, dtype=torch.bfloat16)
    eye = torch.eye(K, dtype=torch.bfloat16, device="cuda") * cb.cuda()
    for m0 in range(0, K, 128):
        A = eye[m0:m0 + 128].contiguous()
        if fmt == "nvfp4":
            one = torch.ones(1, dtype=torch.float32, device="cuda")
            C = lib.gemm_w4a16_nvfp4(A, q[0], q[1], one)
            deq = oracle.dequantize_nvfp4(oq[0], oq[1], np.float32(1.0))[:, m0:m0 + 128].T
        else:
            C = lib.gemm_w4a16_mxfp4(A, *q)
            deq = oracle.dequantize_mxfp4(*oq)[:, m0:m0 + 128].T
        exact = deq.astype(np.float64) * float(cb)
        assert np.array_equal(exact.astype(np.float32).astype(np.float64), exact)
        want = torch.from_numpy(exact.astype(np.float32)).to(torch.bfloat16)
        assert torch.equal(C.cpu(), want)
    assert lib.sync_status() == 0


@pytest.mark.parametrize("M", [4, 16])
def test_w4a16_nvfp4_activations_outside_f16_range(lib, M):
    """Activations that f16 could not hold (above 65504, or below 2^-17 in
    magnitude where f16 would round them) next to ordinary ones, in groups of
    both CTAs of the K split: the products stay exact (bf16 x bf16 in the
    MMA) and the output agrees with the oracle."""
    N, K = 512, 2048  # 16 groups, 8 per CTA
    A, w = workloads.decode(M, seed=77 + M, N=N, K=K)
    a = A.float()
    a[0, 130] = 3.0e5      # group 1: above 65504
    a[M - 1, 700] = -7.0e4  # group 5
    a[1, 1500] = 3.0e-7    # group 11 (the second CTA's fourth): f16 would round it
    a[2, 1900] = 2.0 ** -20  # group 14: an f16 subnormal power of two, exact
    A = a.to(torch.bfloat16)
    q, oq = _fp4_weights(lib, w, "nvfp4")
    C = lib.gemm_w4a16_nvfp4(A.cuda(), *q)
    R = oracle.gemm_w4a16_nvfp4(A.float().numpy(), *oq)
    assert_gemm_close(C.float().cpu().numpy(), R)
    assert lib.sync_status() == 0


def test_w4a16_right_after_quantizing_its_weights(lib):
    """Weights quantized into poisoned buffers and read by the very next launch
    on the same stream, with no host synchronization in between: the GEMM
    starts early (programmatic dependent launch) but must see the new codes."""
    N, K, M = 1024, 2048, 4
    A = torch.randn(M, K, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16).cuda()
    w = (torch.randn(N, K, generator=torch.Generator().manual_seed(5)) * 0.02).cuda()
    wq0, ws0 = lib.quantize_int4_g128(w)
    want = lib.gemm_w4a16_int4(A, wq0, ws0)
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(8):
        wq = torch.full((N, K // 2), 0x77, dtype=torch.uint8, device="cuda")
        ws = torch.full((N, K // 128), 0x7BFF, dtype=torch.int16, device="cuda")
        C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        torch.cuda.synchronize()
        assert lib.lib().quantize_int4_g128(w.data_ptr(), q4.F32, N, K, wq.data_ptr(),
                                            ws.data_ptr(), stream) == 0
        assert lib.lib().gemm_w4a16_int4(A.data_ptr(), wq.data_ptr(), ws.data_ptr(), M, N, K,
                                         C.data_ptr(), None, 0, stream) == 0
        torch.cuda.synchronize()
        assert torch.equal(C, want)
    assert lib.sync_status() == 0


def test_w4a16_scales_off_16_byte_boundary(lib):
    """Ws only needs 2-byte alignment: scales that start 2 bytes past a 16-byte
    boundary give the same result as an aligned copy."""
    M, N, K = 4, 512, 1024  # 8 groups per row: the aligned path would take 16-byte loads
    A, W = workloads.decode(M, seed=21, N=N, K=K)
    A = A.cuda()
    wq, ws = lib.quantize_int4_g128(torch.from_numpy(W).cuda())
    want = lib.gemm_w4a16_int4(A, wq, ws)
    shifted = torch.zeros(N * K // 128 + 8, dtype=torch.int16, device="cuda")
    shifted[1:1 + N * K // 128].copy_(ws.view(torch.int16).reshape(-1))
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.lib().gemm_w4a16_int4(A.data_ptr(), wq.data_ptr(), shifted.data_ptr() + 2, M, N, K,
                                     C.data_ptr(), None, 0, stream) == 0
    torch.cuda.synchronize()
    assert torch.equal(C, want)
    assert lib.sync_status() == 0


def test_w4a16_chain_of_launches(lib):
    """Each launch reads the previous launch's output as its activations, with
    no host synchronization: the next kernel starts early and prefetches its
    weights, but reads its activations only after its predecessor is done."""
    N = K = 2048
    Ws = []
    for i in range(6):
        _, W = workloads.decode(1, seed=40 + i, N=N, K=K)
        Ws.append(lib.quantize_int4_g128(torch.from_numpy(W).cuda()))
    for M in (1, 4, 16):
        a0 = (torch.randn(M, K, generator=torch.Generator().manual_seed(M)) * 0.05).to(torch.bfloat16).cuda()
        want, x = [], a0
        for wq, ws in Ws:  # one launch at a time
            x = lib.gemm_w4a16_int4(x, wq, ws)
            torch.cuda.synchronize()
            want.append(x)
        outs = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in Ws]
        stream = torch.cuda.current_stream().cuda_stream
        torch.cuda.synchronize()
        x = a0
        for (wq, ws), out in zip(Ws, outs):
            assert lib.lib().gemm_w4a16_int4(x.data_ptr(), wq.data_ptr(), ws.data_ptr(), M, N, K,
                                             out.data_ptr(), None, 0, stream) == 0
            x = out
        torch.cuda.synchronize()
        for got, w in zip(outs, want):
            assert torch.equal(got, w)
    assert lib.sync_status() == 0


def test_w4a16_repeatable(lib):
    A, W = workloads.decode(16, seed=9, N=1024, K=4096)
    wq, ws = lib.quantize_int4_g128(torch.from_numpy(W).cuda())
    c1 = lib.gemm_w4a16_int4(A.cuda(), wq, ws)
    c2 = lib.gemm_w4a16_int4(A.cuda(), wq, ws)
    assert torch.equal(c1, c2)  # deterministic split-K reduction


def _grouped_case(T, E, N, K, top, seed):
    tok = workloads.to_bf16(workloads.normal(workloads.rng_for(seed, 1), (T, K), 1.0))
    offs, rt = workloads.route_top_k(T, E, top, seed)
    ws = [workloads.expert_weight(seed, e, N, K) for e in range(E)]
    return tok, offs, rt, ws


@pytest.mark.parametrize("layout", ["mma", "rowmajor"])
@pytest.mark.parametrize("case", [(64, 5, 512, 512, 2), (300, 8, 320, 768, 4), (40, 3, 256, 256, 1)])
def test_grouped_moe(lib, case, layout):
    """Both weight-scale layouts (row-major ones are re-laid out by the call;
    N = 320 is not a whole number of 128-row blocks)."""
    T, E, N, K, top = case
    tok, offs, rt, ws = _grouped_case(T, E, N, K, top, seed=T + E)
    wc, wsf, wg = [], [], []
    for w in ws:
        c, s, g = lib.quantize_nvfp4(torch.from_numpy(w).cuda(), scale_layout=layout)
        wc.append(c), wsf.append(s.reshape(-1)), wg.append(g)
    C = lib.grouped_gemm_moe(tok.cuda(), torch.from_numpy(offs).cuda(), torch.from_numpy(rt).cuda(),
                             torch.stack(wc), torch.cat(wsf), torch.cat(wg), N, w_scale_layout=layout)
    R = oracle.grouped_gemm_moe(tok.float().numpy(), offs, rt, [oracle.quantize_nvfp4(w) for w in ws])
    assert_gemm_close(C.float().cpu().numpy(), R)
    assert lib.sync_status() == 0


def test_read_probe_reads_every_word_once(lib):
    """The bandwidth probe folds what it reads into its sink with XOR: the XOR
    of the sink words equals the XOR of every 32-bit word of the source, so
    each word was read exactly once (sizes off the grid's stride included)."""
    for n in (16, 4096 + 16, 34_603_008, 8_830_000 // 16 * 16):
        src = torch.randint(-2**31, 2**31 - 1, (n // 4,), dtype=torch.int32, device="cuda")
        sink = lib.read_probe(src)
        want = np.bitwise_xor.reduce(src.cpu().numpy().view(np.uint32))
        got = np.bitwise_xor.reduce(sink.cpu().numpy().view(np.uint32))
        assert got == want

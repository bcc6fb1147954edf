"""Parity at the workloads' full sizes, in the configuration the benchmark
times.  Codes and scales are compared bit for bit over whole tensors; GEMM
outputs in full where the FP64 oracle can afford it, else on sampled rows
(every column of a sampled row, so the row-norm criterion is exact)."""
import numpy as np
import pytest
import torch

import int4_gemm_gb300 as q4
import oracle
import workloads
from tests._util import assert_gemm_close

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def test_decode_full(lib):
    N = K = 8192
    seed = workloads.SEED_BASE + 2
    w = workloads.int4_weights(N, K, seed)
    wq, ws = lib.quantize_int4_g128(torch.from_numpy(w).cuda())
    owq, ows = oracle.quantize_int4_g128(w)
    assert np.array_equal(wq.cpu().numpy(), owq)
    assert np.array_equal(ws.cpu().numpy().view(np.uint16), ows)
    for M in (1, 4, 16):
        A = workloads.to_bf16(workloads.normal(workloads.rng_for(seed, 1), (M, K), 1.0))
        C = lib.gemm_w4a16_int4(A.cuda(), wq, ws)
        R = oracle.gemm_w4a16_int4(A.float().numpy(), owq, ows)
        assert_gemm_close(C.float().cpu().numpy(), R)
    assert lib.sync_status() == 0


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_decode_fp4_weights_full_sampled(lib, fmt):
    """Decode with FP4 weights at N = K = 8192, M = 1, 4, 16: codes and scales
    of 512 sampled weight rows bit for bit, and the outputs of those rows (all
    tokens) against the oracle."""
    N = K = 8192
    seed = workloads.SEED_BASE + 2
    w = workloads.int4_weights(N, K, seed)
    rows = np.sort(np.random.default_rng(7).choice(N, 512, replace=False))
    wt = torch.from_numpy(w).cuda()
    if fmt == "nvfp4":
        c, sc, g = lib.quantize_nvfp4(wt)
        oq = oracle.quantize_nvfp4(w, rows=rows)
        assert g.cpu().numpy()[0] == oq[2]
    else:
        c, sc = lib.quantize_mxfp4(wt)
        oq = oracle.quantize_mxfp4(w, rows=rows)
    assert np.array_equal(c.cpu().numpy()[rows], oq[0])
    assert np.array_equal(sc.cpu().numpy()[rows], oq[1])
    for M in (1, 4, 16):
        A = workloads.to_bf16(workloads.normal(workloads.rng_for(seed, 1), (M, K), 1.0))
        if fmt == "nvfp4":
            C = lib.gemm_w4a16_nvfp4(A.cuda(), c, sc, g)
            R = oracle.gemm_w4a16_nvfp4(A.float().numpy(), *oq)
        else:
            C = lib.gemm_w4a16_mxfp4(A.cuda(), c, sc)
            R = oracle.gemm_w4a16_mxfp4(A.float().numpy(), *oq)
        assert_gemm_close(C.float().cpu().numpy()[:, rows], R)
    assert lib.sync_status() == 0


def test_moe_mxfp4_full(lib):
    a, b = workloads.moe()
    ad, bd = a.cuda(), torch.from_numpy(b).cuda()
    bc, bs = lib.quantize_mxfp4(bd, scale_layout="mma")
    obc, obs = oracle.quantize_mxfp4(b)
    rbc, rbs = lib.quantize_mxfp4(bd)
    assert np.array_equal(rbc.cpu().numpy(), obc) and np.array_equal(rbs.cpu().numpy(), obs)
    C = lib.gemm_w4a4_mxfp4(ad, q4.Fp4Operand(bc, bs, "mma"), 7168, out_dtype=torch.bfloat16)
    R = oracle.gemm_w4a4_mxfp4(*oracle.quantize_mxfp4(a.float().numpy()), obc, obs)
    assert_gemm_close(C.float().cpu().numpy(), R)


def test_prefill_nvfp4_sampled_rows(lib):
    a, b = workloads.prefill()
    M, K = a.shape
    N = b.shape[0]
    ad = a.cuda()
    bd = torch.from_numpy(b).cuda()
    bc, bs, bg = lib.quantize_nvfp4(bd)
    del bd
    ob = oracle.quantize_nvfp4(b)
    assert bg.item() == float(ob[2])
    assert np.array_equal(bs.cpu().numpy(), ob[1])
    assert np.array_equal(bc.cpu().numpy(), ob[0])
    ac, as_, ag = lib.quantize_nvfp4(ad)
    af = a.float().numpy()
    oa = oracle.quantize_nvfp4(af)
    assert ag.item() == float(oa[2])
    assert np.array_equal(as_.cpu().numpy(), oa[1]) and np.array_equal(ac.cpu().numpy(), oa[0])
    del ac, as_
    # the benchmark's configuration: A raw (quantized on the fly), B pre-quantized
    bmma = lib.scales_to_mma(bs)
    C = lib.gemm_w4a4_nvfp4(ad, q4.Fp4Operand(bc, bmma, "mma", bg), K, out_dtype=torch.bfloat16)
    # one random row in every 128-row half of every 256-row M tile pair, and
    # the first and last rows
    rows = np.arange(0, M, 128) + np.random.default_rng(0).integers(0, 128, M // 128)
    rows = np.unique(np.concatenate([rows, [0, M - 1]]))
    b_hat = oracle.dequantize_nvfp4(*ob)
    a_hat = oracle.dequantize_nvfp4(oa[0][rows], oa[1][rows], oa[2])
    R = a_hat @ b_hat.T
    assert_gemm_close(C[torch.from_numpy(rows).cuda()].float().cpu().numpy(), R)
    assert lib.sync_status() == 0


def test_grouped_full_sampled_experts(lib):
    """Every non-empty expert of the grouped workload: its first and last
    routed rows and four random ones, on eight sampled columns of every
    128-column N tile; the largest expert in full."""
    seed = workloads.SEED_BASE + 5
    T, E, N, K = 4096, 64, 2048, 7168
    tok, _, offs, rt = workloads.grouped(seed, experts=False)
    R_rows = int(offs[-1])
    counts = np.diff(offs)
    assert counts[63] == 0 and counts.max() < 1300
    largest = int(np.argmax(counts))
    rng = np.random.default_rng(11)
    cols = np.sort(np.concatenate([t * 128 + rng.choice(128, 8, replace=False)
                                   for t in range(N // 128)]))
    wc = torch.empty((E, N, K // 2), dtype=torch.uint8, device="cuda")
    sfb = q4.mma_scales_bytes(N, K // 16)
    wsf = torch.empty(E * sfb, dtype=torch.uint8, device="cuda")
    wg = torch.empty(E, dtype=torch.float32, device="cuda")
    b_hat = {}
    for e in range(E):
        w = workloads.expert_weight(seed, e, N, K)
        c, s, g = lib.quantize_nvfp4(torch.from_numpy(w).cuda(), scale_layout="mma")
        wc[e].copy_(c), wsf[e * sfb:(e + 1) * sfb].copy_(s), wg[e:e + 1].copy_(g)
        if counts[e] == 0:
            continue
        oq = oracle.quantize_nvfp4(w, rows=None if e == largest else cols)
        assert g.item() == float(oq[2])
        b_hat[e] = oracle.dequantize_nvfp4(*oq)
    assert len(b_hat) == int(np.count_nonzero(counts)) == 63
    C = lib.grouped_gemm_moe(tok.cuda(), torch.from_numpy(offs).cuda(), torch.from_numpy(rt).cuda(),
                             wc, wsf, wg, N)
    assert C.shape == (R_rows, N)
    Cf = C.float().cpu().numpy()
    assert lib.sync_status() == 0
    qa = oracle.quantize_nvfp4(tok.float().numpy())
    a_hat = oracle.dequantize_nvfp4(*qa)
    for e, bh in b_hat.items():
        r0, r1 = int(offs[e]), int(offs[e + 1])
        if e == largest:
            sel, ecols = np.arange(r0, r1), np.arange(N)
        else:
            inner = rng.choice(np.arange(r0, r1), min(4, r1 - r0), replace=False)
            sel, ecols = np.unique(np.concatenate([[r0, r1 - 1], inner])), cols
        Re = a_hat[rt[sel]] @ bh.T
        assert_gemm_close(Cf[sel][:, ecols], Re)

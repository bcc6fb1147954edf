"""Pins for the oracle's FP64 products: brute-force summation on tiny, non-square
shapes (catches a transposed operand or a dropped scale), an identity operand
that reduces the GEMM to dequantization, equal blocks with exact codes, the
per-group form of the W4A16 sum, and the routed grouped product."""
import json
import os

import numpy as np

import oracle
from oracle import formats as F
from oracle.quantize import int4_values, unpack_nibbles
import workloads

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_values.json")))


def _loops(a_hat, b_hat):
    M, K = a_hat.shape
    N = b_hat.shape[0]
    out = np.zeros((M, N))
    for i in range(M):
        for j in range(N):
            acc = 0.0
            for k in range(K):
                acc += float(a_hat[i, k]) * float(b_hat[j, k])
            out[i, j] = acc
    return out


def _nvfp4_value(codes, scales, g, i, k):
    c = unpack_nibbles(codes)[i, k]
    return float(F.e2m1_decode(c)) * float(F.e4m3_decode(scales[i, k // 16])) * float(g)


def test_w4a4_nvfp4_brute_force_from_codes():
    a, b = workloads.nvfp4_pair(3, 5, 32, seed=21)
    qa, qb = oracle.quantize_nvfp4(a), oracle.quantize_nvfp4(b)
    C = oracle.gemm_w4a4_nvfp4(*qa, *qb)
    assert C.shape == (3, 5)
    for i in range(3):
        for j in range(5):
            ref = sum(_nvfp4_value(*qa, i, k) * _nvfp4_value(*qb, j, k) for k in range(32))
            assert abs(C[i, j] - ref) <= 1e-12 * max(1.0, abs(ref))


def test_w4a4_mxfp4_brute_force():
    a, b = workloads.mxfp4_pair(4, 3, 64, seed=22)
    qa, qb = oracle.quantize_mxfp4(a), oracle.quantize_mxfp4(b)
    C = oracle.gemm_w4a4_mxfp4(*qa, *qb)
    ref = _loops(oracle.dequantize_mxfp4(*qa), oracle.dequantize_mxfp4(*qb))
    assert np.allclose(C, ref, rtol=1e-13, atol=1e-13)
    # each operand value really is code * 2^(byte - 127)
    ca = unpack_nibbles(qa[0])
    assert oracle.dequantize_mxfp4(*qa)[2, 37] == F.e2m1_decode(ca[2, 37]) * 2.0 ** (int(qa[1][2, 1]) - 127)


def test_identity_operand_reduces_to_dequantization():
    """B = I (16 x 16): every row has one 1, so (1/6)/g rounds to the E4M3 value
    448 and 1 / (448 g) to the code 6: B_hat = c I with c = 6 * 448 * g, which
    is 1 up to float32 rounding of g = 1/2688, and C = c A_hat."""
    a, _ = workloads.nvfp4_pair(7, 16, 16, seed=23)
    eye = np.eye(16, dtype=np.float32)
    qa, qb = oracle.quantize_nvfp4(a), oracle.quantize_nvfp4(eye)
    c = 6.0 * 448.0 * float(qb[2])
    assert abs(c - 1.0) < 2.0 ** -23
    assert np.array_equal(oracle.dequantize_nvfp4(*qb), c * np.eye(16))
    C = oracle.gemm_w4a4_nvfp4(*qa, *qb)
    assert np.allclose(C, c * oracle.dequantize_nvfp4(*qa), rtol=1e-15, atol=0)


def test_equal_blocks_give_exact_products():
    K = 64
    a = np.full((2, K), 0.75, np.float32)
    b = np.full((3, K), -2.0, np.float32)
    qa, qb = oracle.quantize_nvfp4(a), oracle.quantize_nvfp4(b)
    assert np.all(unpack_nibbles(qa[0]) == 7) and np.all(unpack_nibbles(qb[0]) == 15)
    va = oracle.dequantize_nvfp4(*qa)[0, 0]
    vb = oracle.dequantize_nvfp4(*qb)[0, 0]
    assert abs(va - 0.75) / 0.75 < 2 ** -4 and abs(vb + 2.0) / 2.0 < 2 ** -4
    assert np.all(oracle.gemm_w4a4_nvfp4(*qa, *qb) == K * va * vb)


def test_w4a16_group_form_and_brute_force():
    """C[m, n] = sum_g s16[n, g] * sum_{k in g} a[m, k] q[n, k]."""
    M, N, K = 3, 4, 256
    a = workloads.to_bf16(workloads.normal(workloads.rng_for(24, 1), (M, K), 1.0)).float().numpy()
    w = workloads.int4_weights(N, K, 24)
    wq, ws = oracle.quantize_int4_g128(w)
    C = oracle.gemm_w4a16_int4(a, wq, ws)
    q = int4_values(wq).astype(np.float64)
    s = F.fp16_decode(ws)
    ref = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            for gi in range(K // 128):
                ks = slice(128 * gi, 128 * gi + 128)
                ref[m, n] += s[n, gi] * float(np.dot(a[m, ks].astype(np.float64), q[n, ks]))
    assert np.allclose(C, ref, rtol=1e-12, atol=1e-12)


def _mxfp4_value(codes, scales, i, k):
    c = unpack_nibbles(codes)[i, k]
    return float(F.e2m1_decode(c)) * float(F.e8m0_decode(scales[i, k // 32]))


def test_w4a16_fp4_weights_brute_force():
    """W4A16 with FP4 weights, element by element from the codes: bf16-valued
    activations times e2m1(code) * block scale (* tensor scale for NVFP4)."""
    M, N, K = 3, 5, 64
    a = workloads.to_bf16(workloads.normal(workloads.rng_for(26, 1), (M, K), 1.0)).float().numpy()
    w = workloads.normal(workloads.rng_for(26, 2), (N, K), 0.02)
    w[1, 7] = 1.5  # an outlier: other blocks of row 1 get small scales
    qn = oracle.quantize_nvfp4(w)
    qm = oracle.quantize_mxfp4(w)
    Cn = oracle.gemm_w4a16_nvfp4(a, *qn)
    Cm = oracle.gemm_w4a16_mxfp4(a, *qm)
    assert Cn.shape == (M, N) and Cm.shape == (M, N)
    for i in range(M):
        for j in range(N):
            rn = sum(float(a[i, k]) * _nvfp4_value(*qn, j, k) for k in range(K))
            rm = sum(float(a[i, k]) * _mxfp4_value(*qm, j, k) for k in range(K))
            assert abs(Cn[i, j] - rn) <= 1e-12 * max(1.0, abs(rn))
            assert abs(Cm[i, j] - rm) <= 1e-12 * max(1.0, abs(rm))


def test_w4a16_fp4_identity_activations_give_the_weights():
    """A = I: C^T is the dequantized weight matrix itself."""
    K = 64
    w = workloads.normal(workloads.rng_for(27, 2), (8, K), 0.02)
    qn, qm = oracle.quantize_nvfp4(w), oracle.quantize_mxfp4(w)
    eye = np.eye(K)
    assert np.array_equal(oracle.gemm_w4a16_nvfp4(eye, *qn).T, oracle.dequantize_nvfp4(*qn))
    assert np.array_equal(oracle.gemm_w4a16_mxfp4(eye, *qm).T, oracle.dequantize_mxfp4(*qm))


def test_grouped_moe_matches_per_row_brute_force():
    T, E, N, K, top = 12, 4, 8, 32, 2
    tok = workloads.to_bf16(workloads.normal(workloads.rng_for(25, 1), (T, K), 1.0)).float().numpy()
    offs, rt = workloads.route_top_k(T, E, top, seed=25)
    assert offs[-1] == T * top and offs[E] - offs[E - 1] == 0  # last expert forced empty
    experts = [oracle.quantize_nvfp4(workloads.expert_weight(25, e, N, K)) for e in range(E)]
    C = oracle.grouped_gemm_moe(tok, offs, rt, experts)
    assert C.shape == (T * top, N)
    qa = oracle.quantize_nvfp4(tok)  # the whole token tensor shares one tensor scale
    for e in range(E):
        for r in range(offs[e], offs[e + 1]):
            t = rt[r]
            for n in range(N):
                ref = sum(_nvfp4_value(*qa, t, k) * _nvfp4_value(*experts[e], n, k) for k in range(K))
                assert abs(C[r, n] - ref) <= 1e-12 * max(1.0, abs(ref))


def test_fp32_accumulation_does_not_stall_like_bf16():
    """A BF16 running sum of 1000 ones stops at 256; FP32 (and the FP64 oracle)
    reach 1000.  The GEMM reference and the kernels accumulate in >= FP32."""
    import torch
    p = GOLD["bf16_sum"]
    acc = torch.zeros((), dtype=torch.bfloat16)
    for _ in range(p["ones"]):
        acc = acc + torch.ones((), dtype=torch.bfloat16)
    assert float(acc) == p["bf16_total"]
    ones = np.ones((1, p["ones"] + 24), np.float32)[:, :1024]
    c = oracle.gemm_fp64(ones[:, :p["ones"]], ones[:, :p["ones"]])
    assert c[0, 0] == p["fp32_total"]

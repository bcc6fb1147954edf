"""Pins for the FP8 blockwise oracle: the pages' outlier example run through the
blockwise quantizer, a brute-force signed E4M3 cast, the per-block scale tied
to the block amax, block shapes, and the block-promoted GEMM against plain
loops over dequantized values (two weight block rows and three K blocks, so a
wrong block index fails), and the W4A8 product (INT4 weights converted
exactly to E4M3, FP16 group scales in the promotion) against plain loops."""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import formats as F

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_values.json")))

_ALL = F.e4m3_decode(np.arange(256))


def _brute_e4m3(y):
    """Nearest finite E4M3 byte of the same sign as y (magnitude clamped to
    448), ties to the even code, by scanning all 256 bytes."""
    y = np.float32(y)
    neg = bool(np.signbit(y))
    mag = min(abs(float(y)), 448.0)
    best, bd = None, None
    for c in range(256):
        v = _ALL[c]
        if np.isnan(v) or bool(c & 0x80) != neg:
            continue
        d = abs(abs(v) - mag)
        if bd is None or d < bd or (d == bd and c % 2 == 0):
            best, bd = c, d
    return best


def test_e4m3_signed_cast_brute_force():
    rng = np.random.default_rng(5)
    ys = list(rng.uniform(-500, 500, 300).astype(np.float32))
    ys += list((rng.standard_normal(300) * 0.01).astype(np.float32))
    pos = F.e4m3_decode(np.arange(0x7F))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)     # exact in float32
    ys += list(mids[::7]) + list(-mids[::11])
    ys += [np.float32(v) for v in (0.0, -0.0, 448.0, -448.0, 464.0, 1e-30, -1e-30, 2.0 ** -10, 3 * 2.0 ** -10)]
    got = oracle.e4m3_encode_signed(np.array(ys, dtype=np.float32))
    want = np.array([_brute_e4m3(y) for y in ys], dtype=np.uint8)
    assert np.array_equal(got, want)
    # the special values, by hand
    assert list(got[-9:]) == [0x00, 0x80, 0x7E, 0xFE, 0x7E, 0x00, 0x80, 0x00, 0x02]


def test_blockwise_outlier_example_from_pages():
    """One (1, 128) block holds the outlier 100 and the small values 0.0002 and
    0.0004; the next block's largest magnitude is 1.0.  The first block's
    scale is 100/448 = 0.223: 0.0002 is stored as 0 and 0.0004 as 0.000436
    (9%); in the second block both small values keep a 4.1% error."""
    g = GOLD["e4m3_outlier"]
    x = np.zeros((1, 256), dtype=np.float32)
    x[0, 3] = g["tensor_amax"]
    x[0, 10], x[0, 11] = g["tiny"], g["small"]
    x[0, 128 + 5] = g["block_amax"]
    x[0, 128 + 10], x[0, 128 + 11] = g["tiny"], g["small"]
    q, s = oracle.quantize_fp8_blockwise(x, (1, 128))
    assert s.shape == (1, 2)
    assert round(float(s[0, 0]), 3) == g["tensor_scale"]
    xh = oracle.dequantize_fp8_blockwise(q, s, (1, 128))
    assert xh[0, 10] == g["tiny_stored"]
    assert round(float(xh[0, 11]), 6) == g["small_stored"]
    assert round(abs(xh[0, 11] - g["small"]) / g["small"], 2) == g["small_error"]
    for k in (128 + 10, 128 + 11):
        assert round(float(abs(xh[0, k] - x[0, k]) / x[0, k]), 3) == g["block_error"]
    assert q[0, 3] == 0x7E and q[0, 128 + 5] == 0x7E      # each block's amax lands on 448


@pytest.mark.parametrize("block,shape", [((1, 128), (6, 384)), ((128, 128), (256, 256)), ((128, 128), (40, 128))])
def test_blockwise_codes_are_the_nearest_values_and_scales_follow_amax(block, shape):
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(shape) * np.exp2(rng.integers(-6, 6, shape))).astype(np.float32)
    x[0, :128] = 0.0                                          # an all-zero (1, 128) block
    q, s = oracle.quantize_fp8_blockwise(x, block)
    br = min(block[0], shape[0])
    assert s.shape == (shape[0] // br, shape[1] // 128) and s.dtype == np.float32
    for bi in range(s.shape[0]):
        for bk in range(s.shape[1]):
            blk = x[bi * br:(bi + 1) * br, bk * 128:(bk + 1) * 128]
            qb = q[bi * br:(bi + 1) * br, bk * 128:(bk + 1) * 128]
            sc = s[bi, bk]
            amax = float(np.max(np.abs(blk)))
            if amax == 0.0:
                assert abs(float(sc) * 448.0 / 1e-12 - 1.0) < 2.0 ** -22
                assert np.all(qb == 0)
                continue
            assert abs(float(sc) * 448.0 / amax - 1.0) < 2.0 ** -22
            i, k = np.unravel_index(np.argmax(np.abs(blk)), blk.shape)
            assert qb[i, k] & 0x7F == 0x7E
            for (i, k) in zip(rng.integers(0, blk.shape[0], 40), rng.integers(0, 128, 40)):
                y = np.float32(np.float32(blk[i, k]) / sc)
                assert qb[i, k] == _brute_e4m3(y)


def test_blockwise_scale_invariance_by_powers_of_two():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((4, 256)).astype(np.float32)
    q, s = oracle.quantize_fp8_blockwise(x, (1, 128))
    q2, s2 = oracle.quantize_fp8_blockwise(x * np.float32(8.0), (1, 128))
    assert np.array_equal(q, q2) and np.array_equal(s2, s * np.float32(8.0))


def test_blockwise_rejects_partial_blocks():
    with pytest.raises(ValueError):
        oracle.quantize_fp8_blockwise(np.zeros((200, 128), np.float32), (128, 128))
    with pytest.raises(ValueError):
        oracle.quantize_fp8_blockwise(np.zeros((2, 100), np.float32), (1, 128))


def _loops(qa, sa, qb, sb, br):
    M, K = qa.shape
    N = qb.shape[0]
    out = np.zeros((M, N))
    for i in range(M):
        for j in range(N):
            acc = 0.0
            for k in range(K):
                a = float(F.e4m3_decode(qa[i, k])) * float(sa[i, k // 128])
                b = float(F.e4m3_decode(qb[j, k])) * float(sb[j // br, k // 128])
                acc += a * b
            out[i, j] = acc
    return out


@pytest.mark.parametrize("M,N,K", [(3, 256, 384), (2, 5, 256)])
def test_gemm_fp8_blockwise_brute_force(M, N, K):
    rng = np.random.default_rng(M * N + K)
    a = (rng.standard_normal((M, K)) * np.exp2(rng.integers(-3, 3, (M, K)))).astype(np.float32)
    w = rng.standard_normal((N, K)).astype(np.float32)
    w[:, 128:256] *= np.float32(16.0)                         # K blocks with different scales
    if N > 128:
        w[128:] *= np.float32(0.25)                           # weight block rows with different scales
    qa, sa = oracle.quantize_fp8_blockwise(a, (1, 128))
    qb, sb = oracle.quantize_fp8_blockwise(w, (128, 128))
    C = oracle.gemm_fp8_blockwise(qa, sa, qb, sb)
    ref = _loops(qa, sa, qb, sb, min(128, N))
    assert C.shape == (M, N)
    assert np.allclose(C, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_gemm_fp8_blockwise_identity_gives_dequantized_activations():
    rng = np.random.default_rng(8)
    a = rng.standard_normal((4, 256)).astype(np.float32)
    qa, sa = oracle.quantize_fp8_blockwise(a, (1, 128))
    qb = np.zeros((128, 256), np.uint8)
    qb[np.arange(128), np.arange(128)] = 0x38                 # E4M3 1.0 on the first K block
    sb = np.ones((1, 2), np.float32)
    C = oracle.gemm_fp8_blockwise(qa, sa, qb, sb)
    assert np.array_equal(C, oracle.dequantize_fp8_blockwise(qa, sa, (1, 128))[:, :128])
    assert F.e4m3_decode(0x38) == 1.0


def test_int4_values_convert_exactly_to_e4m3():
    """W4A8's weight conversion: every INT4 value -8..7 is an E4M3 value, and
    the bytes are the ones the E4M3 bit fields give (sign, exponent - 7, three
    mantissa bits): 1 = 0x38, 2 = 0x40, 3 = 0x44, 7 = 0x4E, -8 = 0xD0."""
    q = np.arange(-8, 8)
    b = oracle.int4_to_e4m3(q)
    assert np.array_equal(F.e4m3_decode(b), q.astype(np.float64))
    by_value = dict(zip(q.tolist(), b.tolist()))
    assert by_value[0] == 0x00 and by_value[1] == 0x38 and by_value[2] == 0x40
    assert by_value[3] == 0x44 and by_value[7] == 0x4E and by_value[-8] == 0xD0


@pytest.mark.parametrize("M,N,K", [(3, 5, 256), (2, 130, 384)])
def test_gemm_w4a8_brute_force(M, N, K):
    """Plain loops over e4m3(qa) * sa and the INT4 integer times its FP16
    group scale (three K blocks: a wrong block index or a scale taken from the
    wrong row fails)."""
    rng = np.random.default_rng(M + N + K)
    a = (rng.standard_normal((M, K)) * np.exp2(rng.integers(-3, 3, (M, K)))).astype(np.float32)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    w[:, 128:256] *= np.float32(10.0)
    w[1] *= np.float32(0.01)
    qa, sa = oracle.quantize_fp8_blockwise(a, (1, 128))
    wc, ws = oracle.quantize_int4_g128(w)
    C = oracle.gemm_w4a8(qa, sa, wc, ws)
    q = oracle.quantize.int4_values(wc)
    s16 = F.fp16_decode(ws)
    ref = np.zeros((M, N))
    for i in range(M):
        for j in range(N):
            acc = 0.0
            for k in range(K):
                acc += (float(F.e4m3_decode(qa[i, k])) * float(sa[i, k // 128])) * (int(q[j, k]) * float(s16[j, k // 128]))
            ref[i, j] = acc
    assert np.allclose(C, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())

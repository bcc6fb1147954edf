"""Pins for the oracle's quantizers: the pages' worked numbers, closed forms,
brute force over every code on tiny blocks, and the readings' edge cases."""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import formats as F
from oracle.quantize import int4_values, unpack_nibbles
import workloads

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_values.json")))


def _row(values, K):
    r = np.zeros((1, K), np.float32)
    r[0, :len(values)] = values
    return r


# --------------------------------------------------------------------------- worked row

def test_worked_row_nvfp4():
    g = GOLD["worked_row"]
    x = _row(g["weights"], 16)
    codes, scales, ts = oracle.quantize_nvfp4(x)
    S = F.e4m3_decode(scales[0, 0]) * float(ts)
    assert round(S, g["printed_digits"]) == g["scale_fp4"]
    assert round(g["absmax"] / 6, 4) == g["scale_fp4"]
    xh = oracle.dequantize_nvfp4(codes, scales, ts)[0]
    i = g["weights"].index(g["fp4_probe"])
    assert round(xh[i], 2) == g["fp4_stored"]
    assert round(abs(g["fp4_probe"] - xh[i]), 2) == g["fp4_error"]
    # 0.44 and 0.59 are the neighbouring stored values 3*S and 4*S
    assert [round(3 * S, 2), round(4 * S, 2)] == g["fp4_neighbours"]
    # the absmax lands exactly on the largest code, 6 * S
    assert xh[g["weights"].index(g["absmax"])] == 6 * S


def test_worked_row_int4():
    g = GOLD["worked_row"]
    x = _row(g["weights"], 128)
    codes, scales = oracle.quantize_int4_g128(x)
    s = float(F.fp16_decode(scales[0, 0]))
    assert round(s, g["printed_digits"]) == g["scale_int4"]
    xh = oracle.dequantize_int4_g128(codes, scales)[0]
    assert xh[g["weights"].index(g["int4_rounds_to_zero"])] == 0.0
    # every other weight is within half a step
    assert np.all(np.abs(xh[:8] - np.array(g["weights"])) <= s / 2 + 1e-7)


def test_worked_row_int8_scale_arithmetic():
    g = GOLD["worked_row"]
    assert round(g["absmax"] / 127, 5) == g["scale_int8"]


def test_worked_row_mxfp4_power_of_two_scale():
    g = GOLD["worked_row"]
    codes, scales = oracle.quantize_mxfp4(_row(g["weights"], 32))
    S = F.e8m0_decode(scales[0, 0])
    assert S == 0.125  # 0.88 / 0.125 = 7.04 lies in [4, 8)
    assert 4 * S <= g["absmax"] < 8 * S


# --------------------------------------------------------------------------- pages' other examples

def test_mxfp4_vs_nvfp4_block_max_5():
    """MXFP4 against NVFP4 scales: block max 5.0.  MXFP4 scale 1, 5 -> 4 (20%);
    NVFP4 E4M3 scale 0.8125, 5/0.8125 = 6.15 -> 6, stored 4.875 (2.5%).  The
    NVFP4 example has no tensor scale, i.e. g = 1, which a tensor whose amax is
    448 * 6 gives."""
    p = GOLD["mxfp4_vs_nvfp4"]
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 448 * 6
    x[0, 16] = p["block_max"]
    x[0, 17:20] = [1.0, -2.5, 0.3]
    codes, scales, g = oracle.quantize_nvfp4(x)
    assert g == 1.0
    assert F.e4m3_decode(scales[0, 1]) == p["nv_scale"]
    assert round(p["block_max"] / p["nv_scale"], 2) == p["nv_ratio"]
    xh = oracle.dequantize_nvfp4(codes, scales, g)[0]
    assert F.e2m1_decode(unpack_nibbles(codes)[0, 16]) == p["nv_code_value"]
    assert xh[16] == p["nv_stored"]
    assert round(abs(xh[16] - 5.0) / 5.0, 3) == p["nv_error"]

    xm = np.zeros((1, 32), np.float32)
    xm[0, 0] = p["block_max"]
    mc, ms = oracle.quantize_mxfp4(xm)
    assert F.e8m0_decode(ms[0, 0]) == p["mx_scale"]
    xmh = oracle.dequantize_mxfp4(mc, ms)[0]
    assert xmh[0] == p["mx_stored"]
    assert round(abs(xmh[0] - 5.0) / 5.0, 2) == p["mx_error"]


def test_outlier_sets_int4_scale():
    p = GOLD["outlier_int4"]
    x = np.full((1, 128), p["others_magnitude"], np.float32)
    x[0, 1::2] *= -1
    x[0, 7] = p["outlier"]
    x[0, 9] = 0.113
    x[0, 11] = 0.115
    codes, scales = oracle.quantize_int4_g128(x)
    s = float(F.fp16_decode(scales[0, 0]))
    assert round(s, 3) == p["scale"]
    assert round(s / 2, 3) == p["zero_below"]
    q = int4_values(codes)[0]
    assert q[7] == 7
    assert np.all(q[[0, 1, 2, 3, 9]] == 0)
    assert q[11] == 1


def test_bits_per_weight_closed_forms():
    p = GOLD["bits_per_weight"]
    rows, K = 4, 1024
    x = workloads.normal(workloads.rng_for(5, 1), (rows, K), 1.0)
    n = rows * K
    c, s = oracle.quantize_int4_g128(x)
    assert (c.nbytes + s.nbytes) * 8 / n == p["int4_g128"]
    c, s = oracle.quantize_mxfp4(x)
    assert (c.nbytes + s.nbytes) * 8 / n == p["mxfp4"]
    c, s, g = oracle.quantize_nvfp4(x)
    assert (c.nbytes + s.nbytes) * 8 / n == p["nvfp4"]
    assert np.float32(g).nbytes * 8 == p["nvfp4_tensor_scale_bits"]
    assert round((p["nvfp4"] / p["int4_g128"] - 1) * 100) == p["nvfp4_over_int4_percent"]


# --------------------------------------------------------------------------- brute force

def _blocks(seed, rows, K, spread=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, K)).astype(np.float32)
    if spread:
        x *= np.exp2(rng.integers(-12, 12, size=(rows, 1))).astype(np.float32)
    return x


def test_nvfp4_brute_force_every_code():
    x = _blocks(11, 64, 64)
    x[3, :16] = 0.0
    codes, scales, g = oracle.quantize_nvfp4(x)
    # the block scale is the E4M3 value nearest (amax/6)/g, over all 127 values
    pos = F.e4m3_decode(np.arange(0x7F))
    amax = np.abs(x.reshape(64, 4, 16)).max(-1)
    t = (amax / np.float32(6)) / g
    d = np.abs(t[..., None].astype(np.float64) - pos)
    assert np.all(d[np.arange(64)[:, None], np.arange(4)[None, :], scales] == d.min(-1))
    # every element's code is, among all 16 codes, the one nearest x / S
    c = unpack_nibbles(codes).reshape(64, 4, 16)
    S = (np.maximum(F.e4m3_decode(scales).astype(np.float32), F.F32_1E_12) * g).astype(np.float32)
    y = np.clip(x.reshape(64, 4, 16) / S[..., None], -6, 6).astype(np.float64)
    allv = F.e2m1_decode(np.arange(16))
    dist = np.abs(y[..., None] - allv)
    chosen = np.take_along_axis(dist, c[..., None].astype(np.int64), -1)[..., 0]
    live = (scales != 0)[..., None] & np.ones_like(c, bool)
    assert np.all(chosen[live] == dist.min(-1)[live])
    # a zero block stores scale byte 0 and all-zero codes
    assert scales[3, 0] == 0 and np.all(c[3, 0] == 0)


def test_mxfp4_brute_force_scale_and_codes():
    x = _blocks(12, 64, 128)
    codes, scales = oracle.quantize_mxfp4(x)
    S = F.e8m0_decode(scales)
    amax = np.abs(x.reshape(64, 4, 32)).max(-1).astype(np.float64)
    assert np.all((4 * S <= amax) & (amax < 8 * S))  # block max lands in [4, 8) * S
    c = unpack_nibbles(codes).reshape(64, 4, 32)
    y = np.clip(x.reshape(64, 4, 32) / S[..., None], -6, 6)
    allv = F.e2m1_decode(np.arange(16))
    dist = np.abs(y[..., None] - allv)
    chosen = np.take_along_axis(dist, c[..., None].astype(np.int64), -1)[..., 0]
    assert np.all(chosen == dist.min(-1))


def test_mxfp4_exponent_just_below_power_of_two():
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = np.nextafter(np.float32(16.0), np.float32(0))
    _, s = oracle.quantize_mxfp4(x)
    assert F.e8m0_decode(s[0, 0]) == 2.0  # exact floor(log2) = 3, minus 2


def test_int4_brute_force_every_integer():
    x = _blocks(13, 32, 256)
    codes, scales = oracle.quantize_int4_g128(x)
    q = int4_values(codes).reshape(32, 2, 128).astype(np.float64)
    s = F.fp16_decode(scales)
    r = x.reshape(32, 2, 128) / s[..., None].astype(np.float32)
    cand = np.arange(-8, 8, dtype=np.float64)
    dist = np.abs(r[..., None].astype(np.float64) - cand)
    assert np.all(np.abs(r - q) == dist.min(-1))
    assert q.min() >= -7  # |x / s16| <= 7 (1 + 2^-11) < 7.5 never reaches -8
    assert np.all(np.abs(q).max(-1) == 7)


def test_int4_ties_round_half_even():
    s = np.float32(0.5)  # amax 3.5 -> s = 0.5 exactly, and x/s = 2.5, 1.5, 0.5
    x = np.zeros((1, 128), np.float32)
    x[0, :4] = [3.5, 1.25, 0.75, 0.25]
    codes, scales = oracle.quantize_int4_g128(x)
    assert F.fp16_decode(scales[0, 0]) == s
    assert int4_values(codes)[0, :4].tolist() == [7, 2, 2, 0]


# --------------------------------------------------------------------------- readings / edges

def test_sign_bit_is_x_below_zero():
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 6.0
    x[0, 1] = -1e-6  # rounds to 0 but keeps its sign
    x[0, 2] = -0.0
    c, _, _ = oracle.quantize_nvfp4(x)
    u = unpack_nibbles(c)[0]
    assert u[1] == 0x8 and u[2] == 0x0
    c, _ = oracle.quantize_mxfp4(x)
    u = unpack_nibbles(c)[0]
    assert u[1] == 0x8 and u[2] == 0x0


def test_nibble_order_low_first():
    x = np.zeros((1, 32), np.float32)
    x[0, 0], x[0, 1] = 1.0, 6.0  # MXFP4 scale 1: codes 2 (1.0) and 7 (6.0)
    c, s = oracle.quantize_mxfp4(x)
    assert F.e8m0_decode(s[0, 0]) == 1.0
    assert c[0, 0] == 0x72


def test_nvfp4_underflowing_block_scale_gives_zero_codes():
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 1000.0
    x[0, 16:20] = [1e-6, -2e-6, 3e-7, 0.0]  # (amax/6)/g far below 2^-10
    c, s, g = oracle.quantize_nvfp4(x)
    assert s[0, 1] == 0
    assert np.all(unpack_nibbles(c)[0, 16:] == 0)


def test_int4_zero_and_underflowing_scale():
    x = np.zeros((1, 256), np.float32)
    x[0, 128:130] = [1e-9, -1e-9]  # amax/7 underflows FP16 -> scale 0 -> q = 0
    c, s = oracle.quantize_int4_g128(x)
    assert s[0, 0] == 0 and s[0, 1] == 0
    assert np.all(int4_values(c) == 0)


def test_nvfp4_tensor_scale_and_row_subset():
    a, _ = workloads.tiny()
    g = oracle.nvfp4_tensor_scale(a)
    assert g == np.float32(np.abs(a).max()) / np.float32(2688.0)
    c_all, s_all, _ = oracle.quantize_nvfp4(a)
    c_sub, s_sub, g2 = oracle.quantize_nvfp4(a, rows=[3, 0, 15])
    assert g2 == g
    assert np.array_equal(c_sub, c_all[[3, 0, 15]]) and np.array_equal(s_sub, s_all[[3, 0, 15]])
    z = np.zeros((2, 16), np.float32)
    assert oracle.nvfp4_tensor_scale(z) == np.float32(np.float32(1e-12) / np.float32(2688))


def test_dequant_error_bounded_by_half_step():
    """Away from clamping, |x - x_hat| <= half the local E2M1 step times S."""
    x = _blocks(14, 16, 64, spread=False)
    c, s, g = oracle.quantize_nvfp4(x)
    xh = oracle.dequantize_nvfp4(c, s, g)
    S = np.repeat(F.e4m3_decode(s) * float(g), 16, axis=1)
    step = np.where(np.abs(xh) / S < 2, 0.5, np.where(np.abs(xh) / S < 4, 1.0, 2.0))
    assert np.all(np.abs(x - xh) <= step / 2 * S * (1 + 1e-6) + 6 * S * 2.0 ** -4)

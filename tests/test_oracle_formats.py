"""Pins for the oracle's number formats: printed limits, exhaustive enumeration,
library casts as independent cross-checks, and brute force on dense grids."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import formats as F

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_values.json")))


def test_e2m1_value_set_matches_pages():
    vals = GOLD["e2m1_values"]["nonnegative"]
    assert F.e2m1_decode(np.arange(8)).tolist() == vals
    assert F.e2m1_decode(np.arange(8, 16)).tolist() == [-v for v in vals]


def test_e2m1_bit_fields():
    # s | e1 e0 | m with exponent bias 1: subnormal 0.5*m at e=0, else 2^(e-1)*(1+m/2)
    for code in range(16):
        s, e, m = code >> 3, (code >> 1) & 3, code & 1
        v = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1 + 0.5 * m)
        assert F.e2m1_decode(code) == (-v if s else v)


def _grid_with_midpoints():
    vals = np.array(GOLD["e2m1_values"]["nonnegative"], dtype=np.float32)
    mids = (vals[:-1] + vals[1:]) / 2
    pts = [np.linspace(0, 6, 600001, dtype=np.float32), vals, mids]
    for m in mids:  # one float32 ulp either side of every midpoint
        pts.append(np.array([np.nextafter(m, np.float32(0)), np.nextafter(m, np.float32(7))], np.float32))
    return np.unique(np.concatenate(pts))


def test_e2m1_nearest_brute_force_and_ties_to_smaller():
    y = _grid_with_midpoints()
    idx = F.e2m1_nearest(y)
    vals = F.E2M1_MAGNITUDES
    dist = np.abs(y[:, None].astype(np.float64) - vals[None, :])
    best = dist.min(axis=1)
    assert np.all(dist[np.arange(y.size), idx] == best)
    tie = (dist == best[:, None]).sum(axis=1) > 1
    assert tie.sum() == 7  # exactly the seven midpoints
    # on a tie the smaller magnitude (the first table entry) wins
    first = np.argmax(dist == best[:, None], axis=1)
    assert np.all(idx[tie] == first[tie])
    # the seven midpoints, explicitly
    assert F.e2m1_nearest(np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])).tolist() == [0, 1, 2, 3, 4, 5, 6]


def test_e2m1_nearest_ties_to_even_is_ieee_half_even():
    """ties="even" agrees with rounding to one mantissa bit with numpy's round
    half to even, binade by binade (0.5 steps below 2, 1 in [2, 4), 2 in
    [4, 6]), on a dense grid that includes every midpoint; and it differs from
    the pages' rule exactly at the midpoints of an odd lower neighbour."""
    mags = np.concatenate([np.arange(0, 6.0001, 1 / 64), [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]])
    step = np.where(mags < 2, 0.5, np.where(mags < 4, 1.0, 2.0))
    want = np.minimum(np.round(mags / step) * step, 6.0)
    got = F.E2M1_MAGNITUDES[F.e2m1_nearest(mags, ties="even")]
    assert np.array_equal(got, want)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    assert list(F.e2m1_nearest(mids, ties="even")) == [0, 2, 2, 4, 4, 6, 6]
    assert list(F.e2m1_nearest(mids)) == [0, 1, 2, 3, 4, 5, 6]
    off = ~np.isin(mags, mids)
    assert np.array_equal(F.e2m1_nearest(mags[off], ties="even"), F.e2m1_nearest(mags[off]))


def test_quantizers_round_half_even_on_request():
    """MXFP4 with scale 1 (block max 6): the seven midpoints and their
    negatives quantize to the even codes with rounding="rne" and to the
    smaller ones by default; NVFP4 with S = 1 likewise."""
    import oracle
    from oracle.quantize import unpack_nibbles
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    row = np.array([6.0] + mids + [-m for m in mids] + [0.0] * 17, np.float32)[None, :]
    pages = unpack_nibbles(oracle.quantize_mxfp4(row)[0])[0, 1:15]
    rne = unpack_nibbles(oracle.quantize_mxfp4(row, rounding="rne")[0])[0, 1:15]
    assert list(pages) == [0, 1, 2, 3, 4, 5, 6] + [8, 9, 10, 11, 12, 13, 14]
    assert list(rne) == [0, 2, 2, 4, 4, 6, 6] + [8, 10, 10, 12, 12, 14, 14]
    nv = np.array([2688.0] + [0.0] * 15 + [6.0] + mids + [0.0] * 8, np.float32)[None, :]  # g = 1, S = 1
    c_p = unpack_nibbles(oracle.quantize_nvfp4(nv)[0])[0, 17:24]
    c_r = unpack_nibbles(oracle.quantize_nvfp4(nv, rounding="rne")[0])[0, 17:24]
    assert list(c_p) == [0, 1, 2, 3, 4, 5, 6] and list(c_r) == [0, 2, 2, 4, 4, 6, 6]


def test_e4m3_limits_from_pages():
    g = GOLD["e4m3_limits"]
    pos = F.e4m3_decode(np.arange(0x7F))
    assert pos.max() == g["max"]
    assert pos[pos > 0].min() == g["min_subnormal"]
    assert F.e4m3_decode(0x08) == g["min_normal"]  # exponent field 1, mantissa 0
    assert np.isnan(F.e4m3_decode(0x7F)) and np.isnan(F.e4m3_decode(0xFF))
    # 3 mantissa bits: the step just above 1 is 2^-3, unit roundoff 2^-4
    assert F.e4m3_decode(0x39) - F.e4m3_decode(0x38) == 2 * g["unit_roundoff"]


def test_e4m3_decode_matches_torch_for_all_bytes():
    b = torch.arange(256, dtype=torch.uint8)
    ref = b.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = F.e4m3_decode(np.arange(256))
    assert np.array_equal(np.isnan(ref), np.isnan(ours))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], ours[ok])


def test_e4m3_encode_matches_torch_rne():
    rng = np.random.default_rng(0)
    pos = F.e4m3_decode(np.arange(0x7F))
    mids = (pos[:-1] + pos[1:]) / 2
    pts = [rng.uniform(0, 448, 200000), np.exp2(rng.uniform(-14, 8.8, 200000)), pos, mids]
    x = np.concatenate(pts).astype(np.float32)
    x = np.concatenate([x, np.nextafter(mids.astype(np.float32), np.float32(0)),
                        np.nextafter(mids.astype(np.float32), np.float32(500))])
    x = x[(x >= 0) & (x <= 448)]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(F.e4m3_encode(x), ref)


def test_e4m3_encode_exhaustive_nearest():
    # every representable value and every midpoint: nearest, ties to even code
    pos = F.e4m3_decode(np.arange(0x7F))
    assert np.array_equal(F.e4m3_encode(pos), np.arange(0x7F, dtype=np.uint8))
    mids = (pos[:-1] + pos[1:]) / 2
    got = F.e4m3_encode(mids)
    lo = np.arange(0x7E)
    assert np.array_equal(got, np.where(lo % 2 == 0, lo, lo + 1))
    assert F.e4m3_encode(np.array([1000.0]))[0] == 0x7E  # saturates


def test_e4m3_outlier_example_from_pages():
    """One outlier sets the scale: amax 100 -> scale 100/448; 0.0002 -> 0,
    0.0004 -> 0.000436 (9%); per-block scale 1/448 -> 4.1% for both."""
    g = GOLD["e4m3_outlier"]
    s = np.float32(g["tensor_amax"]) / np.float32(448.0)
    assert round(float(s), 3) == g["tensor_scale"]

    def fake(x, scale):
        return F.e4m3_decode(F.e4m3_encode(np.float32(x) / np.float32(scale))) * np.float64(np.float32(scale))

    assert fake(g["tiny"], s) == g["tiny_stored"]
    st = fake(g["small"], s)
    assert round(float(st), 6) == g["small_stored"]
    assert round(abs(st - g["small"]) / g["small"], 2) == g["small_error"]
    sb = np.float32(g["block_amax"]) / np.float32(448.0)
    for v in (g["tiny"], g["small"]):
        err = abs(fake(v, sb) - v) / v
        assert round(float(err), 3) == g["block_error"]


def test_fp16_encode_matches_torch():
    rng = np.random.default_rng(1)
    x = np.concatenate([np.exp2(rng.uniform(-30, 17, 100000)), rng.uniform(0, 2, 1000)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(F.fp16_encode(x), ref)


def test_floor_log2_exact_including_just_below_powers_of_two():
    vals = []
    for e in range(-40, 127):
        p = np.float32(2.0 ** e)
        vals += [p, np.nextafter(p, np.float32(0)), np.nextafter(p, np.float32(np.inf))]
    vals = np.array(vals, dtype=np.float32)
    f = F.floor_log2(vals)
    # the definition of floor(log2 v): 2^f <= v < 2^(f+1), checked in float64
    assert np.all(np.exp2(f.astype(np.float64)) <= vals.astype(np.float64))
    assert np.all(vals.astype(np.float64) < np.exp2(f.astype(np.float64) + 1))
    assert F.floor_log2(np.array([15.999999], np.float32))[0] == 3


def test_e8m0_decode():
    assert F.e8m0_decode(127) == 1.0 and F.e8m0_decode(124) == 0.125 and F.e8m0_decode(130) == 8.0

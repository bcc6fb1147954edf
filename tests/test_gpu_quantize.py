"""GPU quantizers against the CPU oracle: codes, scales and tensor scales must
match bit for bit, on ragged shapes, all input dtypes, both scale layouts and
the edge cases of the method (ties, zero blocks, underflowing scales)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._util import spread, to_mma_layout

pytestmark = pytest.mark.gpu

DTYPES = [torch.float32, torch.bfloat16, torch.float16]


def _dev(x, dtype):
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(dtype)
    return t.cuda(), t.float().numpy()  # the oracle sees exactly the values the GPU sees


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", [(1, 16), (7, 48), (130, 272), (257, 1024), (64, 7168)])
def test_nvfp4_bit_exact(lib, dtype, shape):
    x = spread(shape[0] * 31 + shape[1], *shape, lo=-6, hi=6)
    xd, xh = _dev(x, dtype)
    codes, scales, g = lib.quantize_nvfp4(xd)
    oc, os_, og = oracle.quantize_nvfp4(xh)
    assert g.item() == float(og)
    assert np.array_equal(scales.cpu().numpy(), os_)
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert lib.sync_status() == 0


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", [(1, 32), (5, 96), (130, 288), (257, 2048)])
def test_mxfp4_bit_exact(lib, dtype, shape):
    # fp16 holds +-65504 at most: keep its inputs finite
    lo, hi = (-6, 6) if dtype == torch.float16 else (-20, 20)
    x = spread(shape[0] * 17 + shape[1], *shape, lo=lo, hi=hi)
    xd, xh = _dev(x, dtype)
    codes, scales = lib.quantize_mxfp4(xd)
    oc, os_ = oracle.quantize_mxfp4(xh)
    assert np.array_equal(scales.cpu().numpy(), os_)
    assert np.array_equal(codes.cpu().numpy(), oc)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", [(1, 128), (9, 384), (130, 1152), (300, 8192)])
def test_int4_g128_bit_exact(lib, dtype, shape):
    lo, hi = (-6, 6) if dtype == torch.float16 else (-10, 10)
    x = spread(shape[0] * 13 + shape[1], *shape, lo=lo, hi=hi)
    xd, xh = _dev(x, dtype)
    codes, scales = lib.quantize_int4_g128(xd)
    oc, os_ = oracle.quantize_int4_g128(xh)
    assert np.array_equal(scales.cpu().numpy().view(np.uint16), os_)
    assert np.array_equal(codes.cpu().numpy(), oc)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("shape", [(1, 256), (130, 512), (300, 768)])
def test_mma_scale_layout(lib, fmt, shape):
    x = spread(7, *shape)
    xd, xh = _dev(x, torch.float32)
    if fmt == "nvfp4":
        c1, s_mma, _ = lib.quantize_nvfp4(xd, scale_layout="mma")
        c2, s_row, _ = lib.quantize_nvfp4(xd)
    else:
        c1, s_mma = lib.quantize_mxfp4(xd, scale_layout="mma")
        c2, s_row = lib.quantize_mxfp4(xd)
    want = to_mma_layout(s_row.cpu().numpy())
    assert np.array_equal(s_mma.cpu().numpy(), want)
    assert torch.equal(c1, c2)
    assert np.array_equal(lib.scales_to_mma(s_row).cpu().numpy(), want)


def test_worked_row(lib):
    x = np.zeros((1, 128), np.float32)
    x[0, :8] = workloads.WORKED_ROW
    xd, xh = _dev(x, torch.float32)
    for got, want in ((lib.quantize_nvfp4(xd)[:2], oracle.quantize_nvfp4(xh)[:2]),
                      (lib.quantize_mxfp4(xd), oracle.quantize_mxfp4(xh))):
        assert all(np.array_equal(g.cpu().numpy(), w) for g, w in zip(got, want))
    c, s = lib.quantize_int4_g128(xd)
    oc, os_ = oracle.quantize_int4_g128(xh)
    assert np.array_equal(c.cpu().numpy(), oc) and np.array_equal(s.cpu().numpy().view(np.uint16), os_)


def test_exact_midpoints_tie_to_smaller(lib):
    """Every E2M1 midpoint, positive and negative, at scale exactly 1."""
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    x = np.zeros((2, 32), np.float32)
    x[0, :7], x[0, 8:15], x[0, 16] = mids, -mids, 6.0        # MXFP4: amax 6 -> scale 1
    x[1, 0] = 2688.0                                          # NVFP4: g = 1
    x[1, 16:23], x[1, 24:31] = mids, -mids
    x[1, 31] = 6.0                                            # block amax 6 -> E4M3 1 -> S = 1
    xd, xh = _dev(x, torch.float32)
    c, s = lib.quantize_mxfp4(xd)
    oc, os_ = oracle.quantize_mxfp4(xh)
    assert np.array_equal(c.cpu().numpy(), oc) and np.array_equal(s.cpu().numpy(), os_)
    c, s, g = lib.quantize_nvfp4(xd)
    oc, os_, og = oracle.quantize_nvfp4(xh)
    assert g.item() == 1.0 == float(og)
    assert np.array_equal(c.cpu().numpy(), oc) and np.array_equal(s.cpu().numpy(), os_)


def test_int4_half_integer_ties(lib):
    x = np.zeros((1, 128), np.float32)
    x[0, :6] = [3.5, 1.25, 0.75, 0.25, -0.25, -1.25]  # s = 0.5: x/s = 7, 2.5, 1.5, 0.5, ...
    xd, xh = _dev(x, torch.float32)
    c, s = lib.quantize_int4_g128(xd)
    oc, os_ = oracle.quantize_int4_g128(xh)
    assert np.array_equal(c.cpu().numpy(), oc) and np.array_equal(s.cpu().numpy().view(np.uint16), os_)


def test_zero_and_underflowing_blocks(lib):
    x = np.zeros((3, 256), np.float32)
    x[1, 0] = 1000.0
    x[1, 16:20] = [1e-6, -2e-6, 3e-7, -0.0]   # NVFP4 block scale rounds to 0
    x[2, 128:130] = [1e-9, -1e-9]            # INT4 scale underflows FP16
    x[2, 0] = -1e-30
    xd, xh = _dev(x, torch.float32)
    for got, want in ((lib.quantize_nvfp4(xd), oracle.quantize_nvfp4(xh)),
                      (lib.quantize_mxfp4(xd), oracle.quantize_mxfp4(xh))):
        assert np.array_equal(got[0].cpu().numpy(), want[0])
        assert np.array_equal(got[1].cpu().numpy(), want[1])
    c, s = lib.quantize_int4_g128(xd)
    oc, os_ = oracle.quantize_int4_g128(xh)
    assert np.array_equal(c.cpu().numpy(), oc) and np.array_equal(s.cpu().numpy().view(np.uint16), os_)
    z = torch.zeros((4, 64), device="cuda")
    c, s, g = lib.quantize_nvfp4(z)
    assert g.item() == float(np.float32(np.float32(1e-12) / np.float32(2688)))
    assert int(c.sum()) == 0 and int(s.sum()) == 0


def test_nonfinite_input_is_reported(lib):
    x = torch.ones((4, 64), device="cuda")
    x[2, 5] = float("nan")
    lib.quantize_nvfp4(x)
    assert lib.sync_status() == -5
    assert lib.sync_status() == 0  # cleared by the read


def test_empty_rows(lib):
    x = torch.empty((0, 64), device="cuda")
    c, s, g = lib.quantize_nvfp4(x)
    assert c.numel() == 0
    c, s = lib.quantize_mxfp4(x)
    c, s = lib.quantize_int4_g128(torch.empty((0, 128), device="cuda"))
    assert lib.sync_status() == 0


def _neighbours(c, n=2):
    """float32 values c-n ulp .. c+n ulp around the float32 nearest to c."""
    f = np.float32(c)
    out = [f]
    lo = hi = f
    for _ in range(n):
        lo = np.nextafter(lo, np.float32(0))
        hi = np.nextafter(hi, np.float32(np.inf))
        out += [lo, hi]
    return out


@pytest.mark.parametrize("rounding", ["pages", "rne"])
def test_nvfp4_decisions_next_to_midpoints(lib, rounding):
    """Values within two ulps of m_k * S, the real numbers whose float32
    quotients by S sit on the E2M1 midpoints, for block scales that are not
    powers of two.  The tensor scale is 1 (tensor amax 2688), so S is the E4M3
    block scale itself.  Both tie rules."""
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    s0s = [1.125, 1.375, 2.75, 0.8125, 13.0, 208.0, 0.0390625, 0.001953125 * 5]
    rows = [[2688.0] + [0.0] * 15]
    for s0 in s0s:
        for t in mids:
            ulp_half = 2.0 ** (np.floor(np.log2(t)) - 24)
            c = (t + ulp_half) * s0            # exact in float64
            near = _neighbours(c) + _neighbours(t * s0)
            vals = [6.0 * s0] + [float(v) for v in near[:7]] + [-float(v) for v in near[:7]]
            rows.append(vals + [0.0] * (16 - len(vals)))
    x = np.array(rows, np.float32).reshape(1, -1)
    xd, xh = _dev(x, torch.float32)
    c, s, g = lib.quantize_nvfp4(xd, rounding=rounding)
    oc, os_, og = oracle.quantize_nvfp4(xh, rounding=rounding)
    assert g.item() == 1.0 == float(og)
    assert np.array_equal(s.cpu().numpy(), os_)
    assert np.array_equal(c.cpu().numpy(), oc)


def test_nvfp4_block_scales_next_to_e4m3_midpoints(lib):
    """Blocks whose t = (amax / 6) / g lies within a few ulp of an E4M3
    rounding boundary -- every midpoint between consecutive E4M3 values,
    subnormal ones included -- with g = 1 (tensor amax 2688): scale bytes and
    codes match the oracle bit for bit.  (t cannot pass 448: a block's amax is
    at most the tensor's, 2688 g.)"""
    from oracle import formats as F
    vals = np.unique(F.e4m3_decode(np.arange(0, 127)))
    mids = (vals[1:] + vals[:-1]) / 2
    rows = [[2688.0] + [0.0] * 15]
    for m in mids:
        for a in _neighbours(6.0 * m, 4):
            rows.append([float(a), -0.5 * float(a)] + [0.0] * 14)
    x = np.array(rows, np.float32).reshape(1, -1)
    xd, xh = _dev(x, torch.float32)
    c, s, g = lib.quantize_nvfp4(xd)
    oc, os_, og = oracle.quantize_nvfp4(xh)
    assert g.item() == 1.0 == float(og)
    assert np.array_equal(s.cpu().numpy(), os_)
    assert np.array_equal(c.cpu().numpy(), oc)


@pytest.mark.parametrize("rounding", ["pages", "rne"])
def test_mxfp4_decisions_next_to_midpoints(lib, rounding):
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    rows = []
    for e in (-40, -7, 0, 3, 60, 120):
        for t in mids:
            near = _neighbours(t * 2.0 ** e, 3)
            vals = [6.0 * 2.0 ** e] + [float(v) for v in near] + [-float(v) for v in near]
            rows.append(vals + [0.0] * (32 - len(vals)))
    x = np.array(rows, np.float32).reshape(1, -1)
    xd, xh = _dev(x, torch.float32)
    c, s = lib.quantize_mxfp4(xd, rounding=rounding)
    oc, os_ = oracle.quantize_mxfp4(xh, rounding=rounding)
    assert np.array_equal(s.cpu().numpy(), os_)
    assert np.array_equal(c.cpu().numpy(), oc)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_round_half_even_matches_oracle_on_random_data(lib, fmt, dtype):
    """rounding="rne" on ordinary data with injected midpoint values (exact
    ties under MXFP4's power-of-two scales; NVFP4 ties are covered by the
    midpoint test) and ragged rows, both scale layouts: bit-exact against the
    oracle."""
    rows, K = 300, 1024
    x = workloads.normal(workloads.rng_for(41, 1), (rows, K), 1.0)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    r = np.random.default_rng(42)
    pick = r.random((rows, K)) < 0.2
    x[pick] = (mids[r.integers(0, 7, pick.sum())] * np.float32(2.0) ** r.integers(-3, 3, pick.sum())
               * np.where(r.random(pick.sum()) < 0.5, -1, 1)).astype(np.float32)
    xd, xh = _dev(x, dtype)
    for layout in ("rowmajor", "mma"):
        if fmt == "nvfp4":
            c, s, _ = lib.quantize_nvfp4(xd, scale_layout=layout, rounding="rne")
            oc, os_, _ = oracle.quantize_nvfp4(xh, rounding="rne")
            op = oracle.quantize_nvfp4(xh)[0]
        else:
            c, s = lib.quantize_mxfp4(xd, scale_layout=layout, rounding="rne")
            oc, os_ = oracle.quantize_mxfp4(xh, rounding="rne")
            op = oracle.quantize_mxfp4(xh)[0]
        assert np.array_equal(c.cpu().numpy(), oc)
        if layout == "rowmajor":
            assert np.array_equal(s.cpu().numpy(), os_)
    if fmt == "mxfp4":  # power-of-two scales: the injected midpoints are exact ties
        assert not np.array_equal(oc, op)
    assert lib.sync_status() == 0

"""Exactness facts the W4A16 decode kernel's weight forms rest on, checked
exhaustively on the host (no GPU, no library): every product the MMAs form
must be exact, so that the only rounding is the FP32 accumulation and the
final bf16 store."""
import numpy as np
import torch

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])  # magnitudes of codes 0..7


def e4m3_values():
    """Every finite E4M3 value, from torch's own decoder."""
    b = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    v = b.float().numpy().astype(np.float64)
    return v[np.isfinite(v)]


def bf16_values():
    """Every bf16 value (all 65536 bit patterns) as float64."""
    b = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    with np.errstate(invalid="ignore"):  # the NaN patterns
        return b.float().numpy().astype(np.float64)


def bf16_bits_value(bits: int) -> float:
    """The value of a 16-bit bf16 pattern."""
    return float(np.array([bits << 16], dtype=np.uint32).view(np.float32)[0])


def significant_bits(v: float) -> int:
    m = int(np.ldexp(np.frexp(abs(v))[0], 53))
    return m.bit_length() - (m & -m).bit_length() + 1


def exact_in(dtype, v):
    return np.array_equal(v.astype(dtype).astype(np.float64), v)


def test_int4_nibble_becomes_136_plus_q():
    """(n ^ 8) | 0x4300, n the two's-complement nibble of q, is the bf16 bit
    pattern of 136 + q for every q in -8..7 (exponent of 128, mantissa 8 + q)."""
    for q in range(-8, 8):
        bits = ((q & 0xF) ^ 8) | 0x4300
        assert bf16_bits_value(bits) == 136 + q


def test_e2m1_bits_at_6_to_8_are_code_times_2_pow_minus_126():
    """Magnitude bits of an E2M1 code placed at bf16 bits 6..8 (sign at 15)
    give code * 2^-126 exactly, the subnormal 0.5 included."""
    for c in range(16):
        bits = ((c & 7) << 6) | ((c >> 3) << 15)
        want = (-1.0 if c >> 3 else 1.0) * E2M1[c & 7] * 2.0 ** -126
        v = bf16_bits_value(bits)
        assert v == want and np.signbit(v) == bool(c >> 3)


def test_nvfp4_weight_values_fit_bf16_and_f16():
    """code * E4M3 scale * 2^-10, the weight value both NVFP4 forms build, is
    exact in bf16 and in f16 (subnormals included) for every code and every
    finite scale; code * scale alone exceeds neither format's range."""
    s = e4m3_values()
    w = (E2M1[None, :] * s[:, None]).ravel() * 2.0 ** -10
    w = np.concatenate([w, -w])
    assert exact_in(np.float16, w)
    wt = torch.from_numpy(w)
    assert torch.equal(wt.to(torch.bfloat16).double(), wt)
    assert np.abs(w).max() == 6 * 448 * 2.0 ** -10  # 2.625
    nz = np.abs(w[w != 0])
    assert nz.min() == 0.5 * 2.0 ** -9 * 2.0 ** -10  # 2^-20 >= the f16 subnormal step 2^-24


def test_e4m3_scale_times_2_pow_116_is_a_normal_bf16():
    """The bf16 form stores the E4M3 scale times 2^116: normal and exact in
    bf16 for every nonzero finite scale, so one bf16 multiply of the
    code * 2^-126 pattern gives code * scale * 2^-10 without rounding."""
    s = e4m3_values()
    s = s[s != 0] * 2.0 ** 116
    st = torch.from_numpy(s)
    assert torch.equal(st.to(torch.bfloat16).double(), st)
    assert np.abs(s).min() >= 2.0 ** -126  # normal


def test_bf16_activations_exact_in_f16_window():
    """The f16 form needs the activations of a group to be f16 values.  Every
    bf16 value with 2^-17 <= |a| <= 65504 is one, as are zero and the
    infinities; every larger finite bf16 value is not (f16 overflows), and the
    kernel's test (round trip through f16) tells them apart exactly."""
    a = bf16_values()
    fin = np.isfinite(a)
    with np.errstate(over="ignore"):
        rt = a.astype(np.float16).astype(np.float64)
    exact = (rt == a) | np.isnan(a)
    window = fin & (np.abs(a) >= 2.0 ** -17) & (np.abs(a) <= 65504)
    assert exact[window].all()
    assert exact[a == 0].all() and exact[np.isinf(a)].all()
    assert not exact[fin & (np.abs(a) > 65504)].any()
    # below the window some values are f16 values (powers of two down to
    # 2^-24) and some are not (f16 would round them): the round trip decides
    small = fin & (a != 0) & (np.abs(a) < 2.0 ** -17)
    assert exact[small].any() and not exact[small].all()
    assert exact[a == 2.0 ** -20].all()


def test_products_fit_fp32():
    """A bf16 activation (8 significant bits) times any weight value of the
    forms above (at most 6 significant bits) has at most 14 significant bits:
    FP32 holds every product the MMA forms."""
    s = e4m3_values()
    w = np.unique(np.abs((E2M1[None, :] * s[:, None]).ravel() * 2.0 ** -10))
    w = w[w != 0]
    assert max(significant_bits(v) for v in w) == 6
    a = bf16_values()
    a = a[np.isfinite(a) & (a != 0)]
    assert max(significant_bits(v) for v in a[::97]) == 8

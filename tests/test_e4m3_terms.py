"""Host-side checks of the FP8 arithmetic the group-128 decode kernels rely on.

E4M3 here is the 8-bit float with a sign bit, 4 exponent bits (bias 7) and 3
mantissa bits, no infinities, 0x7F/0xFF NaN, largest finite 448; it is modelled
from those bit fields alone (decode) and by nearest-value search with ties to an
even mantissa (encode, saturating at 448), so the checks below do not depend on
any GPU conversion.  What is checked:
  * the byte of a nibble u in 0..15, read as E4M3, is exactly u * 2^-9 (so the
    kernels' weight codes are exact and a mask is the whole decode);
  * an activation v, scaled per 128-group so that the group's largest |v| lies
    in [128, 256), split into terms t_j = 2^-4j * E4M3(2^4j * r_j) with r_0 = v,
    r_(j+1) = r_j - t_j:
      - two terms give a bf16 value back exactly when it is at least 2^-13 of
        its group's largest, and within 2^-14 (absolute, scaled units) below;
      - four terms keep an fp32 value within 2^-16 relative plus 2^-22 absolute.
"""
import numpy as np
import pytest

rng = np.random.default_rng(20261202)


def e4m3_value(code: int) -> float:
    """Value of an E4M3 byte from its bit fields (NaN codes excluded)."""
    sign = -1.0 if code & 0x80 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0:
        return sign * man * 2.0 ** -9          # subnormal: man/8 * 2^(1-7)
    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)


POS_CODES = [c for c in range(0x7F)]          # 0x00 .. 0x7E: every non-negative finite code
POS_VALUES = np.array([e4m3_value(c) for c in POS_CODES])


def e4m3_round(x: np.ndarray) -> np.ndarray:
    """Round to the nearest finite E4M3 value, ties to the code with an even
    mantissa, saturating at +-448 (the SATFINITE conversion)."""
    a = np.minimum(np.abs(x), 448.0)
    hi = np.searchsorted(POS_VALUES, a, side="left")
    hi = np.minimum(hi, len(POS_VALUES) - 1)
    lo = np.maximum(hi - 1, 0)
    dlo, dhi = a - POS_VALUES[lo], POS_VALUES[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & ((np.array(POS_CODES)[hi] & 1) == 0))
    r = np.where(pick_hi, POS_VALUES[hi], POS_VALUES[lo])
    return np.sign(x) * r


def split_terms(v: np.ndarray, n_terms: int) -> np.ndarray:
    """Sum of the n_terms scaled E4M3 terms of v (already group-scaled)."""
    rem = v.copy()
    rep = np.zeros_like(v)
    for j in range(n_terms):
        lift = 2.0 ** (4 * j)
        t = e4m3_round(rem * lift) / lift
        rep += t
        rem -= t
    return rep


def group_scale(x: np.ndarray) -> float:
    """2^e with max|x| * 2^e in [128, 256)."""
    m = np.max(np.abs(x))
    return 2.0 ** (7 - np.floor(np.log2(m))) if m > 0 else 1.0


def to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest even) and back to float64."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_model_matches_the_format():
    # a few anchor values of the format, by hand
    assert e4m3_value(0x00) == 0.0
    assert e4m3_value(0x01) == 2.0 ** -9             # smallest subnormal
    assert e4m3_value(0x08) == 2.0 ** -6             # smallest normal
    assert e4m3_value(0x38) == 1.0
    assert e4m3_value(0x7E) == 448.0                 # largest finite
    assert e4m3_value(0xB8) == -1.0
    assert np.all(np.diff(POS_VALUES) > 0)
    assert e4m3_round(np.array([1.0625]))[0] == 1.0          # tie between 1 and 1.125 -> even mantissa
    assert e4m3_round(np.array([1.1875]))[0] == 1.25         # tie between 1.125 and 1.25 -> even
    assert e4m3_round(np.array([1000.0]))[0] == 448.0        # saturation


def test_nibble_byte_is_u_times_2_pow_minus_9():
    for u in range(16):
        assert e4m3_value(u) == u * 2.0 ** -9
    # packed word -> the two code words of the kernel (low nibbles, high nibbles)
    w = int(rng.integers(0, 2 ** 32))
    lo, hi = w & 0x0F0F0F0F, (w >> 4) & 0x0F0F0F0F
    for i in range(4):
        assert (lo >> (8 * i)) & 0xFF == (w >> (8 * i)) & 0xF          # element 2i
        assert (hi >> (8 * i)) & 0xFF == (w >> (8 * i + 4)) & 0xF      # element 2i + 1


@pytest.mark.parametrize("dist", ["normal", "wide"])
def test_two_terms_hold_bf16_exactly(dist):
    for _ in range(200):
        x = rng.standard_normal(128)
        if dist == "wide":
            x *= 2.0 ** rng.integers(-20, 20, size=128)   # exponents spread far beyond one group
        x = to_bf16(x)
        s = group_scale(x)
        v = x * s
        got = split_terms(v, 2)
        big = np.abs(x) >= 2.0 ** -13 * np.max(np.abs(x))
        np.testing.assert_array_equal(got[big], v[big])
        assert np.all(np.abs(got - v) <= 2.0 ** -14)


@pytest.mark.parametrize("dist", ["swiglu", "wide"])
def test_four_terms_keep_16_bits_of_fp32(dist):
    for _ in range(200):
        if dist == "swiglu":
            g, u = rng.standard_normal(128) * 1.3, rng.standard_normal(128) * 1.3
            h = g / (1.0 + np.exp(-g)) * u
        else:
            h = rng.standard_normal(128) * 2.0 ** rng.integers(-30, 30, size=128)
        h = h.astype(np.float32).astype(np.float64)
        s = group_scale(h)
        v = h * s
        got = split_terms(v, 4)
        assert np.all(np.abs(got - v) <= 2.0 ** -16 * np.abs(v) + 2.0 ** -22)
    # three unscaled terms (the rejected variant) are visibly worse on small elements
    v = np.array([200.0, 3.0e-3])
    rep = np.zeros(2)
    rem = v.copy()
    for _ in range(3):
        t = e4m3_round(rem)
        rep += t
        rem -= t
    assert abs(rep[1] - v[1]) > 2.0 ** -16 * abs(v[1]) + 2.0 ** -22

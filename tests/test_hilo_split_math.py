"""The arithmetic claim behind the hi/lo activation codes of the e4m3 decode block, on every
bf16 value (CPU, no GPU).  With s a power of two per token, each activation y = x / s is
written as hi = e4m3(y) and lo = e4m3(y - hi), both nearest-even (the remainder is exact in
binary32: y has 8 significant bits, hi the top 4).  Then hi + lo == y exactly for
2^-2 <= |y| < 256, and |hi + lo - y| <= 2^-10 below that; the kernel picks s so that a token's
largest |y| lies in [128, 256).  The e4m3 rounding is the oracle's encoder."""
import numpy as np

from oracle import tp_oracle as O


def all_bf16_values():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = O.bf16_bits_to_f64(bits)
    return v[np.isfinite(v)]


def hilo(y):
    hi = O.e4m3_bits_to_f64(O.f32_to_e4m3_bits_satfinite(y.astype(np.float32)))
    rem = (y.astype(np.float32) - hi.astype(np.float32)).astype(np.float64)   # binary32, as the kernel
    assert np.array_equal(rem, y - hi)                                          # exact: no rounding
    lo = O.e4m3_bits_to_f64(O.f32_to_e4m3_bits_satfinite(rem.astype(np.float32)))
    return hi, lo


def test_hi_plus_lo_is_exact_in_the_scaled_range():
    v = all_bf16_values()
    y = v[(np.abs(v) >= 0.25) & (np.abs(v) < 256.0)]
    assert y.size == 2 * 10 * 128          # ten binades of 128 significands, both signs
    hi, lo = hilo(y)
    assert np.array_equal(hi + lo, y)


def test_small_values_lose_at_most_2_to_minus_10():
    v = all_bf16_values()
    y = v[np.abs(v) < 0.25]
    hi, lo = hilo(y)
    err = np.abs(hi + lo - y)
    assert err.max() <= 2.0 ** -10
    assert err.max() > 0          # the bound is met, not vacuous: tiny values do lose bits


def test_token_scale_puts_the_largest_value_in_128_256():
    """s = 2^(E - 7) for a largest value with binary exponent E: largest / s in [128, 256),
    so no code saturates (e4m3's largest finite value is 448) and everything from 2^-10 of
    the largest value up is exact."""
    rng = np.random.default_rng(0)
    mx = np.abs(rng.standard_normal(1000)) * 10.0 ** rng.uniform(-20, 20, 1000)
    e = np.frexp(mx)[1] - 1 - 7
    r = mx / np.ldexp(1.0, e)
    assert np.all((r >= 128.0) & (r < 256.0))
    hi, lo = hilo(np.array([255.9375, -255.9375, 128.0, 248.0]))   # top of the range: no saturation
    assert np.array_equal(hi + lo, [255.9375, -255.9375, 128.0, 248.0])

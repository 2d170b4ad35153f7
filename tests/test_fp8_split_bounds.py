"""The error bounds the e4m3 path states for its two-term operands, checked on
the arithmetic alone (no GPU).

The kernel multiplies an e4m3 cache as stored.  q enters as hi + lo, two
e4m3 terms of 2^k q, with k putting the largest |q| of a 64-row head group
in [2^7, 2^8).  The softmax weights P (at most 2^8 under the lazy rescale)
enter as an e4m3 hi term plus an e5m2 lo term.  The header states these
bounds:
  * hi + lo is exact for elements down to 2^-9 of the largest |q|, and
    off by at most 2^-10 (in units of 2^k q) below that;
  * the weights' relative error is <= 2^-7 down to 2^-6 of the running
    maximum, and weights keep a nonzero value down to 2^-16 of it.
Each term is rounded as its format defines: nearest, ties to the even code,
saturating.  e4m3 comes from the oracle's encoder, e5m2 from the encoder
below, written from the format's bit layout.
"""
import numpy as np

import oracle


def e4m3(x):
    return oracle.e4m3_to_f64(oracle.f32_to_e4m3(np.asarray(x, dtype=np.float32)))


def _e5m2_finite():
    """Non-negative finite OCP e5m2 values, ascending, with their codes:
    exponent bits 6..2 (bias 15), mantissa bits 1..0; exponent 0 is
    subnormal, m/4 * 2^-14; exponent 31 is Inf / NaN."""
    codes = np.arange(0x7C)
    e = (codes >> 2) & 0x1F
    m = (codes & 3).astype(np.float64)
    vals = np.where(e == 0, m / 4.0 * 2.0 ** -14, (1.0 + m / 4.0) * np.exp2(e - 15.0))
    return vals, codes


def e5m2(x):
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    vals, codes = _e5m2_finite()
    a = np.abs(x)
    hi = np.minimum(np.searchsorted(vals, a, side="left"), len(vals) - 1)
    lo = np.maximum(hi - 1, 0)
    dlo, dhi = a - vals[lo], vals[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & ((codes[hi] & 1) == 0))
    v = np.where(a >= vals[-1], vals[-1], np.where(pick_hi, vals[hi], vals[lo]))
    v = np.where(vals[hi] == a, vals[hi], v)
    return np.where(np.signbit(x), -v, v)


def test_e5m2_encoder_against_its_definition():
    vals, _ = _e5m2_finite()
    assert vals[1] == 2.0 ** -16 and vals[-1] == 57344.0 and np.all(np.diff(vals) > 0)
    assert np.array_equal(e5m2(vals), vals)                       # exact values stay
    mid = (vals[1:] + vals[:-1]) / 2                              # ties go to the even code
    got = e5m2(mid)
    even = np.where((np.arange(1, len(vals)) & 1) == 0, vals[1:], vals[:-1])
    assert np.array_equal(got, even)
    assert e5m2(1e9) == 57344.0                                   # saturates
    assert e5m2(-3e-6) == 0 and e5m2(-8e-6) == -(2.0 ** -16)      # below / above half the step


def _split_q(q):
    """The kernel's split of one head group's rows: k from the largest |q|'s
    exponent, x = 2^k q, hi = e4m3(x), lo = e4m3(x - hi)."""
    mx = np.abs(q).max()
    e = int(np.frexp(mx)[1]) - 1                 # the bf16 exponent of the maximum
    k = min(126, max(-126, 7 - e))
    x = q.astype(np.float64) * 2.0 ** k
    hi = e4m3(x)
    lo = e4m3(x - hi)
    return x, hi, lo, mx


def _bf16(x):
    b = np.asarray(x, dtype=np.float32).view(np.uint32)
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return b.view(np.float32)


def test_q_hi_plus_lo_exact_down_to_2_pow_minus_9_of_the_max():
    rng = np.random.default_rng(5)
    for scale_exp in (-20, -3, 0, 6, 30):
        q = _bf16(rng.standard_normal((64, 576)) * 2.0 ** rng.uniform(-14, 2, (64, 576))
                  * 2.0 ** scale_exp)
        x, hi, lo, mx = _split_q(q)
        big = np.abs(q) >= 2.0 ** -9 * mx
        assert big.sum() > 1000 and (~big).sum() > 1000
        assert np.array_equal(hi[big] + lo[big], x[big])
        assert np.abs(hi + lo - x).max() <= 2.0 ** -10
        assert np.abs(x).max() < 2.0 ** 8                         # below e4m3's 448


def test_weights_relative_error_and_floor():
    p = np.exp2(np.linspace(-20.0, 8.0, 200001)).astype(np.float32).astype(np.float64)
    hi = e4m3(p)
    lo = e5m2(p - hi)
    rel = np.abs(hi + lo - p) / p
    assert rel[p >= 2.0 ** -6].max() <= 2.0 ** -7
    assert np.all(hi[p >= 2.0 ** -16] + lo[p >= 2.0 ** -16] > 0)
    assert np.all(hi[p < 2.0 ** -17] + lo[p < 2.0 ** -17] == 0)


def test_an_e4m3_lo_term_would_drop_weights_below_2_pow_minus_10():
    """What the e5m2 lo term is for: with e4m3 for both terms every weight
    below 2^-10 of the maximum rounds to zero, e.g. e^-10 (about 2^-14.4)."""
    p = np.float32(np.exp(-10.0))
    assert e4m3(p) + e4m3(p - e4m3(p)) == 0
    assert e4m3(p) + e5m2(p - e4m3(p)) > 0

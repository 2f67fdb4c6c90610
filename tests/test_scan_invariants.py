"""Number-format facts the streaming pass's packed scans rest on, checked on the host.

Draft rows of a top-k request are scanned on raw float32 bit patterns with unsigned integer
maxima, and bf16 target rows are flagged against a threshold rounded down to bf16.  Both
shortcuts are exact only because of the properties below (IEEE 754 binary32 / bfloat16
layouts); a kernel change that leaned on a wrong one would show up in GPU parity, this file
states them where they can be read and checked without a GPU.
"""
import numpy as np


def _bits(x):
    return np.asarray(x, np.float32).view(np.uint32)


def test_unsigned_order_is_float_order_without_sign_bit():
    rng = np.random.default_rng(7)
    # normal, subnormal, zero, huge and infinite non-negative values
    vals = np.concatenate([rng.random(20000, dtype=np.float32),
                           rng.random(2000, dtype=np.float32) * np.float32(1e-40),
                           np.float32([0.0, np.inf, np.finfo(np.float32).max, np.finfo(np.float32).tiny])])
    a, b = rng.choice(vals, 50000), rng.choice(vals, 50000)
    assert np.array_equal(a < b, _bits(a) < _bits(b))
    assert np.array_equal(a >= b, _bits(a) >= _bits(b))
    # the unsigned maximum of the bits is the bits of the float maximum
    assert np.array_equal(np.maximum(_bits(a), _bits(b)), _bits(np.maximum(a, b)))


def test_sign_bit_and_nan_land_outside_the_finite_range():
    top = _bits(np.float32(np.inf))
    # a positive NaN sorts above +inf, still below the sign bit: its max is a NaN
    assert top < _bits(np.float32(np.nan)) < 0x80000000
    # every value with the sign bit set, -0.0 included, compares above all of them
    for v in (-0.0, -1e-45, -1.0, -np.inf):
        assert _bits(np.float32(v)) >= 0x80000000
    assert _bits(np.float32(-0.0)) == 0x80000000
    # -0.0 is a valid probability: it is not below zero as a float
    assert np.float32(-0.0) >= np.float32(0.0)


def test_threshold_bits_for_non_positive_thresholds():
    # a threshold <= 0 (or NaN) becomes 0 as bits, which every non-negative value reaches,
    # a superset of the float comparison against it
    rng = np.random.default_rng(8)
    vals = rng.random(1000, dtype=np.float32)
    for th in (np.float32(0.0), np.float32(-0.0), np.float32(-3.0), np.float32(-np.inf)):
        assert np.all((vals >= th) <= (_bits(vals) >= 0))


def _bf16_round_down(x):
    """Largest bfloat16 value <= x (x finite float32): truncate the low 16 bits of a
    non-negative value; step one bf16 ulp further from zero for a negative one that had any."""
    b = _bits(x).astype(np.uint64)
    hi = b & 0xFFFF0000
    neg = (b & 0x80000000) != 0
    lost = (b & 0xFFFF) != 0
    hi = np.where(neg & lost, hi + 0x10000, hi)
    return (hi.astype(np.uint32)).view(np.float32)


def test_bf16_values_reaching_th_reach_its_rounding_down():
    rng = np.random.default_rng(9)
    th = (rng.standard_normal(20000) * 4).astype(np.float32)
    v = (rng.standard_normal(20000) * 4).astype(np.float32)
    v = (_bits(v) & 0xFFFF0000).view(np.float32)          # bf16-representable values
    rd = _bf16_round_down(th)
    assert np.all(rd <= th)
    assert np.all(_bits(rd) & 0xFFFF == 0)                  # rd is a bf16 value
    # the flag set against rd contains the flag set against th, and differs from it only by
    # values in [rd, th), i.e. by values equal to rd
    hit_th, hit_rd = v >= th, v >= rd
    assert np.all(hit_th <= hit_rd)
    assert np.all(v[hit_rd & ~hit_th] == rd[hit_rd & ~hit_th])

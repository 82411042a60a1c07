"""Pins of the oracle's binary16 conversions against numpy's own float16
implementation (an independent conversion routine), on every binary16 value,
every rounding midpoint and its neighbours, special values and random bits."""

import numpy as np

import oracle


def test_f16_to_f64_all_patterns():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_bits_to_f64(h)
    ref = h.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signs of zeros too
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def _check(x32):
    x32 = np.ascontiguousarray(x32, dtype=np.float32)
    got = oracle.f32_to_f16_bits(x32)
    with np.errstate(over="ignore", invalid="ignore"):
        ref = x32.astype(np.float16)
    refb = ref.view(np.uint16)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got.view(np.float16)), nan)
    bad = np.nonzero((got != refb) & ~nan)[0]
    assert bad.size == 0, (x32[bad[:5]], got[bad[:5]], refb[bad[:5]])


def test_f32_to_f16_exact_values_roundtrip():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    _check(h.view(np.float16).astype(np.float32))


def test_f32_to_f16_midpoints_and_neighbours():
    # midpoints between consecutive finite binary16 values of the same sign,
    # where round-half-to-even decides, and one float32 ulp either side
    pos = np.arange(0, 0x7C00, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float64)
    mids = (pos[:-1] + pos[1:]) / 2.0  # exact in float64, representable in float32
    mids32 = mids.astype(np.float32)
    assert np.array_equal(mids32.astype(np.float64), mids)
    below = np.nextafter(mids32, np.float32(0))
    above = np.nextafter(mids32, np.float32(np.inf))
    allv = np.concatenate([mids32, below, above])
    _check(allv)
    _check(-allv)


def test_f32_to_f16_specials_and_overflow():
    vals = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 65504.0, 65519.0, 65519.996, 65520.0,
                     -65520.0, 1e10, 2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001, 2.0 ** -26,
                     2.0 ** -14, 2.0 ** -14 * (1 - 2.0 ** -11), 6.1e-5, 1e-45, -1e-45,
                     3.4028235e38], dtype=np.float32)
    _check(vals)


def test_f32_to_f16_random_bits():
    rng = np.random.default_rng(1234)
    bits = rng.integers(0, 2 ** 32, size=1 << 21, dtype=np.uint64).astype(np.uint32)
    _check(bits.view(np.float32))
    # random values concentrated in the binary16 range, including subnormals
    e = rng.integers(-30, 17, size=1 << 20)
    m = rng.random(1 << 20) + 1.0
    s = np.where(rng.random(1 << 20) < 0.5, -1.0, 1.0)
    _check((s * m * np.exp2(e)).astype(np.float32))

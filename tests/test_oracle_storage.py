"""Pins of the oracle's storage conversions against numpy's IEEE conversions."""
import numpy as np

import dsa_synth
import oracle


def test_f16_decode_all_bit_patterns():
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def test_f16_encode_matches_numpy_rne():
    rng = np.random.default_rng(0)
    xs = np.concatenate([
        rng.standard_normal(20000) * 0.1,
        rng.standard_normal(2000) * 1e-6,           # subnormal range
        rng.standard_normal(2000) * 3e4,            # near overflow
        [65504.0, 65519.99, 65520.0, -65520.0, 0.0, -0.0, 2.0 ** -25, 2.0 ** -24 * 1.5,
         2.0 ** -14, 2.0 ** -14 * (1 - 2 ** -12)],
    ])
    # exact ties: midpoints between adjacent fp16 values
    a = rng.integers(0x0001, 0x7BFE, 3000).astype(np.uint16)
    lo = a.view(np.float16).astype(np.float64)
    hi = (a + 1).astype(np.uint16).view(np.float16).astype(np.float64)
    xs = np.concatenate([xs, (lo + hi) / 2, -(lo + hi) / 2])
    with np.errstate(over="ignore"):
        ref = xs.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f64_to_f16_bits(float(x)) for x in xs], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_generator_rounding_is_rne():
    # the generator's bf16 rounding against an exact big-integer construction
    rng = np.random.default_rng(1)
    a = rng.integers(0x0080, 0x7F00, 4000).astype(np.uint32)
    lo = (a << 16).view(np.float32).astype(np.float64)
    hi = ((a + 1) << 16).view(np.float32).astype(np.float64)
    mid = (lo + hi) / 2
    got = dsa_synth.f64_to_bf16_bits(mid)
    even = np.where(a % 2 == 0, a, a + 1).astype(np.uint16)
    assert np.array_equal(got, even)
    near_lo = lo + (hi - lo) * 0.49
    assert np.array_equal(dsa_synth.f64_to_bf16_bits(near_lo), a.astype(np.uint16))
    near_hi = lo + (hi - lo) * 0.51
    assert np.array_equal(dsa_synth.f64_to_bf16_bits(near_hi), (a + 1).astype(np.uint16))

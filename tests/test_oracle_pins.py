"""The fp64 oracle against facts fixed by the pages and the mathematics (CPU only)."""
import fractions

import numpy as np
import pytest

import oracle
from oracle_pins import ALL_PINS


@pytest.fixture(scope="module")
def lib():
    return oracle.load_library()


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(lib, pin):
    pin(lib)


def _rne_fp16_exact(v: float) -> float:
    """Round a double to binary16 by exact rational arithmetic (brute force over the grid)."""
    q = fractions.Fraction(v)
    if q == 0:
        return 0.0
    sign = -1 if q < 0 else 1
    q = abs(q)
    # binary16: 10 fraction bits, exponent -14..15, subnormal step 2^-24
    e = max(-14, q.numerator.bit_length() - q.denominator.bit_length())
    while fractions.Fraction(2) ** e > q and e > -14:
        e -= 1
    while fractions.Fraction(2) ** (e + 1) <= q:
        e += 1
    step = fractions.Fraction(2) ** (max(e, -14) - 10)
    k, rem = divmod(q, step)
    if rem * 2 > step or (rem * 2 == step and k % 2 == 1):
        k += 1
    r = k * step
    if r > 65504:
        return sign * float("inf")
    return sign * float(r)


def _rne_exact(v: float, frac_bits: int, emin: int, max_finite: float) -> float:
    """Round a double to a binary format with `frac_bits` fraction bits and minimum normal
    exponent `emin` by exact rational arithmetic (ties to even; past max_finite: inf)."""
    q = fractions.Fraction(v)
    if q == 0:
        return 0.0
    sign = -1 if q < 0 else 1
    q = abs(q)
    e = max(emin, q.numerator.bit_length() - q.denominator.bit_length())
    while fractions.Fraction(2) ** e > q and e > emin:
        e -= 1
    while fractions.Fraction(2) ** (e + 1) <= q:
        e += 1
    step = fractions.Fraction(2) ** (max(e, emin) - frac_bits)
    k, rem = divmod(q, step)
    if rem * 2 > step or (rem * 2 == step and k % 2 == 1):
        k += 1
    r = k * step
    if r > max_finite:
        return sign * float("inf")
    return sign * float(r)


BF16_MAX = float((2 - 2 ** -7) * 2 ** 127)


def test_round_bf16_is_round_to_nearest_even():
    """The oracle's fp64 -> bf16 rounding (used for bf16 residual sums) against exact
    rational rounding (7 fraction bits, fp32 exponent range) at half-way points between
    neighbouring bf16 values, one fp64 ulp to either side, large values near overflow and
    random values; ties must go to the even neighbour."""
    rng = np.random.default_rng(1)
    bits = rng.integers(0x0080, 0x7F7F, size=3000, dtype=np.uint32) << 16  # normal bf16
    a = bits.view(np.float32).astype(np.float64)
    b = (bits + (1 << 16)).view(np.float32).astype(np.float64)
    mids = (a + b) / 2
    probes = np.concatenate([mids, np.nextafter(mids, np.inf), np.nextafter(mids, -np.inf),
                             -mids, rng.standard_normal(2000) * 50,
                             [BF16_MAX, BF16_MAX * (1 + 2 ** -9), BF16_MAX * (1 + 2 ** -8), 1.0,
                              1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8)]])
    got = oracle.round_bf16(probes)
    want = np.array([_rne_exact(float(v), 7, -126, BF16_MAX) for v in probes])
    assert np.array_equal(got, want)
    # the ties above: 1 + 2^-8 rounds down to 1 (even), 1 + 3*2^-8 up to 1 + 2^-6
    assert oracle.round_bf16([1 + 2 ** -8])[0] == 1.0
    assert oracle.round_bf16([1 + 3 * 2 ** -8])[0] == 1 + 2 ** -6


def test_round_fp16_is_round_to_nearest_even():
    """numpy's fp64 -> fp16 conversion (used for the stored residual sum) rounds to nearest
    even, checked against exact rational rounding at every half-way point of a sweep of
    binades and one fp64 ulp to either side of it."""
    rng = np.random.default_rng(0)
    halves = rng.integers(0, 0x7BFF, size=4000, dtype=np.uint16).view(np.float16)
    a = halves.astype(np.float64)
    b = np.nextafter(halves, np.float16(np.inf)).astype(np.float64)
    mids = (a + b) / 2  # exact in fp64
    probes = np.concatenate([mids, np.nextafter(mids, np.inf), np.nextafter(mids, -np.inf),
                             -mids, rng.standard_normal(2000) * 100])
    got = oracle.round_fp16(probes).astype(np.float64)
    want = np.array([_rne_fp16_exact(float(v)) for v in probes])
    assert np.array_equal(got, want)

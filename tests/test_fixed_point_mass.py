"""The select kernel's fixed-point arithmetic, restated on the host, against exact values.

The boundary select turns each softmax weight e in [0, 1] (fp32) into the
integer round(e * 2^40), ties to even, with integer operations on the fp32 bit
pattern, and the Top-p threshold into ceil(top_p * T) for an fp32 top_p and a
64-bit total T, from a 128-bit product.  The Top-p working sets ("GrowPage:
On-Demand KV Budgeting for Efficient LLM Reasoning Serving", evolve.pub review,
section "Summary") are counted on those integers, so the counts are exact once
these two are.  This file restates both integer procedures step by step and
checks them against exact rational arithmetic on every exponent, on the
rounding ties and on the extremes.
"""
from fractions import Fraction
from math import ceil

import numpy as np
import pytest

M64 = (1 << 64) - 1


def mass_q_bits(b: int) -> int:
    """round(e * 2^40) from the bit pattern b of e >= 0: e = m * 2^(E - 150)."""
    E = b >> 23
    if E == 0:
        return 0                      # zero or subnormal: below 2^-86
    m = (b & 0x7FFFFF) | 0x800000
    sh = 110 - E
    if sh <= 0:
        return (m << -sh) if -sh <= 40 else 0
    if sh > 25:
        return 0                      # m < 2^24 < half of 2^sh
    q, rem, half = m >> sh, m & ((1 << sh) - 1), 1 << (sh - 1)
    return q + (1 if rem > half or (rem == half and q & 1) else 0)


def mass_exact(b: int) -> int:
    """Round-to-nearest-even of the exact value e * 2^40."""
    x = Fraction(float(np.uint32(b).view(np.float32))) * (1 << 40)
    fl = x.numerator // x.denominator
    frac = x - fl
    if frac > Fraction(1, 2) or (frac == Fraction(1, 2) and fl & 1):
        fl += 1
    return fl


def ceil_mul_bits(top_p_bits: int, T: int) -> int:
    """ceil(top_p * T) from a 128-bit product M * T, top_p = M * 2^-r."""
    E = (top_p_bits >> 23) & 0xFF
    M = (top_p_bits & 0x7FFFFF) if E == 0 else ((top_p_bits & 0x7FFFFF) | 0x800000)
    r = 150 - (1 if E == 0 else E)
    prod = M * T
    lo, hi = prod & M64, prod >> 64
    if r >= 128:
        return 1 if (lo | hi) else 0
    if r >= 64:
        qv = hi if r == 64 else hi >> (r - 64)
        rem = lo | (0 if r == 64 else hi & ((1 << (r - 64)) - 1))
    elif r == 0:
        qv, rem = lo, 0
    else:
        qv = ((lo >> r) | (hi << (64 - r))) & M64
        rem = lo & ((1 << r) - 1)
    return qv + (1 if rem else 0)


def _weights(rng):
    """Bit patterns of weights in [0, 1]: every exponent with random
    mantissas, exact rounding ties, 1.0, zero and subnormals."""
    out = [0, 1, 0x007FFFFF, 0x00800000, 0x3F800000]
    for E in range(1, 128):
        out += [(E << 23) | int(x) for x in rng.integers(0, 1 << 23, 40)]
        sh = 110 - E
        if 1 <= sh <= 23:             # mantissas whose remainder is exactly half (odd and even q)
            for q in ((1 << (23 - sh)) + 1, (1 << (24 - sh)) - 2, (1 << (24 - sh)) - 1):
                m = (q << sh) | (1 << (sh - 1))
                if (1 << 23) <= m < (1 << 24):
                    out.append((E << 23) | (m & 0x7FFFFF))
    return out


def test_mass_matches_round_to_nearest_even_of_the_exact_product():
    rng = np.random.default_rng(7)
    for b in _weights(rng):
        assert mass_q_bits(b) == mass_exact(b), hex(b)


def test_mass_of_one_and_monotone():
    assert mass_q_bits(0x3F800000) == 1 << 40
    rng = np.random.default_rng(8)
    bs = sorted(_weights(rng))
    ms = [mass_q_bits(b) for b in bs]
    assert all(a <= c for a, c in zip(ms, ms[1:]))   # order kept (ties allowed)


@pytest.mark.parametrize("top_p", [1.0, 0.999, 0.99, 0.9, 0.5, 0.05, 1e-6, 1e-30, 1e-40])
def test_threshold_is_the_exact_ceiling(top_p):
    b = int(np.float32(top_p).view(np.uint32))
    exact_tp = Fraction(float(np.float32(top_p)))
    rng = np.random.default_rng(b)
    totals = [0, 1, 2, 3, 1 << 40, (1 << 40) + 1, (1 << 52) + 12345, M64 >> 1, M64 - 1]
    totals += [int(x) for x in rng.integers(1, 1 << 62, 50, dtype=np.int64)]
    for T in totals:
        assert ceil_mul_bits(b, T) == ceil(exact_tp * T), (top_p, T)

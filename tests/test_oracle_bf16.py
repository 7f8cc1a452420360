"""Pins for the two bf16 rounding routines: the oracle's (from float64) and
the input generator's (from float32).

Every rounding point of the oracle's layer, attention and SFT definitions runs
through ``oracle.bf16.round_bf16``, and every seeded input through
``seeded_inputs.round_bf16``.  Neither is checked against itself here:

* float32 inputs against torch's own float32 -> bfloat16 conversion (a
  library routine: round to nearest, ties to even), over every binade,
  subnormals, hand-built exact ties with even and odd lower mantissas, values
  one step either side of a tie, carries into the next binade, the largest
  finite value, overflow, infinities, signed zeros and NaN;
* float64 inputs that float32 cannot hold against an exact rational
  nearest-even computation (``fractions.Fraction``): a routine that went
  through float32 first would round twice and fail these;
* planted mistakes (ties away from zero, truncation, rounding via float32,
  a wrong shift, overflow of the largest finite value) fail the same pins.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle.bf16 import round_bf16

# float32 signalling-NaN patterns widen to float64 with an "invalid" warning
pytestmark = pytest.mark.filterwarnings("ignore:invalid value encountered in cast")


def _f32_from_bits(bits):
    return np.asarray(bits, dtype=np.uint32).view(np.float32)


def _torch_bf16(x32):
    """torch's conversion of float32 values to bfloat16, back as float64."""
    return torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def _same(a, b):
    """Bitwise-equal as float64 (so -0 != +0 and NaN == NaN)."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    both_nan = np.isnan(a) & np.isnan(b)
    return both_nan | (a.view(np.uint64) == b.view(np.uint64))


def _f32_cases():
    """float32 inputs spanning the whole range, with every edge the format has."""
    g = np.random.default_rng(123)
    # random bit patterns: every binade, both signs, subnormals included
    rnd = g.integers(0, 0x7F800000, size=20000, dtype=np.uint32)
    rnd |= (g.integers(0, 2, size=rnd.size, dtype=np.uint32) << np.uint32(31))
    # exact ties between two bf16 neighbours: low 16 bits 0x8000, with an even
    # and an odd bf16 mantissa below the tie, and one float32 step either side
    hi = g.integers(0x0001, 0x7F7F, size=4000, dtype=np.uint32)
    hi_even, hi_odd = hi & ~np.uint32(1), hi | np.uint32(1)
    ties = []
    for h in (hi_even, hi_odd):
        for low in (0x8000, 0x7FFF, 0x8001, 0x0000, 0xFFFF):
            ties.append((h << np.uint32(16)) | np.uint32(low))
    ties = np.concatenate(ties)
    ties = np.concatenate([ties, ties | np.uint32(0x80000000)])
    edges = np.array([
        0x3FFF8000,  # 1.9921875 + half a step: odd mantissa, carries to 2.0
        0x3F7F8000,  # the same one binade lower: carries to 1.0
        0x007F8000,  # largest subnormal mantissa + half: carries to the smallest normal
        0x00008000,  # half the smallest subnormal step: tie between 0 and 2^-133, stays 0
        0x00018000,  # one and a half steps: tie, rounds to the even 2 steps
        0x00000001,  # smallest float32 subnormal: rounds to 0
        0x7F7F0000,  # largest finite bf16: stays
        0x7F7F7FFF,  # just below the overflow midpoint: largest finite
        0x7F7F8000,  # the overflow midpoint (odd mantissa): infinity
        0x7F7FFFFF,  # largest float32: infinity
        0x7F800000,  # +inf
        0x00000000,  # +0
        0x7FC00000,  # NaN
        0x7F800001,  # signalling-NaN pattern
    ], dtype=np.uint32)
    edges = np.concatenate([edges, edges | np.uint32(0x80000000)])
    return _f32_from_bits(np.concatenate([rnd, ties, edges]))


def _exact_nearest_bf16(v: float) -> float:
    """Nearest bf16 of a float64 by exact rational arithmetic, ties to even."""
    if math.isnan(v) or math.isinf(v) or v == 0.0:
        return v
    a = Fraction(abs(v))
    e = math.frexp(abs(v))[1] - 1                  # 2^e <= |v| < 2^(e+1)
    step = Fraction(2) ** (max(e, -126) - 7)       # 8 significant bits, or the subnormal step
    n = a / step
    k = math.floor(n)
    rem = n - k
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and k % 2 == 1):
        k += 1
    val = k * step
    if val >= Fraction(2) ** 128:
        return math.copysign(math.inf, v)
    return math.copysign(float(val), v)


def _f64_cases():
    """float64 values float32 cannot hold, including values within one
    float64 step of a bf16 tie (where rounding via float32 rounds twice)."""
    g = np.random.default_rng(7)
    e = g.integers(-140, 128, size=3000)
    m = 1.0 + g.random(3000)
    rnd = np.ldexp(m, e) * np.where(g.random(3000) < 0.5, -1.0, 1.0)
    # bf16 ties +- one float64 ulp, in normal binades
    base = g.integers(1 << 7, 1 << 8, size=1000).astype(np.float64)   # 8-bit significands
    ex = g.integers(-120, 120, size=1000)
    tie = np.ldexp(base + 0.5, ex - 7)
    near = np.concatenate([np.nextafter(tie, np.inf), np.nextafter(tie, -np.inf), -np.nextafter(tie, np.inf)])
    # the overflow boundary from float64
    mid = float.fromhex("0x1.ffp127")              # midpoint between the largest finite and 2^128
    edges = np.array([np.nextafter(mid, 0.0), mid, np.nextafter(mid, np.inf), float.fromhex("0x1.fep127"),
                      2.0 ** -126 - 2.0 ** -140, 2.0 ** -134, 2.0 ** -134 + 2.0 ** -160, 1e-300, -1e-300])
    return np.concatenate([rnd, near, edges])


def _f32_violations(fn):
    x = _f32_cases()
    got = np.asarray(fn(x), dtype=np.float64)
    return int(np.count_nonzero(~_same(got, _torch_bf16(x))))


def _f64_violations(fn):
    x = _f64_cases()
    got = np.asarray(fn(x), dtype=np.float64)
    ref = np.array([_exact_nearest_bf16(float(v)) for v in x])
    return int(np.count_nonzero(~_same(got, ref)))


def test_oracle_rounding_matches_torch_on_float32_inputs():
    assert _f32_violations(lambda x: round_bf16(np.asarray(x, dtype=np.float64))) == 0


def test_oracle_rounding_is_exact_nearest_even_from_float64():
    assert _f64_violations(round_bf16) == 0


def test_generator_rounding_matches_torch():
    assert _f32_violations(lambda x: si.round_bf16(x).astype(np.float64)) == 0


def test_hand_checked_values():
    # 1 + 2^-8 is the tie between 1 and 1 + 2^-7: the even neighbour is 1
    assert round_bf16(1.0 + 2.0 ** -8) == 1.0
    # 1 + 3 * 2^-8 is the tie between 1 + 2^-7 (odd) and 1 + 2^-6 (even)
    assert round_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    assert round_bf16(-(1.0 + 3 * 2.0 ** -8)) == -(1.0 + 2.0 ** -6)
    assert round_bf16(1.0 + 2.0 ** -8 + 2.0 ** -40) == 1.0 + 2.0 ** -7
    assert round_bf16(255.5) == 256.0                 # carry into the next binade
    assert round_bf16(float.fromhex("0x1.fep127")) == float.fromhex("0x1.fep127")
    assert round_bf16(float.fromhex("0x1.ffp127")) == np.inf
    assert round_bf16(-float.fromhex("0x1.c4p127") - 2.0 ** 118) == -float.fromhex("0x1.c4p127")
    assert np.signbit(round_bf16(-0.0))
    assert np.isnan(round_bf16(np.nan))


def _ties_away(x):
    d = np.asarray(x, dtype=np.float64)
    u = d.view(np.uint64)
    r = ((u + np.uint64(1 << 44)) >> np.uint64(45)) << np.uint64(45)
    return round_bf16(r.view(np.float64))


def _truncate(x):
    d = np.asarray(x, dtype=np.float64)
    u = d.view(np.uint64)
    return round_bf16(((u >> np.uint64(45)) << np.uint64(45)).view(np.float64))


def _via_float32(x):
    return round_bf16(np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64))


def _shift_44(x):
    d = np.asarray(x, dtype=np.float64)
    u = d.view(np.uint64)
    keep = (u >> np.uint64(44)) & np.uint64(1)
    r = ((u + np.uint64((1 << 43) - 1) + keep) >> np.uint64(44)) << np.uint64(44)
    return r.view(np.float64)


def _max_finite_overflows(x):
    out = round_bf16(x)
    d = np.asarray(x, dtype=np.float64)
    return np.where(np.abs(d) >= float.fromhex("0x1.fep127"), np.copysign(np.inf, d), out)


@pytest.mark.parametrize("mutant", [_ties_away, _truncate, _shift_44, _max_finite_overflows])
def test_planted_mistakes_fail_the_float32_pins(mutant):
    assert _f32_violations(mutant) > 0


@pytest.mark.parametrize("mutant", [_ties_away, _truncate, _via_float32, _shift_44])
def test_planted_mistakes_fail_the_float64_pins(mutant):
    assert _f64_violations(mutant) > 0

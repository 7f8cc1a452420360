"""Pins for the NF4 oracle: facts fixed by the data type's definition, not by the oracle itself."""
import math
import os

import numpy as np
import pytest

import seeded_inputs as si
from oracle import nf4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "nf4_levels_qlora.txt")


def acklam_quantile(p):
    """Acklam's rational approximation of the normal quantile, refined by Halley steps on erfc."""
    a = [-3.969683028665376e+01, 2.209460984245205e+02, -2.759285104469687e+02,
         1.383577518672690e+02, -3.066479806614716e+01, 2.506628277459239e+00]
    b = [-5.447609879822406e+01, 1.615858368580409e+02, -1.556989798598866e+02,
         6.680131188771972e+01, -1.328068155288572e+01]
    c = [-7.784894002430293e-03, -3.223964580411365e-01, -2.400758277161838e+00,
         -2.549732539343734e+00, 4.374664141464968e+00, 2.938163982698783e+00]
    d = [7.784695709041462e-03, 3.224671290700398e-01, 2.445134137142996e+00,
         3.754408661907416e+00]
    plow = 0.02425
    if p < plow:
        q = math.sqrt(-2 * math.log(p))
        x = (((((c[0] * q + c[1]) * q + c[2]) * q + c[3]) * q + c[4]) * q + c[5]) / \
            ((((d[0] * q + d[1]) * q + d[2]) * q + d[3]) * q + 1)
    elif p <= 1 - plow:
        q = p - 0.5
        r = q * q
        x = (((((a[0] * r + a[1]) * r + a[2]) * r + a[3]) * r + a[4]) * r + a[5]) * q / \
            (((((b[0] * r + b[1]) * r + b[2]) * r + b[3]) * r + b[4]) * r + 1)
    else:
        q = math.sqrt(-2 * math.log(1 - p))
        x = -(((((c[0] * q + c[1]) * q + c[2]) * q + c[3]) * q + c[4]) * q + c[5]) / \
            ((((d[0] * q + d[1]) * q + d[2]) * q + d[3]) * q + 1)
    for _ in range(3):
        e = 0.5 * math.erfc(-x / math.sqrt(2)) - p
        u = e * math.sqrt(2 * math.pi) * math.exp(x * x / 2)
        x = x - u / (1 + x * u / 2)
    return x


def table_from(quantile):
    delta = 1.0 - 0.5 * (1.0 / 30.0 + 1.0 / 32.0)
    pos = [quantile(p) for p in np.linspace(delta, 0.5, 9)[:-1]]
    neg = [-quantile(p) for p in np.linspace(delta, 0.5, 8)[:-1]]
    v = np.array(sorted(pos + [0.0] + neg))
    return (v / v.max()).astype(np.float32)


def test_table_structure():
    T = nf4.code_table()
    assert T.dtype == np.float32 and T.shape == (16,)
    assert np.all(np.diff(T) > 0)
    assert T[0] == -1.0 and T[7] == 0.0 and T[15] == 1.0
    assert np.sum(T > 0) == 8 and np.sum(T < 0) == 7


def test_table_matches_independent_quantiles_bitwise():
    T = nf4.code_table()
    assert np.array_equal(table_from(acklam_quantile).view(np.uint32), T.view(np.uint32))
    from scipy.special import ndtri
    assert np.array_equal(table_from(lambda p: float(ndtri(p))).view(np.uint32), T.view(np.uint32))


def test_table_matches_published_levels():
    vals = [float(l) for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    assert len(vals) == 16
    np.testing.assert_allclose(nf4.code_table(), vals, rtol=0, atol=6e-5)


def test_exact_levels_map_to_their_codes():
    T = nf4.code_table()
    for scale in (1.0, 0.25, 2.0 ** -7, 8.0):
        row = np.tile(T * np.float32(scale), 4).astype(np.float32)   # 64 values, absmax = scale
        codes, absmax = nf4.quantize(row[None, :])
        assert absmax[0] == np.float32(scale)
        assert np.array_equal(nf4.unpack(codes, 1, 64)[0], np.tile(np.arange(16), 4))
        assert np.array_equal(nf4.dequantize(codes, absmax, 1, 64)[0], row)


def test_midpoint_ties_and_neighbours():
    T = nf4.code_table().astype(np.float64)
    for j in range(15):
        mid = (T[j] + T[j + 1]) / 2
        mid32 = np.float32(mid)
        below = np.nextafter(np.float32(min(mid32, mid)), np.float32(-2))
        above = np.nextafter(np.float32(max(mid32, mid)), np.float32(2))
        assert nf4.nearest_code(np.array([below]))[0] == j
        assert nf4.nearest_code(np.array([above]))[0] == j + 1
        if float(mid32) == mid:          # an exactly representable midpoint: tie -> lower level
            assert nf4.nearest_code(np.array([mid32]))[0] == j


def test_nearest_is_brute_force_nearest():
    g = np.random.default_rng(5)
    x = g.uniform(-1, 1, 20000).astype(np.float32)
    T = nf4.code_table()
    got = nf4.nearest_code(x)
    for xi, ci in zip(x[:3000], got[:3000]):
        d = [abs(float(xi) - float(t)) for t in T]
        best = min(d)
        assert ci == d.index(best)


def test_quantize_round_trip_and_extremes():
    g = np.random.default_rng(7)
    W = (g.standard_normal((8, 256)) * 0.02).astype(np.float32)
    codes, absmax = nf4.quantize(W)
    assert codes.shape == (8 * 256 // 2,) and absmax.shape == (8 * 256 // 64,)
    np.testing.assert_array_equal(absmax, np.abs(W.reshape(-1, 64)).max(axis=1))
    What = nf4.dequantize(codes, absmax, 8, 256).reshape(-1, 64)
    T = nf4.code_table()
    for b in range(What.shape[0]):
        allowed = set((T * absmax[b]).astype(np.float32).tolist())
        assert set(What[b].tolist()) <= allowed
        i = np.argmax(np.abs(W.reshape(-1, 64)[b]))
        assert What[b, i] == W.reshape(-1, 64)[b, i]        # |w| = absmax maps to +-absmax exactly
    # nearest-level error bound: half the widest gap times absmax
    gap = np.max(np.diff(T.astype(np.float64))) / 2
    err = np.abs(What - W.reshape(-1, 64)) / absmax[:, None]
    assert np.all(err <= gap + 1e-7)


def test_packing_high_nibble_first():
    T = nf4.code_table()
    row = np.zeros(64, np.float32)
    row[0], row[1] = T[15], T[0]          # codes 15, 0 -> byte 0xF0
    row[2], row[3] = T[3], T[12]          # codes 3, 12 -> byte 0x3C
    codes, _ = nf4.quantize(row[None, :])
    assert codes[0] == 0xF0 and codes[1] == 0x3C
    assert np.all(codes[2:] == 0x77)      # zeros -> code 7 in both nibbles


def test_zero_block_and_nonfinite():
    W = np.zeros((2, 128), np.float32)
    W[1, 64:] = 0.5
    codes, absmax = nf4.quantize(W)
    assert np.all(nf4.unpack(codes, 2, 128)[0] == 7) and absmax[0] == 0
    assert np.all(nf4.dequantize(codes, absmax, 2, 128)[0] == 0)
    W[0, 3] = np.inf
    with pytest.raises(ValueError):
        nf4.quantize(W)
    with pytest.raises(ValueError):
        nf4.quantize(np.zeros((1, 96), np.float32))


# ------------------------------------------------------ double quantisation
def test_fma32_is_one_rounding_of_the_exact_value():
    from fractions import Fraction
    rng = np.random.default_rng(7)
    n = 3000
    s = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    c = (rng.standard_normal(n) * np.exp(rng.uniform(-25, 25, n))).astype(np.float32)   # c >> s q too
    q = rng.integers(-127, 128, n)
    r = nf4.fma32(s, q, c)
    for i in range(n):
        ex = Fraction(float(s[i])) * int(q[i]) + Fraction(float(c[i]))
        f = np.float32(float(ex))
        cands = [f, np.nextafter(f, np.float32(np.inf)), np.nextafter(f, np.float32(-np.inf))]
        best = min(cands, key=lambda v: (abs(Fraction(float(v)) - ex), int(np.float32(v).view(np.uint32)) & 1))
        assert r[i] == best, i


def test_dq_block_mean_scale_and_extremes():
    # values on a 2^-12 grid: float64 sums are exact, the mean is a plain average
    rng = np.random.default_rng(3)
    N, K = 512, 128                                   # 2 transposed rows x 2 blocks of 256
    a = (rng.integers(100, 400, size=N * K // 64) * 2.0 ** -12).astype(np.float32)
    q, a2 = nf4.double_quantize(a, N, K)
    at = a.reshape(N, K // 64).T.reshape(K // 64, N // 256, 256)
    for j in range(K // 64):
        for b in range(N // 256):
            v = at[j, b].astype(np.float64)
            c = np.float32(v.sum() / 256)
            assert a2[j, b, 0] == c
            d = (at[j, b] - c).astype(np.float32)
            s = np.float32(np.max(np.abs(d)) / np.float32(127))
            assert a2[j, b, 1] == s
            qq = q[j, b * 256:(b + 1) * 256].astype(np.int32)
            k = int(np.argmax(np.abs(d)))
            assert abs(qq[k]) == 127 and np.sign(qq[k]) == np.sign(d[k])
            assert np.all(np.abs(qq) <= 127)


def test_dq_nearest_level_brute_force_and_error_bound():
    rng = np.random.default_rng(11)
    N, K = 256, 64 * 6
    W = si.normal_bf16(5, (N, K), 0.02)
    _, a = nf4.quantize(W)
    q, a2 = nf4.double_quantize(a, N, K)
    ap = nf4.dq_absmax(q, a2, N, K)
    at = a.reshape(N, K // 64).T
    apt = ap.reshape(N, K // 64).T
    for j in range(K // 64):
        c, s = a2[j, 0]
        d = (at[j] - c).astype(np.float32)
        r = (d / s).astype(np.float32)                         # the float32 quotient the rule rounds
        cand = np.arange(-127, 128, dtype=np.float64)
        dist = np.abs(r.astype(np.float64)[:, None] - cand[None, :])
        best = dist.min(axis=1)
        for n in range(N):                                     # nearest integer, ties to even
            ks = cand[dist[n] == best[n]]
            want = ks[0] if len(ks) == 1 else ks[np.argmin(np.abs(ks) % 2)]
            assert q[j, n] == want
        # |a' - a| <= s / 2 (plus the final float32 rounding)
        assert np.all(np.abs(apt[j].astype(np.float64) - at[j]) <= s / 2 * (1 + 1e-6) + np.spacing(at[j]))


def test_dq_constant_block_is_exact():
    N, K = 256, 64
    a = np.full(N, 0.03125, np.float32)
    q, a2 = nf4.double_quantize(a, N, K)
    assert np.all(q == 0) and a2[0, 0, 1] == 0
    assert np.array_equal(nf4.dq_absmax(q, a2, N, K), a)


def test_dq_layer_bytes_match_the_pages_buffer():
    # 8B layer: 218.1M params; 4-bit codes + 8-bit absmax per 64 + (c, s) per 256 blocks
    params = sum(n * k for n, k in ((4096, 4096), (1024, 4096), (1024, 4096), (4096, 4096),
                                    (14336, 4096), (14336, 4096), (4096, 14336)))
    dq = params // 2 + params // 64 + params // (64 * 256) * 8
    assert abs(dq / 1e6 - 113) / 113 < 0.01            # the pages' two 113 MB layer buffers
    assert abs(32 * dq / 1e9 - 3.60) / 3.60 < 0.01     # and the 3.60 GB pinned base store

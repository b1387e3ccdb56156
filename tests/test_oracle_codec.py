"""Pins for the oracle's MX element codecs, encoders and block-scaled products.

Each check ties the oracle to something other than itself: the printed table
of "Kimi K3: 2.8 Trillion Parameters, Four Bits at a Time" (section "Four
bits from the start"), the OCP MX element definitions the pages cite
("Kimi K3 and the New Open-Weights Moat", section "Precision and
deployment", Fig. 6), exact rational arithmetic, or a numpy matmul in the
special case where the MX scales are all 2^0.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from conftest import read_golden

E2M1_GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


# ------------------------------------------------------------------ element tables
def test_e2m1_grid_and_sign():
    # The page lists the eight magnitudes; bit 3 is the sign.
    for c in range(8):
        assert oracle.e2m1_decode(c) == E2M1_GRID[c]
        assert oracle.e2m1_decode(c | 8) == -E2M1_GRID[c] or (c == 0 and oracle.e2m1_decode(8) == 0.0)


def test_e4m3_hand_cases():
    d = oracle.e4m3_decode
    assert d(0x00) == 0.0
    assert d(0x01) == 2.0 ** -9          # smallest subnormal
    assert d(0x07) == 7 * 2.0 ** -9      # largest subnormal
    assert d(0x08) == 2.0 ** -6          # smallest normal
    assert d(0x38) == 1.0                # exponent field 7 = bias
    assert d(0x78) == 256.0
    assert d(0x7E) == 448.0              # largest finite
    assert np.isnan(d(0x7F)) and np.isnan(d(0xFF))
    assert d(0xFE) == -448.0
    assert d(0xB8) == -1.0


def test_e8m0_hand_cases():
    assert oracle.e8m0_decode(127) == 1.0
    assert oracle.e8m0_decode(0) == 2.0 ** -127
    assert oracle.e8m0_decode(254) == 2.0 ** 127
    assert np.isnan(oracle.e8m0_decode(255))


# ------------------------------------------------------------------ MXFP4 encoder
def _page_metrics(w, q):
    rel = np.linalg.norm(w - q) / np.linalg.norm(w)
    small = np.abs(w) < np.quantile(np.abs(w), 0.99)
    rel_small = np.linalg.norm(w[small] - q[small]) / np.linalg.norm(w[small])
    dead = (q[small] == 0).mean() * 100
    return rel, rel_small, dead


def test_mxfp4_reproduces_printed_table():
    rows = {r[0]: tuple(float(v) for v in r[1:]) for r in read_golden("mxfp4_vs_int4_table.txt")}
    rng = np.random.default_rng(7)
    w = rng.normal(0, 0.02, 1 << 20)
    c, s = oracle.mxfp4_encode(w[None])
    got = _page_metrics(w, oracle.mxfp4_decode(c, s)[0])
    assert (round(got[0], 4), round(got[1], 4), round(got[2], 2)) == rows["gaussian"]
    w_out = w.copy()
    hit = rng.choice(w_out.size, w_out.size // 500, replace=False)
    w_out[hit] = rng.choice([-1, 1], hit.size) * 0.6
    c, s = oracle.mxfp4_encode(w_out[None])
    got = _page_metrics(w_out, oracle.mxfp4_decode(c, s)[0])
    assert (round(got[0], 4), round(got[1], 4), round(got[2], 2)) == rows["gaussian+outliers"]


def test_mxfp4_tie_rule_and_clip():
    # amax = 4 -> shared exponent floor(log2 4) - 2 = 0, scale 1: the scaled
    # values are the raw ones.  A tie goes to the first (smaller) level.
    vals = [4.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.75, 0.0, 0.1, 0.3, 2.9, -4.0, 1.0, 6.0]
    vals += [0.0] * (32 - len(vals))
    c, s = oracle.mxfp4_encode(np.array([vals]))
    assert s[0, 0] == 127
    dec = oracle.mxfp4_decode(c, s)[0]
    expect = [4.0, 0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, -0.5, 0.0, 0.0, 0.5, 3.0, -4.0, 1.0, 6.0]
    assert list(dec[:16]) == expect
    # the clip at 6: amax 7 -> exponent floor(log2 7) - 2 = 0, 7 -> 6
    v = np.zeros((1, 32)); v[0, 0] = 7.0; v[0, 1] = -7.0
    c, s = oracle.mxfp4_encode(v)
    assert s[0, 0] == 127 and list(oracle.mxfp4_decode(c, s)[0, :2]) == [6.0, -6.0]
    # element 2i sits in the low nibble: 4.0 is level 6, 0.25 -> level 0
    c, _ = oracle.mxfp4_encode(np.array([vals]))
    assert c[0, 0] == 0x06


def test_mxfp4_zero_block():
    c, s = oracle.mxfp4_encode(np.zeros((2, 64)))
    assert (c == 0).all() and (s == 0).all()


def test_mxfp4_scale_tracks_amax():
    rng = np.random.default_rng(3)
    for n in (-20, -5, 0, 7, 30):
        v = rng.normal(size=(1, 32)) * 2.0 ** n
        _, s = oracle.mxfp4_encode(v)
        amax = np.abs(v).max()
        assert int(s[0, 0]) - 127 == int(np.floor(np.log2(amax))) - 2


# ------------------------------------------------------------------ MXFP8 quantiser
def _round_half_even(fr: Fraction) -> int:
    n, r = divmod(fr.numerator, fr.denominator)
    twice = 2 * r
    if twice > fr.denominator or (twice == fr.denominator and n % 2 == 1):
        n += 1
    return n


def _floor_log2(fr: Fraction) -> int:
    n = fr.numerator.bit_length() - fr.denominator.bit_length()
    while Fraction(2) ** n > fr:
        n -= 1
    while Fraction(2) ** (n + 1) <= fr:
        n += 1
    return n


def _e4m3_rne_sat(q: Fraction, negative: bool) -> int:
    """Exact E4M3 encoding by integer arithmetic on the significand."""
    s = 0x80 if negative else 0
    a = abs(q)
    if a >= 448:
        return s | 0x7E
    if a < Fraction(1, 64):                      # below the smallest normal
        m = _round_half_even(a * 512)            # quantum 2^-9
        return s | m                             # m == 8 is exactly 2^-6
    n = _floor_log2(a)
    m = _round_half_even(a / Fraction(2) ** (n - 3))   # 8 <= m <= 16
    if m == 16:
        n, m = n + 1, 8
    code = ((n + 7) << 3) | (m - 8)
    return s | (0x7E if code > 0x7E else code)


def _bf16_value(bits: int) -> Fraction:
    e = (bits >> 7) & 0xFF
    m = bits & 0x7F
    v = Fraction(m, 1) * Fraction(2) ** -133 if e == 0 else Fraction(128 + m) * Fraction(2) ** (e - 134)
    return -v if bits & 0x8000 else v


def _reference_block(bits_block):
    vals = [_bf16_value(b) for b in bits_block]
    amax = max(abs(v) for v in vals)
    e = -127 if amax == 0 else max(-127, min(127, _floor_log2(amax) - 8))
    codes = [_e4m3_rne_sat(v * Fraction(2) ** -e, bool(b & 0x8000)) for v, b in zip(vals, bits_block)]
    return codes, e + 127


def _bits_to_f32(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


def _finite_bf16_patterns():
    allb = np.arange(65536, dtype=np.uint32)
    finite = ((allb >> 7) & 0xFF) != 0xFF
    return allb[finite]


def test_mxfp8_exhaustive_bf16_against_exact_rounding():
    pats = _finite_bf16_patterns()
    pats = pats[: (len(pats) // 32) * 32]
    rng = np.random.default_rng(11)
    # consecutive patterns share a binade; shuffled ones mix magnitudes
    blocks = np.concatenate([pats.reshape(-1, 32), rng.permutation(pats).reshape(-1, 32)[:600]])
    codes, scales = oracle.mxfp8_quantize(_bits_to_f32(blocks).reshape(blocks.shape))
    for b in range(blocks.shape[0]):
        rc, rs = _reference_block([int(x) for x in blocks[b]])
        assert scales[b, 0] == rs, b
        assert list(codes[b]) == rc, b


def test_mxfp8_hand_cases():
    v = np.zeros((1, 32), np.float32)
    v[0, 0] = 1.0
    v[0, 1] = -0.5
    c, s = oracle.mxfp8_quantize(v)
    assert s[0, 0] == 119                 # floor(log2 1) - 8 = -8
    assert c[0, 0] == 0x78                # 1.0 * 2^8 = 256
    assert c[0, 1] == 0xF0                # -128
    v = np.zeros((1, 32), np.float32)
    v[0, 0] = 500.0                       # floor(log2 500) = 8 -> scale 2^0
    v[0, 1] = 300.0
    c, s = oracle.mxfp8_quantize(v)
    assert s[0, 0] == 127 and c[0, 0] == 0x7E and oracle.e4m3_decode(c[0, 1]) == 288.0
    z = np.zeros((1, 32), np.float32)
    z[0, 5] = -0.0
    c, s = oracle.mxfp8_quantize(z)
    assert s[0, 0] == 0 and c[0, 5] == 0x80 and c[0, 0] == 0


def test_mxfp8_scale_equivariance():
    rng = np.random.default_rng(5)
    v = rng.normal(size=(64, 32)).astype(np.float32)
    c0, s0 = oracle.mxfp8_quantize(v)
    for n in (-30, -3, 4, 40):
        c1, s1 = oracle.mxfp8_quantize(v * np.float32(2.0 ** n))
        assert (c1 == c0).all()
        assert (s1.astype(int) == s0.astype(int) + n).all()


def test_e4m3_encode_round_trip():
    for code in range(256):
        if code & 0x7F == 0x7F:
            continue
        v = oracle.e4m3_decode(code)
        got = oracle.e4m3_encode(v)
        assert got == code or (v == 0.0 and got & 0x7F == 0)


# ------------------------------------------------------------------ block-scaled product
def _random_mx4(rng, M, K, scale_lo=120, scale_hi=134):
    codes = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    scales = rng.integers(scale_lo, scale_hi, size=(M, K // 32), dtype=np.uint8)
    return codes, scales


def _random_mx8(rng, N, K, scale_lo=110, scale_hi=130):
    codes = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3F       # no NaN codes
    scales = rng.integers(scale_lo, scale_hi, size=(N, K // 32), dtype=np.uint8)
    return codes, scales


# Tables typed from the OCP element definitions, independent of the oracle.
_E2M1 = np.array(E2M1_GRID + [-x for x in E2M1_GRID])


def _e4m3_table():
    t = np.zeros(256)
    for c in range(256):
        e, m = (c >> 3) & 15, c & 7
        v = m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        t[c] = -v if c & 0x80 else v
        if c & 0x7F == 0x7F:
            t[c] = np.nan
    return t


def test_mx_matmul_unit_scales_is_numpy_matmul():
    rng = np.random.default_rng(1)
    M, N, K = 24, 10, 96
    ac, _ = _random_mx4(rng, M, K)
    bc, _ = _random_mx8(rng, N, K)
    a_s = np.full((M, K // 32), 127, np.uint8)
    b_s = np.full((N, K // 32), 127, np.uint8)
    A = np.empty((M, K))
    A[:, 0::2] = _E2M1[ac & 15]
    A[:, 1::2] = _E2M1[ac >> 4]
    B = _e4m3_table()[bc]
    got = oracle.mx_matmul(ac, a_s, bc, b_s)
    assert got.shape == (N, M)
    np.testing.assert_array_equal(got, B @ A.T)   # small exact dyadics: no rounding


def test_mx_matmul_exact_rational():
    rng = np.random.default_rng(2)
    M, N, K = 5, 3, 128
    ac, as_ = _random_mx4(rng, M, K)
    bc, bs = _random_mx8(rng, N, K)
    got = oracle.mx_matmul(ac, as_, bc, bs)
    e4 = _e4m3_table()
    for n in range(N):
        for m in range(M):
            exact = Fraction(0)
            mag = Fraction(0)
            for k in range(K):
                nib = (ac[m, k // 2] >> (4 * (k & 1))) & 15
                term = (Fraction(_E2M1[nib]) * Fraction(2) ** (int(as_[m, k // 32]) - 127)
                        * Fraction(e4[bc[n, k]]) * Fraction(2) ** (int(bs[n, k // 32]) - 127))
                exact += term
                mag += abs(term)
            assert abs(Fraction(got[n, m]) - exact) <= mag * K * Fraction(2) ** -52

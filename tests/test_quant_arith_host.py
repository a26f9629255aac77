"""The quantiser's division-free quotients, checked on the host.

For a 1x16 group with e4m3 scale s the codes are e2m1_rne_sat(RN(x / s))
("GPU kernel porting with AI agents", section "Sage Attention 3": 1x16 NVFP4
groups with e4m3 scales).  The kernel forms the quotient as
RN(x * yh + RN(x * yl)) with yh = RD(1/s) and yl = RN((1 - s * yh) * yh),
i.e. without a divide and with one correction term.  These tests confirm that
the two-term product gives the same e2m1 code as the correctly rounded
quotient for every finite bf16 x (Q and V) and every positive finite e4m3
scale; for float32 x (K' = K - mean), for every significand within 2^12 ulps
of s times each e2m1 boundary, for every scale significand (exponents only
shift both sides; away from a boundary a 2^-45 error cannot change a code);
and that dropping the correction term (one rounded product with RN(1/s))
would not do: it misses exact ties.  Cases near a boundary are settled with
exact rational arithmetic.
"""

from fractions import Fraction

import numpy as np

from oracle.formats import e2m1_encode, e4m3_decode

F32 = np.float32
BOUNDARIES = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


def _all_bf16():
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    x = bits.view(np.float32)
    return x[np.isfinite(x)]


def _scales():
    codes = np.arange(1, 127, dtype=np.uint8)          # every positive finite e4m3 value
    return e4m3_decode(codes).astype(np.float32)


def _rd_recip(s):
    v = F32(1.0 / np.float64(s))
    if Fraction(float(v)) > 1 / Fraction(float(s)):
        v = np.nextafter(v, F32(0))
    return v


def _f32_round(r):
    """Correctly rounded float32 of a Fraction (ties to even)."""
    v = F32(float(r))
    cands = [v, np.nextafter(v, F32(np.inf)), np.nextafter(v, F32(-np.inf))]
    def key(c):
        bits = int(np.array([c], dtype=np.float32).view(np.uint32)[0])
        return (abs(Fraction(float(c)) - r), bits & 1)
    return min(cands, key=key)


def test_two_term_product_gives_the_quotients_codes_for_every_bf16_value():
    x = _all_bf16()
    checked_exactly = 0
    for s in _scales():
        yh = _rd_recip(s)
        res = Fraction(1) - Fraction(float(s)) * Fraction(float(yh))
        assert res >= 0 and Fraction(float(F32(float(res)))) == res      # exact residual
        yl = F32(np.float64(F32(float(res))) * np.float64(yh))
        t = (x.astype(np.float64) * np.float64(yl)).astype(np.float32)     # RN(x * yl)
        q = (x.astype(np.longdouble) * np.longdouble(yh) + t.astype(np.longdouble)).astype(np.float32)
        want = e2m1_encode((x / s).astype(np.float32))
        got = e2m1_encode(q)
        aq = np.abs(q.astype(np.float64))
        near = np.zeros(x.size, dtype=bool)
        for b in BOUNDARIES:
            near |= np.abs(aq - b) <= b * 2.0 ** -16
        near |= want != got
        for i in np.nonzero(near)[0]:
            exact = _f32_round(Fraction(float(x[i])) * Fraction(float(yh)) + Fraction(float(t[i])))
            got[i] = e2m1_encode(np.array([exact]))[0]
            checked_exactly += 1
        assert np.array_equal(got, want), float(s)
    assert checked_exactly > 1000


def test_signed_zero_survives_the_two_term_product():
    for s in _scales():
        yh = _rd_recip(s)
        yl = F32(np.float64(F32(float(Fraction(1) - Fraction(float(s)) * Fraction(float(yh))))) * np.float64(yh))
        assert yl >= 0
        for z in (F32(0.0), F32(-0.0)):
            q = F32(z * yh) + F32(z * yl)
            assert np.signbit(q) == np.signbit(z)


def test_one_rounded_product_is_not_enough():
    """RN(x * RN(1/s)) misses ties: x / s = 1.25 with s = 1.875 rounds up."""
    x = _all_bf16()
    misses = 0
    for s in _scales():
        y = F32(1.0) / s
        misses += int(np.sum(e2m1_encode((x * y).astype(np.float32)) != e2m1_encode((x / s).astype(np.float32))))
    assert misses > 0


def test_two_term_product_gives_the_quotients_codes_near_every_boundary_float32():
    checked_exactly = 0
    for m in range(8, 16):                               # every scale significand
        s = F32(m / 8.0)
        yh = _rd_recip(s)
        res = Fraction(1) - Fraction(float(s)) * Fraction(float(yh))
        yl = F32(np.float64(F32(float(res))) * np.float64(yh))
        for b in BOUNDARIES:
            centre = F32(b * float(s))                   # exact: <= 7 significant bits
            bits = int(np.array([centre], np.float32).view(np.uint32)[0])
            x = (np.arange(bits - 4096, bits + 4097, dtype=np.int64).astype(np.uint32)).view(np.float32)
            t = (x.astype(np.float64) * np.float64(yl)).astype(np.float32)
            q = (x.astype(np.longdouble) * np.longdouble(yh) + t.astype(np.longdouble)).astype(np.float32)
            want = e2m1_encode((x / s).astype(np.float32))
            got = e2m1_encode(q)
            near = (np.abs(np.abs(q.astype(np.float64)) - b) <= b * 2.0 ** -20) | (want != got)
            for i in np.nonzero(near)[0]:
                exact = _f32_round(Fraction(float(x[i])) * Fraction(float(yh)) + Fraction(float(t[i])))
                got[i] = e2m1_encode(np.array([exact]))[0]
                checked_exactly += 1
            assert np.array_equal(got, want), (m, b)
    assert checked_exactly > 100

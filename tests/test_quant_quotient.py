"""The activation quant's fp32-scale quotient, checked exhaustively on the CPU.

The CUDA activation quant does not divide each value by its scale.  With
r = fp32(1/s) it forms q0 = fp32(x*r), the exact residual e = x - q0*s (one
FMA) and q1 = fp32(q0 + e*r) (one FMA): P. Markstein's correction step
("Computation of elementary functions on the IBM RISC System/6000 processor",
IBM J. Res. Develop. 34(1), 1990).  The method computes (e4m3 or int8
codes of) fp32(x/s), the IEEE quotient, only if q1 equals it.  This test
models the three steps in exact integer arithmetic with round-to-nearest-even
to 24 bits and checks q1 == fp32(x/s) for every pair the kernel can meet:
every bf16 (8-bit) or fp16 (11-bit) input significand against the scale
fp32(A/Q) of every amax significand A of the same format, Q = 448 (e4m3) and
127 (int8), and against the eps scale fp32(fp32(1e-10)/Q).  Powers of two
commute with every step while the values stay normal, so significands cover
every exponent; quotients below 2^-126 give a zero code either way (the
kernel keeps the sign of x for a zero, as the division does).
"""
import struct
from fractions import Fraction

import pytest


def rn24(num, den):
    """Round-to-nearest-even of the positive rational num/den to 24
    significant bits: (m, e) with value m * 2^e, 2^23 <= m < 2^24."""
    e = num.bit_length() - den.bit_length()
    if (num << max(0, -e)) < (den << max(0, e)):
        e -= 1
    sh = e - 23
    n2, d2 = (num, den << sh) if sh >= 0 else (num << -sh, den)
    q, r = divmod(n2, d2)
    if 2 * r > d2 or (2 * r == d2 and q & 1):
        q += 1
    if q == 1 << 24:
        q, sh = q >> 1, sh + 1
    return q, sh


def rn(num, den):
    """fp32 round-to-nearest-even of the signed rational num/den, as an exact
    rational (num, den) with den > 0."""
    if num == 0:
        return 0, 1
    m, e = rn24(abs(num), den)
    if num < 0:
        m = -m
    return (m << e, 1) if e >= 0 else (m, 1 << -e)


def corrected_quotient(x, s):
    """The kernel's three steps on exact rationals (num, den)."""
    r = rn(s[1], s[0])
    q0 = rn(x[0] * r[0], x[1] * r[1])
    # the residual x - q0*s, rounded once (the FMA)
    e = rn(x[0] * q0[1] * s[1] - q0[0] * s[0] * x[1], x[1] * q0[1] * s[1])
    # q0 + e*r, rounded once (the FMA)
    return rn(q0[0] * e[1] * r[1] + e[0] * r[0] * q0[1], q0[1] * e[1] * r[1])


def same(a, b):
    return a[0] * b[1] == b[0] * a[1]


def scales(bits, Q):
    one = 1 << (bits - 1)
    out = {rn(A, one * Q) for A in range(one, 2 * one)}
    eps32 = Fraction(struct.unpack("<f", struct.pack("<f", 1e-10))[0])
    out.add(rn(eps32.numerator, eps32.denominator * Q))
    return sorted(out)


@pytest.mark.parametrize("Q", [448, 127])
@pytest.mark.parametrize("bits", [8, 11])
def test_corrected_quotient_is_the_ieee_quotient(bits, Q):
    one = 1 << (bits - 1)
    bad = []
    for s in scales(bits, Q):
        for X in range(one, 2 * one):
            x = (X, one)
            if not same(corrected_quotient(x, s), rn(x[0] * s[1], x[1] * s[0])):
                bad.append((x, s))
    assert not bad, f"{len(bad)} pairs differ, e.g. {bad[:3]}"


def test_model_detects_a_missing_correction():
    # the product alone is not always the IEEE quotient: the model must see it
    one = 1 << 7
    wrong = 0
    for s in scales(8, 448):
        r = rn(s[1], s[0])
        for X in range(one, 2 * one):
            wrong += not same(rn(X * r[0], one * r[1]), rn(X * s[1], one * s[0]))
    assert wrong > 0
    # and one case by hand: 3 / 1.75 = 12/7
    assert same(corrected_quotient((3, 1), (7, 4)), rn(12, 7))

"""Pins for the oracle's MXFP4 decode (CPU only).

The oracle decodes E2M1 with a value table and E8M0 with ldexp.  These tests pin
it to things other than itself:
  * a generic sign/exponent/mantissa minifloat decoder, itself checked against
    numpy's float16 and the float32 bit pattern of bf16 over every bit pattern,
    evaluated at the E2M1 field widths (2 exponent bits, bias 1, 1 mantissa bit);
  * IEEE float32 bit construction for 2^(s-127);
  * hand-built bytes from the vendor convention (tests/golden);
  * brute-force decoding of whole matrices.
"""
import math
import os

import numpy as np
import pytest

import datagen
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def minifloat(bits: int, e_bits: int, m_bits: int, bias: int, ieee_specials: bool) -> float:
    """Value of a sign|exponent|mantissa bit pattern (generic binary floating point)."""
    sign = -1.0 if (bits >> (e_bits + m_bits)) & 1 else 1.0
    e = (bits >> m_bits) & ((1 << e_bits) - 1)
    m = bits & ((1 << m_bits) - 1)
    if ieee_specials and e == (1 << e_bits) - 1:
        return sign * math.inf if m == 0 else math.nan
    if e == 0:
        return sign * math.ldexp(m / (1 << m_bits), 1 - bias)
    return sign * math.ldexp(1.0 + m / (1 << m_bits), e - bias)


def same(a: float, b: float) -> bool:
    if math.isnan(a) or math.isnan(b):
        return math.isnan(a) and math.isnan(b)
    return a == b and math.copysign(1.0, a) == math.copysign(1.0, b)


def test_minifloat_decoder_matches_float16_everywhere():
    ref = np.arange(1 << 16, dtype=np.uint16).view(np.float16).astype(np.float64)
    for b in range(1 << 16):
        assert same(minifloat(b, 5, 10, 15, True), float(ref[b])), hex(b)


def test_minifloat_decoder_matches_bf16_everywhere():
    ref = (np.arange(1 << 16, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)
    for b in range(1 << 16):
        assert same(minifloat(b, 8, 7, 127, True), float(ref[b])), hex(b)


def test_e2m1_matches_format_definition():
    # OCP MX E2M1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit, no inf/nan
    for code in range(16):
        assert same(oracle.e2m1(code), minifloat(code, 2, 1, 1, False)), code
    assert math.copysign(1.0, oracle.e2m1(8)) == -1.0  # code 8 is negative zero


def test_doubled_e2m1_values_are_small_integers():
    # colibri PR #676 item 7: "The doubled e2m1 values are exact int8"
    for code in range(16):
        v2 = 2.0 * oracle.e2m1(code)
        assert v2 == int(v2) and -127 <= v2 <= 127


def test_ue8m0_is_power_of_two_from_float32_bits():
    for s in range(1, 255):
        f = float(np.array([s << 23], dtype=np.uint32).view(np.float32)[0])
        assert oracle.ue8m0(s) == f, s
    # s = 0: 2^-127 is the float32 subnormal with only mantissa bit 22 set
    assert oracle.ue8m0(0) == float(np.array([1 << 22], dtype=np.uint32).view(np.float32)[0])
    assert math.isnan(oracle.ue8m0(255))


def test_exhaustive_decode_codes_by_scales_100_to_150():
    scales = np.arange(100, 151, dtype=np.uint8)
    # one row per scale byte; 32 columns = each code twice (low and high nibble positions)
    O = scales.size
    q = np.zeros((O, 16), dtype=np.uint8)
    for j in range(16):
        lo, hi = j, (j + 7) % 16  # two different codes per byte
        q[:, j] = lo | (hi << 4)
    s = scales.reshape(O, 1)
    got = oracle.dequant(q, s)
    for r, sc in enumerate(scales):
        f = float(np.array([int(sc) << 23], dtype=np.uint32).view(np.float32)[0])
        for j in range(16):
            lo, hi = j, (j + 7) % 16
            assert same(got[r, 2 * j], minifloat(lo, 2, 1, 1, False) * f)
            assert same(got[r, 2 * j + 1], minifloat(hi, 2, 1, 1, False) * f)


def test_golden_nibble_order():
    rows = []
    with open(os.path.join(GOLDEN, "mxfp4_nibble_order.txt")) as fh:
        for line in fh:
            line = line.strip()
            if line and not line.startswith("#"):
                b, s, v0, v1 = line.split()
                rows.append((int(b, 16), int(s), float(v0), float(v1)))
    assert len(rows) >= 8
    for b, s, v0, v1 in rows:
        got = oracle.dequant(np.full((1, 16), b, dtype=np.uint8), np.full((1, 1), s, dtype=np.uint8))
        assert same(got[0, 0], v0) and same(got[0, 1], v1), (hex(b), s)
        assert same(got[0, 30], v0) and same(got[0, 31], v1)


def test_dequant_matrix_bruteforce():
    O, I = 48, 160
    q = datagen.u8(11, 99, O * I // 2).reshape(O, I // 2)
    s = datagen.int_u8(11, 98, O * I // 32, 110, 140).reshape(O, I // 32)
    got = oracle.dequant(q, s)
    for o in range(O):
        for c in range(I):
            byte = int(q[o, c // 2])
            code = (byte >> 4) if c % 2 else (byte & 15)
            ref = minifloat(code, 2, 1, 1, False) * 2.0 ** (int(s[o, c // 32]) - 127)
            assert same(got[o, c], ref)

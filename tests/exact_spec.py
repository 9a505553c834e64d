"""An independent statement of the correctly rounded block FMA, for pinning the oracle.

d = RNE_or_RTZ_fp32( sum_l a_l*b_l + c ) computed with Python's exact rationals, inputs
decoded with the standard library (struct for binary16/binary32) where it can.  This
is the closed form that the CDNA 1 model ("Accurate Models of AMD Matrix Cores",
Sec. 4.1) and any exact-then-round model must reproduce.
"""
import math
import struct
from fractions import Fraction

NAN, PINF, NINF = "nan", "+inf", "-inf"


def _from_float(x: float):
    if math.isnan(x):
        return NAN
    if math.isinf(x):
        return PINF if x > 0 else NINF
    return (Fraction(x), math.copysign(1.0, x) < 0)


def decode(fmt: str, bits: int, enc: str = "ocp"):
    """-> NAN | PINF | NINF | (Fraction value, sign bit)."""
    if fmt == "fp16":
        return _from_float(struct.unpack("<e", struct.pack("<H", bits))[0])
    if fmt == "fp32":
        return _from_float(struct.unpack("<f", struct.pack("<I", bits))[0])
    if fmt == "bf16":
        return _from_float(struct.unpack("<f", struct.pack("<I", bits << 16))[0])
    if fmt == "xf32":
        x = struct.unpack("<f", struct.pack("<I", bits))[0]
        if math.isnan(x) or math.isinf(x):
            return _from_float(x)
        return _from_float(struct.unpack("<f", struct.pack("<I", bits & 0xFFFFE000))[0])
    if fmt in ("e4m3", "e5m2"):
        e, m = (4, 3) if fmt == "e4m3" else (5, 2)
        bias = (7 if fmt == "e4m3" else 15) + (1 if enc == "fnuz" else 0)
        s, ef, mf = bits >> 7, (bits >> m) & ((1 << e) - 1), bits & ((1 << m) - 1)
        if enc == "fnuz" and bits == 0x80:
            return NAN
        if enc == "ocp" and fmt == "e4m3" and ef == 15 and mf == 7:
            return NAN
        if enc == "ocp" and fmt == "e5m2" and ef == 31:
            return NAN if mf else (NINF if s else PINF)
        v = Fraction(mf, 1 << m) * Fraction(2) ** (1 - bias) if ef == 0 else \
            Fraction((1 << m) + mf, 1 << m) * Fraction(2) ** (ef - bias)
        return (-v if s else v, bool(s))
    raise ValueError(fmt)


def round_fp32(x: Fraction, mode: str = "rne", zero_neg: bool = False) -> int:
    if x == 0:
        return 0x80000000 if zero_neg else 0
    sign = 0x80000000 if x < 0 else 0
    ax = abs(x)
    e = ax.numerator.bit_length() - ax.denominator.bit_length()
    if Fraction(2) ** e > ax:
        e -= 1
    e = max(e, -126)
    q = ax / Fraction(2) ** (e - 23)
    n = q.numerator // q.denominator
    r = q - n
    if mode == "rne" and (r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1)):
        n += 1
    if n == 1 << 24:
        n, e = 1 << 23, e + 1
    if e > 127:
        return sign | (0x7F800000 if mode == "rne" else 0x7F7FFFFF)
    if n < (1 << 23):
        return sign | n
    return sign | ((e + 127) << 23) | (n - (1 << 23))


def round_fp16(x: Fraction, mode: str = "rne", zero_neg: bool = False) -> int:
    """binary16 bits of x rounded once (RNE or toward zero) onto the binary16 grid:
    11-bit significands, exponents -14 .. 15, subnormal spacing 2^-24; overflow gives
    Inf under RNE and the largest finite value (65504) under RTZ."""
    if x == 0:
        return 0x8000 if zero_neg else 0
    sign = 0x8000 if x < 0 else 0
    ax = abs(x)
    e = ax.numerator.bit_length() - ax.denominator.bit_length()
    if Fraction(2) ** e > ax:
        e -= 1
    e = max(e, -14)
    q = ax / Fraction(2) ** (e - 10)
    n = q.numerator // q.denominator
    r = q - n
    if mode == "rne" and (r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1)):
        n += 1
    if n == 1 << 11:
        n, e = 1 << 10, e + 1
    if e > 15:
        return sign | (0x7C00 if mode == "rne" else 0x7BFF)
    if n < (1 << 10):
        return sign | n
    return sign | ((e + 15) << 10) | (n - (1 << 10))


def exact_block(fmt, a_bits, b_bits, c_bits, mode="rne", enc="ocp", nan_bits=0x7FC00000, acc="fp32"):
    """Correctly rounded sum_l a_l*b_l + c with IEEE special-value rules; with acc="fp16"
    c is the binary16 in the low half of c_bits and the result is binary16."""
    prods = []
    for x, y in zip(a_bits, b_bits):
        u, v = decode(fmt, int(x), enc), decode(fmt, int(y), enc)
        if NAN in (u, v):
            return nan_bits
        uinf, vinf = u in (PINF, NINF), v in (PINF, NINF)
        if uinf or vinf:
            other = v if uinf else u
            if other not in (PINF, NINF) and other[0] == 0:
                return nan_bits
            su = (u == NINF) if uinf else u[1]
            sv = (v == NINF) if vinf else v[1]
            prods.append(NINF if su != sv else PINF)
        else:
            prods.append((u[0] * v[0], u[1] != v[1]))
    c = decode("fp16", int(c_bits) & 0xFFFF) if acc == "fp16" else decode("fp32", int(c_bits))
    if c == NAN:
        return nan_bits
    terms = prods + [c]
    infs = {t for t in terms if t in (PINF, NINF)}
    if len(infs) == 2:
        return nan_bits
    if infs:
        if acc == "fp16":
            return 0x7C00 if PINF in infs else 0xFC00
        return 0x7F800000 if PINF in infs else 0xFF800000
    total = sum(t[0] for t in terms)
    zero_neg = all(t[0] == 0 and t[1] for t in terms)
    return round_fp16(total, mode, zero_neg) if acc == "fp16" else round_fp32(total, mode, zero_neg)

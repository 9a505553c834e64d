"""Seeded synthetic inputs for the emulator's workloads (host side, numpy only).

This module makes bit patterns; it holds none of the emulated arithmetic.  It
is the one piece shared by the tests, the benchmark and the oracle checks.
The sampling strategies follow "Accurate Models of AMD Matrix Cores":
independent bit sampling (Sec. 5.2) and exponent-mantissa sampling
(Sec. 5.1, Algorithm 3); the GEMM inputs are the shapes and distributions of
the dense, 2:4-sparse and multi-word GEMM workloads.
"""
from __future__ import annotations

import re
from fractions import Fraction

import numpy as np

# container dtype, exponent bits, mantissa bits, bias, IEEE Inf/NaN at the top exponent
_FMT = {
    "fp16": (np.uint16, 5, 10, 15),
    "bf16": (np.uint16, 8, 7, 127),
    "fp32": (np.uint32, 8, 23, 127),
    "xf32": (np.uint32, 8, 23, 127),
    "e4m3": (np.uint8, 4, 3, 7),
    "e5m2": (np.uint8, 5, 2, 15),
}
_FNUZ_BIAS = {"e4m3": 8, "e5m2": 16}

ELEM_DTYPE = {"fp16": np.uint16, "bf16": np.uint16, "xf32": np.uint32, "fp32": np.uint32,
              "e4m3": np.uint8, "e5m2": np.uint8, "int8": np.uint8, "uint8": np.uint8}


def fmt_params(fmt: str, enc: str = "ocp"):
    dt, e, m, bias = _FMT[fmt]
    if enc == "fnuz" and fmt in _FNUZ_BIAS:
        bias = _FNUZ_BIAS[fmt]
    return dt, e, m, bias


def has_inf(fmt: str, enc: str = "ocp") -> bool:
    return fmt in ("fp16", "bf16", "fp32", "xf32") or (fmt == "e5m2" and enc == "ocp")


# ---------------------------------------------------------------------------
# Exact value <-> bits for hand-written fixtures (raises when not representable)
# ---------------------------------------------------------------------------
def parse_value(s: str) -> Fraction | str:
    """'1+2^-23', '-(2^-24+2^-25)', '0x1.8p-3', 'inf', '-inf', 'nan', '-0' -> Fraction or tag."""
    s = s.strip().lower()
    if s in ("inf", "+inf", "-inf", "nan", "-nan", "-0"):
        return s
    if s.startswith(("0x", "-0x", "+0x")):
        return Fraction(float.fromhex(s))
    if not set(s) <= set("0123456789+-*/().^ "):
        raise ValueError(f"bad value expression {s!r}")
    # every number literal becomes an exact Fraction; '^' is a power
    expr = re.sub(r"(\d+\.\d+|\d+)", r'F("\1")', s).replace("^", "**")
    return Fraction(eval(expr, {"__builtins__": {}}, {"F": Fraction}))  # noqa: S307


def encode_exact(x, fmt: str, enc: str = "ocp") -> int:
    """Bit pattern of the exactly representable value x in the format."""
    dt, e, m, bias = fmt_params(fmt, enc)
    width = 1 + e + m
    if isinstance(x, str):
        if x in ("inf", "+inf", "-inf"):
            if not has_inf(fmt, enc):
                raise ValueError(f"{fmt}/{enc} has no Inf")
            sign = 1 if x.startswith("-") else 0
            return (sign << (width - 1)) | (((1 << e) - 1) << m)
        if x in ("nan", "-nan"):
            if enc == "fnuz" and fmt in _FNUZ_BIAS:
                return 0x80
            sign = 1 if x.startswith("-") else 0
            return (sign << (width - 1)) | (((1 << e) - 1) << m) | (1 << (m - 1))
        if x == "-0":
            if enc == "fnuz" and fmt in _FNUZ_BIAS:
                raise ValueError("FNUZ has no -0")
            return 1 << (width - 1)
        raise ValueError(x)
    x = Fraction(x)
    sign = 1 if x < 0 else 0
    ax = abs(x)
    if ax == 0:
        return 0
    E = ax.numerator.bit_length() - ax.denominator.bit_length()
    if Fraction(2) ** E > ax:
        E -= 1
    emin = 1 - bias
    if E < emin:
        E = emin
    q = ax / Fraction(2) ** (E - m)
    if q.denominator != 1:
        raise ValueError(f"{x} not representable in {fmt}")
    q = int(q)
    if q >= (1 << m):
        ef = E + bias
        mf = q - (1 << m)
    else:
        ef = 0
        mf = q
    top = (1 << e) - 1
    if ef > top or (ef == top and has_inf(fmt, enc)):
        raise ValueError(f"{x} overflows {fmt}")
    if fmt == "e4m3" and enc == "ocp" and ef == 15 and mf == 7:
        raise ValueError("448*1.125 is the E4M3 NaN pattern")
    return (sign << (width - 1)) | (ef << m) | mf


def encode_fp32(x) -> int:
    return encode_exact(x, "fp32")


# ---------------------------------------------------------------------------
# Format tables (finite values) for nearest-value conversion of random reals
# ---------------------------------------------------------------------------
def _finite_table(fmt: str, enc: str = "ocp"):
    dt, e, m, bias = fmt_params(fmt, enc)
    codes, vals = [], []
    for code in range(1 << (e + m)):        # non-negative codes only
        ef, mf = code >> m, code & ((1 << m) - 1)
        if has_inf(fmt, enc) and ef == (1 << e) - 1:
            continue
        if fmt == "e4m3" and enc == "ocp" and ef == 15 and mf == 7:
            continue
        v = (mf * 2.0 ** (1 - bias - m)) if ef == 0 else ((1 << m) + mf) * 2.0 ** (ef - bias - m)
        codes.append(code)
        vals.append(v)
    order = np.argsort(vals)
    return np.asarray(codes, dtype=np.int64)[order], np.asarray(vals, dtype=np.float64)[order]


def nearest_even(x: np.ndarray, fmt: str, enc: str = "ocp") -> np.ndarray:
    """Round binary64 samples to the nearest finite value of a small format, ties to the
    even code, saturating at the largest finite value (input preparation only)."""
    dt, e, m, bias = fmt_params(fmt, enc)
    codes, vals = _finite_table(fmt, enc)
    ax = np.minimum(np.abs(x), vals[-1])
    hi = np.clip(np.searchsorted(vals, ax, side="left"), 0, len(vals) - 1)
    lo = np.clip(hi - 1, 0, len(vals) - 1)
    dlo, dhi = ax - vals[lo], vals[hi] - ax
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(codes[lo] % 2 == 0, lo, hi)))
    out = codes[pick]
    neg = (x < 0) & (out != 0) if enc == "fnuz" else (np.signbit(x))
    width = 1 + e + m
    out = out | (neg.astype(np.int64) << (width - 1))
    return out.astype(dt)


def fp32_to_bf16_rne(x32: np.ndarray) -> np.ndarray:
    """binary32 -> bfloat16 bits, round to nearest even (input preparation only)."""
    u = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = (u + 0x7FFF + lsb) >> 16
    return r.astype(np.uint16)


# ---------------------------------------------------------------------------
# Block-FMA vector sets
# ---------------------------------------------------------------------------
def _rand_bits(rng, shape, width):
    return rng.integers(0, 1 << width, size=shape, dtype=np.uint64)


def finite_fp16_bits(rng, shape):
    """Uniform finite fp16 bit patterns (exponent field 31 redrawn)."""
    sign = rng.integers(0, 2, size=shape, dtype=np.uint64)
    ef = rng.integers(0, 31, size=shape, dtype=np.uint64)
    mf = rng.integers(0, 1 << 10, size=shape, dtype=np.uint64)
    return ((sign << 15) | (ef << 10) | mf).astype(np.uint16)


def gen_fp16_cancellation(n: int = 65536, k: int = 4, seed: int = 1):
    """FP16 K=4 vector sets with an FP32 addend: uniform finite FP16 patterns for a, b; the
    odd-indexed vectors get exponents clustered within 4 of a common base (cancellation);
    c is a uniform 32-bit pattern."""
    rng = np.random.default_rng(seed)
    a = finite_fp16_bits(rng, (n, k))
    b = finite_fp16_bits(rng, (n, k))
    odd = np.arange(n) % 2 == 1
    n_odd = int(odd.sum())
    for arr in (a, b):
        base = rng.integers(0, 28, size=(n_odd, 1), dtype=np.uint64)
        ef = base + rng.integers(0, 4, size=(n_odd, k), dtype=np.uint64)
        sign = rng.integers(0, 2, size=(n_odd, k), dtype=np.uint64)
        mf = rng.integers(0, 1 << 10, size=(n_odd, k), dtype=np.uint64)
        arr[odd] = ((sign << 15) | (ef << 10) | mf).astype(np.uint16)
    c = _rand_bits(rng, (n,), 32).astype(np.uint32)
    return a, b, c


def _special_codes(fmt: str, enc: str):
    """Bit patterns (positive, sign added by the caller) of the injected classes."""
    dt, e, m, bias = fmt_params(fmt, enc)
    out = {"zero": 0, "sub": None, "inf": None, "nan": None}
    if has_inf(fmt, enc):
        out["inf"] = ((1 << e) - 1) << m
    if enc == "fnuz" and fmt in _FNUZ_BIAS:
        out["nan"] = 0x80
    elif fmt == "e4m3":
        out["nan"] = 0x7F
    else:
        out["nan"] = (((1 << e) - 1) << m) | (1 << (m - 1))
    return out


def independent_bits(rng, fmt: str, shape, enc: str = "ocp", special_rate: float = 0.01):
    """Independent bit sampling (Sec. 5.2): every bit ~ Bernoulli(1/2); an exponent that
    would encode Inf/NaN is redrawn.  Then `special_rate` of the elements each become
    +-0, a subnormal, +-Inf (when the format has Inf) and NaN."""
    if fmt in ("int8", "uint8"):
        return rng.integers(0, 256, size=shape, dtype=np.uint64).astype(np.uint8)
    dt, e, m, bias = fmt_params(fmt, enc)
    width = 1 + e + m
    sign = rng.integers(0, 2, size=shape, dtype=np.uint64)
    mf = rng.integers(0, 1 << m, size=shape, dtype=np.uint64)
    top = (1 << e) - 1
    if has_inf(fmt, enc):
        ef = rng.integers(0, top, size=shape, dtype=np.uint64)        # never all-ones
    else:
        ef = rng.integers(0, top + 1, size=shape, dtype=np.uint64)
    bits = (sign << (width - 1)) | (ef << m) | mf
    if fmt == "e4m3" and enc == "ocp":                                    # S.1111.111 is NaN
        nanlike = (bits & 0x7F) == 0x7F
        bits[nanlike] = bits[nanlike] & ~np.uint64(1)
    if enc == "fnuz" and fmt in _FNUZ_BIAS:                               # 0x80 is NaN
        bits[bits == 0x80] = 0
    sc = _special_codes(fmt, enc)
    u = rng.random(size=shape)
    r = special_rate
    is_zero = u < r
    is_sub = (u >= r) & (u < 2 * r)
    is_inf = (u >= 2 * r) & (u < 3 * r)
    is_nan = (u >= 3 * r) & (u < 4 * r)
    neg = sign << (width - 1)
    bits = np.where(is_zero, (0 if enc == "fnuz" and fmt in _FNUZ_BIAS else neg), bits)
    submf = rng.integers(1, 1 << m, size=shape, dtype=np.uint64)
    bits = np.where(is_sub, neg | submf, bits)
    if sc["inf"] is not None:
        bits = np.where(is_inf, neg | np.uint64(sc["inf"]), bits)
    bits = np.where(is_nan, np.uint64(sc["nan"]), bits)
    return bits.astype(dt)


def gen_block_fma_set(fmt: str, n: int, k: int, seed: int, enc: str = "ocp",
                      special_rate: float = 0.01):
    """One randomized-validation vector set: a, b [n][k] in `fmt`, c [n] fp32 (int32 for
    integer formats), all by independent bit sampling with injected specials."""
    rng = np.random.default_rng(seed)
    a = independent_bits(rng, fmt, (n, k), enc, special_rate)
    b = independent_bits(rng, fmt, (n, k), enc, special_rate)
    if fmt in ("int8", "uint8"):
        c = rng.integers(0, 1 << 32, size=n, dtype=np.uint64).astype(np.uint32)
    else:
        c = independent_bits(rng, "fp32", (n,), "ocp", special_rate)
    return a, b, c


def algorithm3_rng(seed: int = 0):
    """The Mersenne Twister (MT19937) stream of Algorithm 3 ("mt19937 rng(0)")."""
    return np.random.Generator(np.random.MT19937(seed))


def gen_exp_mantissa(fmt: str, n: int, k: int, e_ab: tuple, e_c: tuple, seed: int = 0,
                     enc: str = "ocp", rng=None):
    """Exponent-mantissa sampling (Sec. 5.1, Algorithm 3): significand ~ U(-2+2^(1-f),
    2-2^(1-f)), exponent ~ U{e-, ..., e+}; the value is rounded to the format (RNE).
    A Mersenne Twister (MT19937) seeded with `seed` drives the draws; pass `rng` (from
    algorithm3_rng) instead to draw a large ensemble in consecutive chunks of one stream."""
    if rng is None:
        rng = algorithm3_rng(seed)
    dt, e, m, bias = fmt_params(fmt if fmt != "xf32" else "fp32", enc)
    f = m + 1 if fmt != "xf32" else 11

    def draw(shape, lo, hi, prec):
        s = rng.uniform(-2 + 2.0 ** (1 - prec), 2 - 2.0 ** (1 - prec), size=shape)
        ex = rng.integers(lo, hi + 1, size=shape)
        return s * np.exp2(ex.astype(np.float64))

    av = draw((n, k), e_ab[0], e_ab[1], f)
    bv = draw((n, k), e_ab[0], e_ab[1], f)
    cv = draw((n,), e_c[0], e_c[1], 24)
    if fmt == "bf16":
        a = fp32_to_bf16_rne(av.astype(np.float32))     # binary64 -> fp32 -> bf16
        b = fp32_to_bf16_rne(bv.astype(np.float32))
    elif fmt in ("fp32", "xf32"):
        a = av.astype(np.float32).view(np.uint32)
        b = bv.astype(np.float32).view(np.uint32)
    elif fmt == "fp16":
        a = av.astype(np.float16).view(np.uint16)
        b = bv.astype(np.float16).view(np.uint16)
    else:
        a = nearest_even(av, fmt, enc)
        b = nearest_even(bv, fmt, enc)
    c = cv.astype(np.float32).view(np.uint32)
    return a, b, c


# ---------------------------------------------------------------------------
# GEMM operands
# ---------------------------------------------------------------------------
def gen_dense_bf16(M: int, N: int, K: int, seed: int = 3):
    """A [M][K], Bt [N][K] = RNE_bf16(N(0,1)); C [M][N] = N(0,1) in fp32."""
    rng = np.random.default_rng(seed)
    A = fp32_to_bf16_rne(rng.standard_normal((M, K), dtype=np.float32))
    Bt = fp32_to_bf16_rne(rng.standard_normal((N, K), dtype=np.float32))
    C = rng.standard_normal((M, N), dtype=np.float32).view(np.uint32)
    return A, Bt, C


def gen_sparse_e4m3(M: int, N: int, K: int, seed: int = 4, c_zero: bool = True):
    """Dense A [M][K] E4M3 (OCP) with exactly two nonzeros in each group of four along K,
    at one of the six position pairs chosen uniformly; values RNE_e4m3(x*448/max|x|) of
    x ~ N(0,1), redrawn when they round to zero.  Bt [N][K] the same scaled N(0,1).
    C = 0 (or N(0,1) fp32 when c_zero is False)."""
    rng = np.random.default_rng(seed)
    pairs = np.array([(0, 1), (0, 2), (0, 3), (1, 2), (1, 3), (2, 3)])

    def scaled(shape):
        x = rng.standard_normal(shape)
        x = x * (448.0 / np.max(np.abs(x)))
        q = nearest_even(x, "e4m3")
        bad = (q & 0x7F) == 0
        while bad.any():
            y = rng.standard_normal(int(bad.sum())) * (448.0 / np.max(np.abs(x)))
            q[bad] = nearest_even(y, "e4m3")
            bad = (q & 0x7F) == 0
        return q

    groups = K // 4
    vals = scaled((M, groups, 2))
    sel = pairs[rng.integers(0, 6, size=(M, groups))]          # [M][groups][2]
    A = np.zeros((M, groups, 4), dtype=np.uint8)
    np.put_along_axis(A, sel, vals, axis=2)
    A = A.reshape(M, K)
    Bt = nearest_even(rng.standard_normal((N, K)) * (448.0 / 5.5), "e4m3")
    if c_zero:
        C = np.zeros((M, N), dtype=np.uint32)
    else:
        C = rng.standard_normal((M, N), dtype=np.float32).view(np.uint32)
    return A, Bt, C


def gen_multiword_fp64(M: int, N: int, K: int, seed: int = 5):
    """A [M][K], Bt [N][K] binary64 with entries N(0,1) * 2^u, u ~ U(-20, 20) continuous."""
    rng = np.random.default_rng(seed)

    def one(shape):
        return rng.standard_normal(shape) * np.exp2(rng.uniform(-20.0, 20.0, size=shape))

    return one((M, K)), one((N, K))


def gen_subnormal_boundary(fmt: str, n: int, k: int, seed: int):
    """Vector sets whose exact sum lies within a few units of 2^-150 of +-2^-126, the
    boundary between the largest fp32 subnormal and the smallest normal: at, just
    above and just below the subnormal ties 2^-126 - 2^-150 and 2^-126 + 2^-150 (half
    the subnormal spacing), with sticky products of either sign far below.  Formats
    whose products reach that far down: bf16, xf32, fp32 (k >= 2).

    Each set has a lead that sits on the boundary -- a product +-2^-126, an addend
    +-(2^-126 + r 2^-149), two products +-2^-125 -+ 2^-126 or two halves +-2^-127, or
    a subnormal addend just below 2^-126 -- then an offset product -+q 2^(t-152)
    (q < 64, |t| <= 2) and, for half of the sets, a product +-2^(-153-u).  Every
    product is realised as (q 2^x) * 2^y with both factors normal, the rest of the
    block holds zero products, and the products are shuffled within the block."""
    if fmt not in ("bf16", "xf32", "fp32") or k < 2:
        raise ValueError("bf16/xf32/fp32 operands and k >= 2")
    rng = np.random.default_rng(seed)
    dt = ELEM_DTYPE[fmt]
    cache = {}

    def code(q: int, x: int) -> int:
        key = (q, x)
        if key not in cache:
            cache[key] = encode_exact(Fraction(q) * Fraction(2) ** x, fmt)
        return cache[key]

    one = code(1, 0)
    a = np.zeros((n, k), dtype=np.uint64)
    b = np.full((n, k), one, dtype=np.uint64)
    c = np.zeros(n, dtype=np.uint64)
    for v in range(n):
        s = int(rng.integers(0, 2))                     # sign of the lead
        terms = []                                      # (negative, q, exponent)
        lead = int(rng.integers(0, 5 if k >= 3 else 4))
        cbits = None
        if lead == 0:
            terms.append((s, 1, -126))
        elif lead == 1:
            cbits = (s << 31) | (0x00800000 + int(rng.integers(0, 3)))
        elif lead == 2:
            cbits = (s << 31) | (0x00800000 - int(rng.integers(1, 4)))
        elif lead == 3:
            terms.append((s, 1, -127))
            cbits = (s << 31) | 0x00400000
        else:
            pair = int(rng.integers(0, 2))
            terms += [(s, 1, -125), (1 - s, 1, -126)] if pair == 0 else [(s, 1, -127), (s, 1, -127)]
        q = int(rng.integers(0, 64))
        if q and len(terms) < k:
            toward = 1 - s if rng.random() < 0.75 else s  # mostly down to the ties below
            terms.append((toward, q, int(rng.integers(-2, 3)) - 152))
        if rng.random() < 0.5 and len(terms) < k:
            terms.append((int(rng.integers(0, 2)), 1, -153 - int(rng.integers(0, 41))))
        if cbits is None:
            r = rng.random()
            cbits = 0 if r < 0.7 else (0x80000000 if r < 0.8 else
                                       (int(rng.integers(0, 2)) << 31) | int(rng.integers(1, 4)))
        pos = rng.permutation(k)[:len(terms)]
        for (neg, qq, x), p in zip(terms, pos):
            xa = x // 2                                 # q 2^xa times 2^(x - xa)
            a[v, p] = code(qq, xa) | (int(neg) << (8 * np.dtype(dt).itemsize - 1))
            b[v, p] = code(1, x - xa)
        c[v] = cbits
    return a.astype(dt), b.astype(dt), c.astype(np.uint32)

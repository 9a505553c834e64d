"""Pins of the CPU oracle against what the paper and the mathematics fix (no GPU).

- the feature vectors printed in "Accurate Models of AMD Matrix Cores" (tests/golden);
- the correctly rounded closed form (Python fractions) and libm fmaf;
- hand-traced cases of the early-c global-alignment reading, invariants, and the
  limits of Table 1.
"""
import ctypes
import ctypes.util
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle.presets import PRESETS, block_models
from bit_exact_emulation_gb300 import workloads as W
from bit_exact_emulation_gb300.workloads import encode_exact, parse_value
from _golden import encode_row, fp32_expect_bits, load_vectors
import exact_spec


def _run_row(row, spec):
    a, b, c = encode_row(row, spec.get("fp8_enc", "ocp"))
    dt = W.ELEM_DTYPE[row["fmt"]]
    if row["kt"] == 0:
        assert len(a) <= spec["n_fma"], row["id"]
        return int(oracle.block_fma(spec, np.array([a], dt), np.array([b], dt),
                                    np.array([c], np.uint32), n_terms=len(a))[0])
    K = len(a)
    return int(oracle.gemm_entries(spec, K, row["kt"], np.array([a], dt), np.array([b], dt),
                                   np.array([[c]], np.uint32), [0], [0])[0])


@pytest.mark.parametrize("fixture", ["cdna3_algorithm1.txt", "cdna1_exact.txt", "cdna3_algorithm2.txt",
                                     "cdna2_pairwise.txt"])
def test_paper_feature_vectors(fixture):
    rows = load_vectors(fixture)
    assert len(rows) > 30
    bad = []
    for row in rows:
        spec = PRESETS[row["preset"]]
        got = _run_row(row, spec)
        want = fp32_expect_bits(row["expect"], spec["nan_bits"])
        if got != want:
            bad.append(f"{row['id']}: got {got:#010x} want {want:#010x} ({row['cite']})")
    assert not bad, "\n".join(bad[:20])


def test_planted_mistake_is_caught():
    """The vectors separate the Algorithm 1 reading from nearby wrong ones: RD of c
    instead of truncation, or the 31-bit RD without normalisation, fail some row."""
    rows = load_vectors("cdna3_algorithm1.txt")
    for wrong in (dict(align_round="rd"), dict(psum_frac=31), dict(post_norm_frac=32),
                  dict(c_zero_exp=None), dict(align_frac=25), dict(prod_overflow=False)):
        fails = 0
        for row in rows:
            spec = dict(PRESETS[row["preset"]], **wrong)
            if _run_row(row, spec) != fp32_expect_bits(row["expect"], spec["nan_bits"]):
                fails += 1
        assert fails > 0, f"feature change {wrong} not detected by any vector"


# ---------------------------------------------------------------------------
# exact-then-round model = the closed form
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("fmt,k", [("fp16", 4), ("bf16", 4), ("xf32", 2), ("e4m3", 8), ("e5m2", 8),
                                   ("fp32", 1), ("bf16", 16)])
@pytest.mark.parametrize("mode", ["rne", "rtz"])
def test_exact_model_is_correctly_rounded_sum(fmt, k, mode):
    a, b, c = W.gen_block_fma_set(fmt, 1500, k, seed=11 + k, special_rate=0.02)
    spec = dict(block_models(fmt, k)["ieee_exact"], out_round=mode)
    d = oracle.block_fma(spec, a, b, c)
    for v in range(len(c)):
        want = exact_spec.exact_block(fmt, a[v], b[v], c[v], mode, nan_bits=spec["nan_bits"])
        assert d[v] == want, (fmt, v, a[v], b[v], hex(c[v]), hex(d[v]), hex(want))


def test_exact_model_bf16_extreme_spread():
    """Exponent-mantissa sampling over the whole bf16 range: sums that span > 500 bits."""
    a, b, c = W.gen_exp_mantissa("bf16", 2000, 4, (-133, 127), (-149, 127), seed=0)
    spec = block_models("bf16", 4)["ieee_exact"]
    d = oracle.block_fma(spec, a, b, c)
    for v in range(len(c)):
        assert d[v] == exact_spec.exact_block("bf16", a[v], b[v], c[v], nan_bits=spec["nan_bits"])



@pytest.mark.parametrize("fmt,k", [("bf16", 4), ("xf32", 2), ("bf16", 8)])
@pytest.mark.parametrize("mode", ["rne", "rtz"])
def test_exact_model_at_the_subnormal_boundary(fmt, k, mode):
    """Sums within a few 2^-150 of +-2^-126 (the ties of the subnormal grid next to the
    smallest normal, sticky bits of both signs): the exact model is the correctly
    rounded sum, rounded once onto the subnormal grid (IEEE 754 Sec. 4.3; "Accurate
    Models of AMD Matrix Cores", Sec. 4.1 keeps subnormals)."""
    a, b, c = W.gen_subnormal_boundary(fmt, 1500, k, seed=3 + k)
    spec = dict(block_models(fmt, k)["ieee_exact"], out_round=mode)
    d = oracle.block_fma(spec, a, b, c)
    for v in range(len(c)):
        want = exact_spec.exact_block(fmt, a[v], b[v], c[v], mode, nan_bits=spec["nan_bits"])
        assert d[v] == want, (fmt, v, a[v], b[v], hex(c[v]), hex(d[v]), hex(want))


def test_subnormal_tie_hand_traced():
    """a = (2^-63, -1.25 * 2^-75, 0, 0), b = (2^-63, 2^-75, 1, 1), c = +0 in bf16: the
    sum is 2^-126 - 1.25 * 2^-150, a quarter of a subnormal step below the tie at
    2^-126 - 2^-150.  Every term lies on the global-alignment grid 2^-152 (e_max = -126,
    F_p = 26), so truncation, RNE and the exact model all give the largest subnormal
    0x007FFFFF; rounding to 24 bits first would reach the tie and round up to 2^-126."""
    a = np.array([[0x2000, 0x9A20, 0, 0]], np.uint16)
    b = np.array([[0x2000, 0x1A00, 0x3F80, 0x3F80]], np.uint16)
    c = np.zeros(1, np.uint32)
    for name in ("ga_trunc", "ga_rne", "ieee_exact"):
        assert int(oracle.block_fma(block_models("bf16", 4)[name], a, b, c)[0]) == 0x007FFFFF, name
    # one unit of 2^-152 less below the tie rounds the other way under RNE only
    a2 = np.array([[0x2000, 0x9A00, 0, 0]], np.uint16)     # 2^-126 - 2^-150: the tie itself
    assert int(oracle.block_fma(block_models("bf16", 4)["ga_rne"], a2, b, c)[0]) == 0x00800000
    assert int(oracle.block_fma(block_models("bf16", 4)["ga_trunc"], a2, b, c)[0]) == 0x007FFFFF

@pytest.mark.parametrize("fmt", ["e5m2", "e4m3"])
def test_exact_fp8_exhaustive_pairs(fmt):
    """Every (a, b) pair of an 8-bit format, K = 1, against a set of addends."""
    codes = np.arange(256, dtype=np.uint8)
    a = np.repeat(codes, 256).reshape(-1, 1)
    b = np.tile(codes, 256).reshape(-1, 1)
    spec = block_models(fmt, 1)["ieee_exact"]
    for cval in ("0", "-0", "2^-149", "-1", "3*2^-30", "1.5*2^20"):
        cb = encode_exact(parse_value(cval), "fp32")
        c = np.full(a.shape[0], cb, np.uint32)
        d = oracle.block_fma(spec, a, b, c)
        for idx in range(0, a.shape[0], 7):          # every 7th pair, all 65536 on one addend
            want = exact_spec.exact_block(fmt, a[idx], b[idx], cb, nan_bits=spec["nan_bits"])
            assert d[idx] == want
        if cval == "-1":
            for idx in range(a.shape[0]):
                want = exact_spec.exact_block(fmt, a[idx], b[idx], cb, nan_bits=spec["nan_bits"])
                assert d[idx] == want


def _fmaf():
    lib = ctypes.CDLL(ctypes.util.find_library("m"))
    f = lib.fmaf
    f.argtypes = [ctypes.c_float] * 3
    f.restype = ctypes.c_float
    return f


def test_fp32_sfma_is_libm_fmaf():
    """CDNA 1 fp32 input is an SFMA (Sec. 4.1.1): K = 1 gives fmaf(a, b, c); a chain of
    two gives fmaf(a2, b2, fmaf(a1, b1, c))."""
    fmaf = _fmaf()
    rng = np.random.default_rng(5)
    n = 4000
    a = W.independent_bits(rng, "fp32", (n, 2), special_rate=0.01)
    b = W.independent_bits(rng, "fp32", (n, 2), special_rate=0.01)
    # move exponents toward the middle so that products mostly stay finite
    a = ((a & np.uint32(0x807FFFFF)) | ((((a >> 23) & 0xFF) // 2 + 64) << 23)).astype(np.uint32)
    c = W.independent_bits(rng, "fp32", (n,), special_rate=0.02)
    spec = PRESETS["cdna1_fp32"]
    af, bf, cf = a.view(np.float32), b.view(np.float32), c.view(np.float32)

    def bits(x):
        x = np.float32(x)
        return spec["nan_bits"] if np.isnan(x) else int(x.view(np.uint32))

    d1 = oracle.block_fma(spec, a[:, :1], b[:, :1], c)
    for v in range(n):
        assert d1[v] == bits(fmaf(af[v, 0], bf[v, 0], cf[v])), (v, hex(a[v, 0]), hex(b[v, 0]), hex(c[v]))
    for v in range(0, n, 4):
        got = oracle.gemm_entries(spec, 2, 2, a[v:v + 1], b[v:v + 1], c[v:v + 1].reshape(1, 1), [0], [0])[0]
        assert got == bits(fmaf(af[v, 1], bf[v, 1], fmaf(af[v, 0], bf[v, 0], cf[v])))


def test_fp16_single_product_is_rounded_binary64_product():
    """K = 1, c = +0: the product of two fp16 values is exact in binary64, so the correctly
    rounded result is numpy's binary64 -> binary32 conversion of it."""
    rng = np.random.default_rng(9)
    a = W.finite_fp16_bits(rng, (20000, 1))
    b = W.finite_fp16_bits(rng, (20000, 1))
    c = np.zeros(20000, np.uint32)
    d = oracle.block_fma(block_models("fp16", 1)["ieee_exact"], a, b, c)
    want = (a.view(np.float16).astype(np.float64) * b.view(np.float16).astype(np.float64)).astype(np.float32)
    want = want.reshape(-1).view(np.uint32)
    # +0 + (-0 product) = +0 under RNE
    want = np.where(want == 0x80000000, 0, want)
    assert np.array_equal(d, want)


# ---------------------------------------------------------------------------
# global alignment, early c (the randomized-workload models)
# ---------------------------------------------------------------------------
def _one(spec, fmt, prods, c):
    a = [encode_exact(parse_value(x), fmt) for x, _ in prods]
    b = [encode_exact(parse_value(y), fmt) for _, y in prods]
    dt = W.ELEM_DTYPE[fmt]
    return int(oracle.block_fma(spec, np.array([a], dt), np.array([b], dt),
                                np.array([encode_exact(parse_value(c), "fp32")], np.uint32),
                                n_terms=len(a))[0])


def test_ga_early_hand_traced():
    """Cases traced by hand through the early-c reading of Table 3 with F_p = 23 + 3."""
    m = block_models("fp16", 4)
    # 1 + 2^-24 + 1.5*2^-28: the 2^-28 term is cut on the 2^-26 grid -> 1 + 2^-24, a tie
    p = [("1", "1"), ("2^-12", "2^-12"), ("1.5*2^-14", "2^-14"), ("0", "1")]
    assert _one(m["ga_trunc"], "fp16", p, "0") == 0x3F800000
    assert _one(m["ga_rne"], "fp16", p, "0") == 0x3F800000
    assert _one(m["ieee_exact"], "fp16", p, "0") == 0x3F800001
    # cancellation: (1+2^-10) - 1 + 2^-30 (subnormal inputs, E = -14 each)
    p = [("1+2^-10", "1"), ("-1", "1"), ("2^-15", "2^-15"), ("0", "1")]
    assert _one(m["ga_trunc"], "fp16", p, "0") == 0x3A800000
    assert _one(m["ga_rne"], "fp16", p, "0") == 0x3A800000
    assert _one(m["ieee_exact"], "fp16", p, "0") == 0x3A800008
    # c joins the alignment: c = 1 and p = 2^-27 -> cut; with RD a negative p takes 2^-26
    p = [("-2^-14", "2^-13"), ("0", "1"), ("0", "1"), ("0", "1")]
    assert _one(m["ga_trunc"], "fp16", p, "1") == 0x3F800000
    assert _one(dict(m["ga_trunc"], align_round="rd"), "fp16", p, "1") == 0x3F7FFFFF
    # RTZ vs RNE of the integer sum: 1 + 2^-24 + 2^-25 (both kept on the 2^-26 grid)
    p = [("1", "1"), ("2^-12", "2^-12"), ("2^-12", "2^-13"), ("0", "1")]
    assert _one(m["ga_trunc"], "fp16", p, "0") == 0x3F800000
    assert _one(m["ga_rne"], "fp16", p, "0") == 0x3F800001
    # c = 0 is discarded (e_{c=0} = -inf); giving it an exponent above the products cuts them
    mb = block_models("bf16", 2)
    p = [("2^-50", "2^-50"), ("2^-65", "2^-65")]
    assert _one(mb["ga_trunc"], "bf16", p, "0") == encode_exact(parse_value("2^-100"), "fp32")
    assert _one(dict(mb["ga_trunc"], emin_lim=-133), "bf16", p, "0") == encode_exact(parse_value("2^-100"), "fp32")
    assert _one(dict(mb["ga_trunc"], c_zero_exp=-60), "bf16", p, "0") == 0
    # overflow of the final sum: RTZ saturates at the largest finite value, RNE gives Inf
    p = [("2^100", "2^27"), ("2^100", "2^27")]
    assert _one(mb["ga_trunc"], "bf16", p, "0") == 0x7F7FFFFF
    assert _one(mb["ga_rne"], "bf16", p, "0") == 0x7F800000


@pytest.mark.parametrize("fmt,k", [("fp16", 4), ("bf16", 4), ("e5m2", 8)])
@pytest.mark.parametrize("mode", ["rtz", "rne"])
def test_ga_early_wide_alignment_equals_exact(fmt, k, mode):
    """With F_p wider than any exponent spread of the inputs, truncation drops nothing
    and the early-c model is the correctly rounded sum."""
    rng = np.random.default_rng(3)
    if fmt == "fp16":
        a, b, c = W.gen_exp_mantissa("fp16", 1000, k, (-10, 10), (-30, 30), seed=4)
    elif fmt == "bf16":
        a, b, c = W.gen_exp_mantissa("bf16", 1000, k, (-40, 40), (-90, 90), seed=4)
    else:
        a = W.independent_bits(rng, fmt, (1000, k), special_rate=0.0)
        b = W.independent_bits(rng, fmt, (1000, k), special_rate=0.0)
        c = W.gen_exp_mantissa("bf16", 1000, 1, (0, 0), (-40, 40), seed=5)[2]
    base = block_models(fmt, k)["ga_trunc"]
    spec = dict(base, align_frac=200, out_round=mode)
    d = oracle.block_fma(spec, a, b, c)
    ex = oracle.block_fma(dict(block_models(fmt, k)["ieee_exact"], out_round=mode, nan_bits=base["nan_bits"]), a, b, c)
    assert np.array_equal(d, ex)


@pytest.mark.parametrize("name", ["ga_trunc", "ga_rne", "ieee_exact"])
def test_sign_symmetry_of_symmetric_models(name):
    """RZ/RTZ/RNE models are odd functions: d(-a, b, -c) = -d(a, b, c)."""
    a, b, c = W.gen_block_fma_set("bf16", 3000, 4, seed=21, special_rate=0.0)
    spec = block_models("bf16", 4)[name]
    d = oracle.block_fma(spec, a, b, c)
    dn = oracle.block_fma(spec, a ^ np.uint16(0x8000), b, c ^ np.uint32(0x80000000))
    nz = (d & 0x7FFFFFFF) != 0
    assert np.array_equal(dn[nz], d[nz] ^ np.uint32(0x80000000))


def test_algorithm1_is_not_sign_symmetric():
    """The RD steps of Algorithm 1 make it asymmetric (Sec. 4.3.1, c alignment)."""
    spec = PRESETS["cdna3_fp16"]
    pos = _one(spec, "fp16", [("1", "1")], "2^-24+2^-30")
    neg = _one(spec, "fp16", [("-1", "1")], "-(2^-24+2^-30)")
    assert pos == 0x3F800000 and neg == 0xBF800001


@pytest.mark.parametrize("preset", ["cdna3_fp16", "cdna3_bf16", "cdna1_fp16", "b200_fp16"])
def test_permutation_invariance_within_block(preset):
    spec = PRESETS[preset]
    k = min(spec["n_fma"], 8)
    spec = dict(spec, n_fma=k)
    fmt = spec["fmt_a"]
    a, b, c = W.gen_exp_mantissa(fmt, 400, k, (-12, 12) if fmt == "fp16" else (-60, 60), (-40, 40), seed=8)
    d = oracle.block_fma(spec, a, b, c)
    perm = np.random.default_rng(1).permutation(k)
    d2 = oracle.block_fma(spec, a[:, perm], b[:, perm], c)
    assert np.array_equal(d, d2)


@pytest.mark.parametrize("preset", ["cdna3_bf16", "b200_bf16", "cdna1_bf16"])
def test_power_of_two_scaling(preset):
    """Away from the range limits, scaling a and c by 2^s scales d by 2^s."""
    spec = PRESETS[preset]
    k = spec["n_fma"]
    a, b, c = W.gen_exp_mantissa("bf16", 500, k, (-20, 20), (-30, 30), seed=12)
    d = oracle.block_fma(spec, a, b, c)
    s = 7
    a2 = (a.astype(np.uint32) + np.uint32(s << 7)).astype(np.uint16)
    a2 = np.where((a & 0x7FFF) == 0, a, a2)
    c2 = np.where((c & 0x7FFFFFFF) == 0, c, c + np.uint32(s << 23)).astype(np.uint32)
    d2 = oracle.block_fma(spec, a2, b, c2)
    nz = (d & 0x7FFFFFFF) != 0
    assert np.array_equal(d2[nz], d[nz] + np.uint32(s << 23))


def test_pairwise_k1_is_ieee_fp32():
    """The pair-wise model with one product and no flushing is fl(c + fl(a * b)) in IEEE
    fp32 (Sec. 4.2): numpy's float32 arithmetic gives the same bits, including products
    that overflow to an infinity and then meet an infinite c."""
    rng = np.random.default_rng(8)
    n = 20000
    a = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
    b = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
    c = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
    c[::7] = np.where(rng.random(len(c[::7])) < 0.5, 0x7F800000, 0xFF800000)
    spec = dict(fmt_a="fp32", fmt_b="fp32", arch="pairwise", n_fma=1, pair_group=1, nan_bits=0x7FC00000)
    got = oracle.block_fma(spec, a.reshape(n, 1), b.reshape(n, 1), c)
    with np.errstate(all="ignore"):
        ref = (c.view(np.float32) + a.view(np.float32) * b.view(np.float32)).astype(np.float32)
    want = np.where(np.isnan(ref), np.uint32(0x7FC00000), ref.view(np.uint32))
    assert np.array_equal(got, want)


def test_int8_is_integer_dot_product():
    rng = np.random.default_rng(2)
    for fa, fb in (("int8", "int8"), ("uint8", "uint8")):
        a = rng.integers(0, 256, (3000, 16), dtype=np.uint64).astype(np.uint8)
        b = rng.integers(0, 256, (3000, 16), dtype=np.uint64).astype(np.uint8)
        c = rng.integers(0, 1 << 32, 3000, dtype=np.uint64).astype(np.uint32)
        spec = dict(fmt_a=fa, fmt_b=fb, arch="exact", n_fma=16)
        d = oracle.block_fma(spec, a, b, c)
        av = a.view(np.int8).astype(np.int64) if fa == "int8" else a.astype(np.int64)
        bv = b.view(np.int8).astype(np.int64) if fb == "int8" else b.astype(np.int64)
        want = ((av * bv).sum(1) + c.view(np.int32).astype(np.int64)) & 0xFFFFFFFF
        assert np.array_equal(d, want.astype(np.uint32))
        sat = oracle.block_fma(dict(spec, int_saturate=True), a, b, c)
        full = (av * bv).sum(1) + c.view(np.int32).astype(np.int64)
        assert np.array_equal(sat.view(np.int32), np.clip(full, -2 ** 31, 2 ** 31 - 1).astype(np.int32))


# ---------------------------------------------------------------------------
# Table 1 limits through the decoder (K = 1, b = 1, c = 0, exact model)
# ---------------------------------------------------------------------------
TABLE1 = [  # format, encoding, max finite, min normal (Table 1)
    ("fp16", "ocp", "65504", "2^-14"),
    ("bf16", "ocp", "(2-2^-7)*2^127", "2^-126"),
    ("e4m3", "fnuz", "240", "2^-7"),
    ("e4m3", "ocp", "448", "2^-6"),
    ("e5m2", "fnuz", "57344", "2^-15"),
    ("e5m2", "ocp", "57344", "2^-14"),
]


@pytest.mark.parametrize("fmt,enc,mx,mn", TABLE1)
def test_table1_extrema(fmt, enc, mx, mn):
    dt, e, m, bias = W.fmt_params(fmt, enc)
    spec = dict(fmt_a=fmt, fmt_b=fmt, fp8_enc=enc, arch="exact", n_fma=1)
    codes = np.arange(1 << (e + m), dtype=np.uint32).astype(dt).reshape(-1, 1)
    one = np.full_like(codes, encode_exact(1, fmt, enc))
    d = oracle.block_fma(spec, codes, one, np.zeros(codes.shape[0], np.uint32))
    vals = d.view(np.float32)
    finite = np.isfinite(vals)
    assert vals[finite].max() == float(parse_value(mx))
    normal_min = min(v for v in vals[finite] if v > 0 and (np.float32(v).view(np.uint32) >> 23) > 0
                     and v >= float(parse_value(mn)))
    assert normal_min == float(parse_value(mn))
    # the next value below the minimum normal is a subnormal of the format
    assert (vals[finite & (vals > 0)] < float(parse_value(mn))).any()


def test_tf19_max_is_truncated_fp32_max():
    spec = dict(fmt_a="xf32", fmt_b="xf32", arch="exact", n_fma=1)
    d = oracle.block_fma(spec, np.array([[0x7F7FFFFF]], np.uint32),
                         np.array([[0x3F800000]], np.uint32), np.zeros(1, np.uint32))
    assert d[0] == encode_exact(parse_value("(2-2^-10)*2^127"), "fp32")


# ---------------------------------------------------------------------------
# Bayesian mismatch bound of Sec. 5.4 (m = 0 rows of Table 2)
# ---------------------------------------------------------------------------
def test_table2_bounds():
    from math import expm1, log
    eps = 1e-6
    for n, printed in ((1e5, 1.38e-4), (1e6, 1.38e-5), (1e7, 1.38e-6), (2e6, 6.91e-6), (2e7, 6.91e-7)):
        p = -expm1(log(eps) / (n + 1))
        assert abs(p - printed) / printed < 0.005


def test_table2_bounds_of_the_harness():
    """The validation harness's p_eps: Table 2's m = 0 rows, and for m = 1 the (1 - eps)
    quantile of the Beta(2, N) posterior of Sec. 5.4 (1.669e-5 at N = 10^6; the printed
    1.69e-5 and 1.35e-5 for N = 1.25 * 10^6 are that quantile rounded up)."""
    pytest.importorskip("scipy")
    import validate_algorithm3 as V
    for n, printed in ((10**6, 1.38e-5), (10**7, 1.38e-6), (2 * 10**7, 6.91e-7), (2 * 10**6, 6.91e-6)):
        assert abs(V.p_eps(n, 0) - printed) / printed < 0.005
    # m = 1: solve (N + 1) N \int_0^p t (1 - t)^(N - 1) dt = 1 - eps by bisection, independently of scipy
    from math import exp, log1p
    for n, want in ((10**6, 1.669e-5), (1_250_000, 1.335e-5)):
        def cdf(p):   # regularized incomplete beta I_p(2, N) = 1 - (1 - p)^N (1 + N p)
            return 1.0 - exp(n * log1p(-p)) * (1.0 + n * p)
        lo, hi = 0.0, 1e-3
        for _ in range(200):
            mid = (lo + hi) / 2
            lo, hi = (mid, hi) if cdf(mid) < 1 - 1e-6 else (lo, mid)
        assert abs(V.p_eps(n, 1) - lo) / lo < 1e-6
        assert abs(lo - want) / want < 0.002


def test_harness_chain_is_the_instruction_chain():
    """The validation harness evaluates a k-element vector set as the chain of k / N_FMA
    block FMAs; that chain is the oracle's 1 x 1 x k tile GEMM with instruction K = k."""
    import validate_algorithm3 as V
    for preset, fmt, k in (("cdna3_fp16", "fp16", 16), ("cdna3_xf32", "xf32", 8)):
        spec = PRESETS[preset]
        a, b, c = W.gen_exp_mantissa(fmt, 200, k, (-14, 15) if fmt == "fp16" else (-126, 63), (-126, 127), seed=0)
        got = V._chain(lambda s, x, y, z: oracle.block_fma(s, x, y, z), spec, k, a, b, c)
        for v in range(0, 200, 7):
            want = oracle.gemm_entries(spec, k, k, a[v:v + 1], b[v:v + 1], c[v:v + 1].reshape(1, 1), [0], [0])[0]
            assert got[v] == want, (preset, v)


# ---------------------------------------------------------------------------
# fp16 output (Table 3's note: NVIDIA fp16 and fp8 inputs with fp16 c and d)
# ---------------------------------------------------------------------------
def test_round_fp16_is_numpy_binary16():
    """The closed-form binary16 rounding used below agrees with numpy's binary64 ->
    binary16 conversion (IEEE RNE) on values binary64 holds exactly, subnormals and
    overflow included."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal(20000) * np.exp2(rng.integers(-30, 18, 20000))
    x[:50] = [65504.0, 65519.99, 65520.0, 2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0001, 3 * 2.0 ** -26,
              -2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, 1e-9] + list(rng.standard_normal(40) * 2.0 ** -20)
    with np.errstate(over="ignore"):
        want16 = x.astype(np.float16).view(np.uint16)
    for v, want in zip(x, want16.tolist()):
        assert exact_spec.round_fp16(Fraction(float(v))) == want, v


@pytest.mark.parametrize("fmt,k", [("fp16", 4), ("fp16", 16), ("e4m3", 8), ("e5m2", 8)])
@pytest.mark.parametrize("mode", ["rne", "rtz"])
def test_fp16_output_exact_model_is_correctly_rounded(fmt, k, mode):
    a, b, _ = W.gen_block_fma_set(fmt, 1500, k, seed=40 + k, special_rate=0.02)
    c = W.independent_bits(np.random.default_rng(41), "fp16", (1500,), "ocp", 0.02).astype(np.uint32)
    spec = dict(fmt_a=fmt, fmt_b=fmt, arch="exact", n_fma=k, out_round=mode, acc_fmt="fp16", nan_bits=0x7E00)
    d = oracle.block_fma(spec, a, b, c)
    for v in range(len(c)):
        want = exact_spec.exact_block(fmt, a[v], b[v], c[v], mode, nan_bits=0x7E00, acc="fp16")
        assert d[v] == want, (fmt, v, a[v], b[v], hex(c[v]), hex(d[v]), hex(want))


def test_fp16_output_wide_alignment_equals_exact_rtz():
    """Early-c global alignment keeping more fraction bits than the exponent spread of
    the terms is the exact sum rounded toward zero to binary16."""
    a, b, _ = W.gen_exp_mantissa("fp16", 3000, 8, (-6, 6), (-14, 15), seed=0)
    c = W.gen_exp_mantissa("fp16", 3000, 1, (-8, 8), (-14, 15), seed=1)[0].reshape(-1).astype(np.uint32)
    spec = dict(PRESETS["b200_fp16_f16"], n_fma=8, align_frac=60, emin_lim=None)
    d = oracle.block_fma(spec, a, b, c)
    for v in range(len(c)):
        assert d[v] == exact_spec.exact_block("fp16", a[v], b[v], c[v], "rtz", nan_bits=0x7E00, acc="fp16"), v


def test_fp16_output_hand_traced():
    """B200 fp16-output model (F_p = 25, e_min^lim = -21, RTZ, c = 0 discarded):
      p1 = 2^-12 * 2^-12 = 2^-24 (e = -24), p2 = -2^-23 * 2^-24 = -2^-47 (e = -28).
      e_max = max(-24, -28, -21) = -21, grid 2^-46: p2 truncates to 0, the sum is 2^-24,
      the smallest binary16 subnormal (0x0001).  Without the limit e_max = -24, the grid
      2^-49 keeps p2, and 2^-24 - 2^-47 rounds toward zero to 0; so does the exact sum.
    Overflow: 65504 * 2 gives 0x7BFF (RTZ) and 0x7C00 (RNE); an Inf operand gives
    0x7C00; Inf - Inf the binary16 NaN."""
    spec = PRESETS["b200_fp16_f16"]
    e16 = lambda x: encode_exact(parse_value(x), "fp16")
    k = spec["n_fma"]

    def run(s, av, bv, cbits=0):
        a = np.array([[e16(x) for x in av] + [0] * (k - len(av))], np.uint16)
        b = np.array([[e16(x) for x in bv] + [0] * (k - len(bv))], np.uint16)
        return int(oracle.block_fma(s, a, b, np.array([cbits], np.uint32))[0])

    assert run(spec, ["2^-12", "-2^-23"], ["2^-12", "2^-24"]) == 0x0001
    assert run(dict(spec, emin_lim=None), ["2^-12", "-2^-23"], ["2^-12", "2^-24"]) == 0x0000
    assert run(dict(spec, arch="exact"), ["2^-12", "-2^-23"], ["2^-12", "2^-24"]) == 0x0000
    assert run(spec, ["65504"], ["2"]) == 0x7BFF
    assert run(dict(spec, out_round="rne"), ["65504"], ["2"]) == 0x7C00
    assert run(spec, ["inf"], ["2"]) == 0x7C00
    assert run(spec, ["inf", "-inf"], ["1", "1"]) == 0x7E00
    assert run(spec, ["1"], ["1"], e16("-1")) == 0x0000            # exact cancellation: +0
    k = 1
    assert run(dict(spec, n_fma=1), ["-0"], ["1"], 0x8000) == 0x8000   # -0 * 1 + -0
    assert run(dict(spec, n_fma=1), ["-0"], ["1"], 0x0000) == 0x0000   # -0 * 1 + +0


def test_fp16_output_chain_carries_binary16():
    """A GEMM chain with the fp16 accumulator: each block's binary16 result is the next
    block's addend (oracle GEMM = repeated block FMAs)."""
    spec = PRESETS["a100_fp16_f16"]
    a, b, _ = W.gen_exp_mantissa("fp16", 60, 32, (-8, 8), (-14, 15), seed=2)
    c = W.gen_exp_mantissa("fp16", 60, 1, (-4, 4), (-14, 15), seed=3)[0].reshape(-1).astype(np.uint32)
    d = c.copy()
    for j in range(0, 32, spec["n_fma"]):
        d = oracle.block_fma(spec, np.ascontiguousarray(a[:, j:j + 8]), np.ascontiguousarray(b[:, j:j + 8]), d)
    for v in range(60):
        want = oracle.gemm_entries(spec, 32, 16, a[v:v + 1], b[v:v + 1], c[v:v + 1].reshape(1, 1), [0], [0])[0]
        assert want == d[v] and d[v] <= 0xFFFF

"""Block-FMA stream on the GPU, bit for bit against the oracle (and the paper's
printed outputs), through the C ABI."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle.presets import PRESETS, block_models
from bit_exact_emulation_gb300 import workloads as W
from _golden import encode_row, fp32_expect_bits, load_vectors

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_exact_emulation_gb300 import build
    build.build()
    from bit_exact_emulation_gb300 import binding
    return binding


def dev(x):
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        x = x.view(np.int16)
    elif x.dtype == np.uint32:
        x = x.view(np.int32)
    return torch.from_numpy(x).cuda()


def gpu_block(L, spec, a, b, c):
    m = L.Model(spec)
    d = L.block_fma(m, dev(a), dev(b), dev(c))
    return d.cpu().numpy().view(np.uint32)


def gpu_chain(L, spec, kt, a, b, c):
    """1 x 1 x K GEMM: the chained block FMAs of one output."""
    m = L.Model(spec)
    t = L.tile(0, 16, 16, kt, 4)
    D = L.tile_gemm(m, t, dev(a), dev(b), dev(np.asarray(c, np.uint32).reshape(1, 1)))
    return int(D.cpu().numpy().view(np.uint32)[0, 0])


def mismatches(got, want, a=None, b=None, c=None, limit=8):
    bad = np.nonzero(got != want)[0]
    msg = [f"{len(bad)} of {len(want)} differ"]
    for v in bad[:limit]:
        extra = f" a={a[v]} b={b[v]} c={c[v]:#010x}" if a is not None else ""
        msg.append(f"  [{v}] gpu {got[v]:#010x} oracle {want[v]:#010x}{extra}")
    return "\n".join(msg)


# ---------------------------------------------------------------------------
# the paper's feature vectors
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("fixture", ["cdna3_algorithm1.txt", "cdna1_exact.txt", "cdna3_algorithm2.txt",
                                     "cdna2_pairwise.txt"])
def test_paper_vectors_gpu(L, fixture):
    bad = []
    for row in load_vectors(fixture):
        spec = PRESETS[row["preset"]]
        a, b, c = encode_row(row, spec.get("fp8_enc", "ocp"))
        dt = W.ELEM_DTYPE[row["fmt"]]
        want = fp32_expect_bits(row["expect"], spec["nan_bits"])
        n = len(a)
        kt = row["kt"] if row["kt"] else spec["n_fma"]
        got_chain = gpu_chain(L, spec, kt, np.array([a], dt), np.array([b], dt), c)
        if got_chain != want:
            bad.append(f"{row['id']} (chain): gpu {got_chain:#010x} printed {want:#010x}")
        if row["kt"] == 0:
            # stream path: pad the vector with zero products (0 * 1) to the block size
            k = spec["n_fma"]
            one = W.encode_exact(1, row["fmt"], spec.get("fp8_enc", "ocp"))
            ap = np.array([a + [0] * (k - n)], dt)
            bp = np.array([b + [one] * (k - n)], dt)
            got = int(gpu_block(L, spec, ap, bp, np.array([c], np.uint32))[0])
            ref = int(oracle.block_fma(spec, ap, bp, np.array([c], np.uint32))[0])
            if got != ref:
                bad.append(f"{row['id']} (stream): gpu {got:#010x} oracle {ref:#010x}")
    assert not bad, "\n".join(bad[:20])


# ---------------------------------------------------------------------------
# randomized vector sets (the validation workloads)
# ---------------------------------------------------------------------------
def test_fp16_cancellation_set_all_models(L):
    """65,536 FP16 K=4 vector sets (half of them with clustered exponents), FP32 c."""
    a, b, c = W.gen_fp16_cancellation(65536, 4, seed=1)
    for name, spec in block_models("fp16", 4).items():
        got = gpu_block(L, spec, a, b, c)
        want = oracle.block_fma_parallel(spec, a, b, c, threads=8)
        assert np.array_equal(got, want), name + "\n" + mismatches(got, want, a, b, c)


FORMAT_SETS = [("fp16", 4, "ocp"), ("bf16", 4, "ocp"), ("xf32", 2, "ocp"), ("e4m3", 8, "ocp"),
               ("e5m2", 8, "ocp"), ("int8", 16, "ocp")]


@pytest.mark.parametrize("fmt,k,enc", FORMAT_SETS)
def test_independent_bits_with_specials(L, fmt, k, enc):
    """Independent bit sampling with 1% each of zeros, subnormals, Inf and NaN."""
    a, b, c = W.gen_block_fma_set(fmt, 40000, k, seed=2 + k, enc=enc)
    for name, spec in block_models(fmt, k).items():
        spec = dict(spec, fp8_enc=enc)
        got = gpu_block(L, spec, a, b, c)
        want = oracle.block_fma_parallel(spec, a, b, c, threads=8)
        assert np.array_equal(got, want), f"{fmt} {name}\n" + mismatches(got, want, a, b, c)


@pytest.mark.parametrize("fmt,k,enc", FORMAT_SETS)
def test_full_size_sampled(L, fmt, k, enc):
    """10^7 vector sets per format on the GPU; a seeded sample is recomputed by the oracle."""
    n = 10_000_000
    a, b, c = W.gen_block_fma_set(fmt, n, k, seed=2 + k, enc=enc)
    idx = np.random.default_rng(7).choice(n, 3000, replace=False)
    for name, spec in block_models(fmt, k).items():
        got = gpu_block(L, spec, a, b, c)[idx]
        want = oracle.block_fma_parallel(spec, a[idx], b[idx], c[idx], threads=8)
        assert np.array_equal(got, want), f"{fmt} {name}\n" + mismatches(got, want)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("enc", ["ocp", "fnuz"])
@pytest.mark.parametrize("k", [8, 16, 32])
def test_fp8_table_kernel_encodings_and_block_sizes(L, fmt, enc, k):
    """The FP8 product-table kernel for both encodings and the block sizes it serves,
    global alignment (truncate, RNE) and exact-then-round, specials included."""
    a, b, c = W.gen_block_fma_set(fmt, 30000, k, seed=50 + k, enc=enc, special_rate=0.01)
    for name, spec in block_models(fmt, k).items():
        spec = dict(spec, fp8_enc=enc)
        got = gpu_block(L, spec, a, b, c)
        want = oracle.block_fma_parallel(spec, a, b, c, threads=8)
        assert np.array_equal(got, want), f"{fmt} {enc} k={k} {name}\n" + mismatches(got, want)


# exponent-mantissa sampling (Algorithm 3, seed 0) at the exponent limits of Sec. 5.1
CDNA3_SAMPLING = [
    ("cdna3_fp16", "fp16", (-14, 15), (-126, 127)), ("cdna3_fp16", "fp16", (-24, -14), (-149, -126)),
    ("cdna3_bf16", "bf16", (-126, 63), (-126, 127)), ("cdna3_bf16", "bf16", (-133, -126), (-149, -126)),
    ("cdna3_xf32", "xf32", (-126, 63), (-126, 127)), ("cdna3_xf32", "xf32", (-136, -126), (-149, -126)),
    ("cdna3_fp8", "e4m3", (-7, 7), (-126, 127)), ("cdna3_fp8", "e4m3", (-10, -7), (-149, -126)),
    ("cdna3_bf8", "e5m2", (-15, 15), (-126, 127)), ("cdna3_bf8", "e5m2", (-17, -15), (-149, -126)),
]


@pytest.mark.parametrize("preset,fmt,eab,ec", CDNA3_SAMPLING)
def test_cdna3_exponent_mantissa_sampling(L, preset, fmt, eab, ec):
    spec = PRESETS[preset]
    a, b, c = W.gen_exp_mantissa(fmt, 60000, spec["n_fma"], eab, ec, seed=0,
                                 enc=spec.get("fp8_enc", "ocp"))
    got = gpu_block(L, spec, a, b, c)
    want = oracle.block_fma_parallel(spec, a, b, c, threads=8)
    assert np.array_equal(got, want), preset + "\n" + mismatches(got, want, a, b, c)


def _cancellation_set(fmt, n, seed):
    """K=4 vector sets built to stress exact-then-round: c nearly cancels the first
    product, the other products sit 10-40 and 50-110 binades lower, so the sum keeps
    few bits above the far terms and sticky information decides the rounding."""
    rng = np.random.default_rng(seed)
    to_bits = {"bf16": lambda x: W.fp32_to_bf16_rne(x.astype(np.float32)),
               "fp16": lambda x: x.astype(np.float16).view(np.uint16),
               "xf32": lambda x: (x.astype(np.float32).view(np.uint32) & np.uint32(0xFFFFE000))}[fmt]
    lo = {"bf16": (-60, -110), "fp16": (-10, -22), "xf32": (-60, -110)}[fmt]

    def vals(e_lo, e_hi, size):
        return rng.uniform(1, 2, size) * np.exp2(rng.integers(e_lo, e_hi + 1, size)) * rng.choice([-1, 1], size)

    a = np.empty((n, 4), dtype=W.ELEM_DTYPE[fmt])
    b = np.empty((n, 4), dtype=W.ELEM_DTYPE[fmt])
    a[:, 0], b[:, 0] = to_bits(vals(0, 0, n)), to_bits(vals(0, 0, n))
    half = 5 if fmt == "fp16" else 20
    a[:, 1], b[:, 1] = to_bits(vals(-half, -3, n)), to_bits(vals(-half, -3, n))
    a[:, 2], b[:, 2] = to_bits(vals(lo[1] // 2, lo[0] // 2, n)), to_bits(vals(lo[1] // 2, lo[0] // 2, n))
    a[:, 3], b[:, 3] = to_bits(vals(-half, -2, n)), to_bits(vals(-half, -2, n))
    a[n // 2:, 3] = 0                                   # half of them without the fourth product
    # c: minus the first product rounded to fp32, moved by a few units in the last place
    if fmt == "bf16":
        fa = (a[:, 0].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        fb = (b[:, 0].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    elif fmt == "fp16":
        fa, fb = a[:, 0].view(np.float16).astype(np.float64), b[:, 0].view(np.float16).astype(np.float64)
    else:
        fa, fb = a[:, 0].view(np.float32).astype(np.float64), b[:, 0].view(np.float32).astype(np.float64)
    c = (-(fa * fb)).astype(np.float32).view(np.int32) + rng.integers(-3, 4, n).astype(np.int32)
    return a, b, c.view(np.uint32)


@pytest.mark.parametrize("fmt", ["bf16", "fp16", "xf32"])
def test_exact_cancellation_and_sticky(L, fmt):
    a, b, c = _cancellation_set(fmt, 100000, seed=17)
    for name in ("ieee_exact", "ga_rne", "ga_trunc"):
        spec = block_models(fmt, 4)[name] if fmt != "xf32" else dict(block_models("xf32", 2)[name], n_fma=4)
        got = gpu_block(L, spec, a, b, c)
        want = oracle.block_fma_parallel(spec, a, b, c, threads=8)
        assert np.array_equal(got, want), f"{fmt} {name}\n" + mismatches(got, want, a, b, c)


def _midpoint_sets(fmt, k, n, seed):
    """Vector sets whose exact sum sits on, just above or just below a rounding
    boundary of c: one product is +-1/2 or +-1 unit in the last place of c (a
    product of two powers of two), some others are tiny products of either sign
    (sticky bits), the rest zero."""
    rng = np.random.default_rng(seed)
    _, e, m, bias = W.fmt_params(fmt)
    emin = 1 - bias - m                                  # smallest subnormal exponent
    emax = (1 << e) - 2 - bias if fmt != "e4m3" else 8
    p2 = {x: W.encode_exact(Fraction(2) ** x, fmt) for x in range(emin, emax + 1)}
    lo_c = max(2 * emin + 24, -120) + 2
    hi_c = min(2 * emax + 23, 120) - 2
    ec = rng.integers(lo_c, hi_c + 1, n)
    c = ((rng.integers(0, 2, n) << 31) | ((ec + 127) << 23) | rng.integers(0, 1 << 23, n)).astype(np.uint32)
    dt = W.ELEM_DTYPE[fmt]
    a = np.zeros((n, k), dtype=dt)
    b = np.zeros((n, k), dtype=dt)
    sgn = 1 << (8 * np.dtype(dt).itemsize - 1)
    for v in range(n):
        x = int(ec[v]) - 24 + int(rng.integers(0, 2))   # half an ulp of c, or a whole one
        xa = max(emin, min(emax, x // 2))
        xb = x - xa
        if not (emin <= xb <= emax):
            continue
        a[v, 0], b[v, 0] = p2[xa], p2[xb] | (sgn if rng.random() < 0.5 else 0)
        for l in range(1, k):
            r = rng.random()
            if r < 0.5:
                continue                                 # zero product
            ta = int(rng.integers(emin, emin + 4))
            tb = int(rng.integers(emin, emin + 4))
            a[v, l] = p2[ta] | (sgn if rng.random() < 0.5 else 0)
            b[v, l] = p2[tb]
    perm = np.argsort(rng.random((n, k)), axis=1)        # the first product anywhere in the set
    return np.take_along_axis(a, perm, 1), np.take_along_axis(b, perm, 1), c


@pytest.mark.parametrize("fmt,k", [("fp16", 4), ("bf16", 4), ("xf32", 2), ("e4m3", 8), ("e5m2", 8)])
@pytest.mark.parametrize("out_round", ["rne", "rtz"])
def test_exact_rounding_boundaries(L, fmt, k, out_round):
    """Exact-then-round with RNE and RTZ on sums at, just above and just below a
    rounding boundary (ties, sticky bits of either sign), and on independent bits."""
    spec = dict(block_models(fmt, k)["ieee_exact"], out_round=out_round)
    sets = [_midpoint_sets(fmt, k, 20000, seed=31), W.gen_block_fma_set(fmt, 40000, k, seed=32)]
    for a, b, c in sets:
        got = gpu_block(L, spec, a, b, c)
        want = oracle.block_fma_parallel(spec, a, b, c, threads=8)
        assert np.array_equal(got, want), f"{fmt} {out_round}\n" + mismatches(got, want, a, b, c)


BOUNDARY_MODELS = [  # format, block size, model
    ("bf16", 4, block_models("bf16", 4)["ga_rne"]), ("bf16", 4, block_models("bf16", 4)["ga_trunc"]),
    ("bf16", 4, block_models("bf16", 4)["ieee_exact"]),
    ("bf16", 4, dict(block_models("bf16", 4)["ieee_exact"], out_round="rtz")),
    ("xf32", 2, block_models("xf32", 2)["ga_rne"]), ("xf32", 2, block_models("xf32", 2)["ga_trunc"]),
    ("xf32", 2, block_models("xf32", 2)["ieee_exact"]),
    ("xf32", 2, dict(block_models("xf32", 2)["ieee_exact"], out_round="rtz")),
    ("bf16", 8, PRESETS["cdna3_bf16"]), ("xf32", 4, PRESETS["cdna3_xf32"]),
    ("bf16", 16, PRESETS["b200_bf16"]), ("xf32", 8, PRESETS["b200_tf19"]),
    ("bf16", 2, PRESETS["cdna1_bf16"]), ("fp32", 2, dict(PRESETS["cdna1_fp32"], n_fma=2)),
    ("bf16", 4, dict(block_models("bf16", 4)["ga_rne"], align_frac=40)),
    ("bf16", 5, dict(block_models("bf16", 4)["ga_rne"], n_fma=5)),
]


@pytest.mark.parametrize("case", range(len(BOUNDARY_MODELS)))
def test_subnormal_boundary(L, case):
    """Exact sums at, just above and just below the ties next to 2^-126 (largest subnormal
    / smallest normal), with sticky products of both signs: a result must be rounded
    once, onto the subnormal grid, never first to 24 bits and then again."""
    fmt, k, spec = BOUNDARY_MODELS[case]
    a, b, c = W.gen_subnormal_boundary(fmt, 20000, k, seed=70 + case)
    got = gpu_block(L, spec, a, b, c)
    want = oracle.block_fma_parallel(spec, a, b, c, threads=8)
    assert np.array_equal(got, want), f"{fmt} k={k}\n" + mismatches(got, want, a, b, c)
    if fmt == "bf16" and k == 4:
        # the hand-traced set 2^-126 - 1.25 * 2^-150: the largest subnormal under every model
        a1 = np.array([[0x2000, 0x9A20, 0, 0]], np.uint16)
        b1 = np.array([[0x2000, 0x1A00, 0x3F80, 0x3F80]], np.uint16)
        assert int(gpu_block(L, spec, a1, b1, np.zeros(1, np.uint32))[0]) == 0x007FFFFF

@pytest.mark.parametrize("fmt,k", [("bf16", 4), ("xf32", 2)])
@pytest.mark.parametrize("prod_overflow", [False, True])
def test_exact_wide_formats_product_overflow(L, fmt, k, prod_overflow):
    """Exact-then-round on BF16 and XF32 random bit patterns (products up to 2^+-266),
    with and without the CDNA 3 rule that makes a product of 2^128 or more an Inf."""
    a, b, c = W.gen_block_fma_set(fmt, 40000, k, seed=61)
    spec = dict(block_models(fmt, k)["ieee_exact"], prod_overflow=prod_overflow)
    for out_round in ("rne", "rtz"):
        s = dict(spec, out_round=out_round)
        got = gpu_block(L, s, a, b, c)
        want = oracle.block_fma_parallel(s, a, b, c, threads=8)
        assert np.array_equal(got, want), f"{fmt} {out_round} {prod_overflow}\n" + mismatches(got, want, a, b, c)


def _scale_extremes(fmt, n, k, seed):
    """Sets built from exponent fields at the ends of the range: a product of two
    largest binades with c anywhere; c in the largest binade with products 120-135
    binades below it (terms dropped or kept at the scale limit); a subnormal c with
    the smallest products (the scale of every term rises by up to 2^128); one product
    on top and the others 120-135 binades below; sums that round up to 2^128."""
    rng = np.random.default_rng(seed)
    mb = 7 if fmt == "bf16" else 23
    dt = np.uint16 if fmt == "bf16" else np.uint32

    def elem(field, size):
        field = np.clip(field, 0, 254)
        m = rng.integers(0, 1 << mb, size)
        if fmt == "xf32":
            m &= ~((1 << 13) - 1)
        s = rng.integers(0, 2, size)
        return ((s << (mb + 8)) | (field << mb) | m).astype(dt)

    fa = rng.integers(1, 255, (n, k))
    fb = rng.integers(1, 255, (n, k))
    fc = rng.integers(0, 255, n)
    mode = rng.integers(0, 5, n)
    top = mode == 0                                       # products in the top binades
    fa[top], fb[top] = rng.integers(250, 255, (2, top.sum(), k))
    big_c = mode == 1                                     # c on top, products far below
    fc[big_c] = rng.integers(250, 255, big_c.sum())
    gap = rng.integers(120, 136, (big_c.sum(), k))
    s = fc[big_c][:, None] + 127 - gap                    # the products' field sums
    fa[big_c] = np.clip(s // 2, 1, 254)
    fb[big_c] = np.clip(s - fa[big_c], 1, 254)
    sub_c = mode == 2                                     # subnormal c, tiny products
    fc[sub_c] = 0
    fa[sub_c], fb[sub_c] = rng.integers(0, 4, (2, sub_c.sum(), k))
    spread = mode == 3                                    # one product on top, the rest far below
    s = rng.integers(200, 400, spread.sum())[:, None] - np.concatenate(
        [np.zeros((spread.sum(), 1), np.int64), rng.integers(120, 136, (spread.sum(), k - 1))], 1)
    fa[spread] = np.clip(s // 2, 1, 254)
    fb[spread] = np.clip(s - fa[spread], 1, 254)
    fc[spread] = rng.integers(0, 100, spread.sum())
    a, b = elem(fa, (n, k)), elem(fb, (n, k))
    c = ((rng.integers(0, 2, n) << 31) | (fc << 23) | rng.integers(0, 1 << 23, n)).astype(np.uint32)
    ovf = np.flatnonzero(mode == 4)                       # c = +-max finite plus a product near its ulp
    c[ovf] = (c[ovf] & 0x80000000) | 0x7F7FFFFF
    a[ovf], b[ovf] = elem(rng.integers(120, 128, (ovf.size, k)), (ovf.size, k)), elem(
        rng.integers(230, 250, (ovf.size, k)), (ovf.size, k))
    cancel = np.flatnonzero(top & (rng.random(n) < 0.5))  # the top product cancelled exactly
    for l in range(0, k, 2):
        a[cancel, l + 1] = a[cancel, l]
        b[cancel, l + 1] = b[cancel, l] ^ dt(1 << (mb + 8))
    b[cancel, k - 1] ^= dt(rng.integers(0, 2) << 4)      # one pair left slightly off
    return a, b, c


def _special_mix(fmt, n, k, seed):
    """Elements drawn from +-Inf, NaN, +-0, the largest and smallest binades and
    random bits (an Inf next to a tiny element while other products are huge, Inf * 0,
    Inf - Inf, NaN among huge terms), c likewise."""
    rng = np.random.default_rng(seed)
    mb = {"bf16": 7, "fp16": 10, "xf32": 23, "e4m3": 3, "e5m2": 2}[fmt]
    eb = {"fp16": 5, "e4m3": 4, "e5m2": 5}.get(fmt, 8)
    dt = {"xf32": np.uint32, "e4m3": np.uint8, "e5m2": np.uint8}.get(fmt, np.uint16)
    emax = (1 << eb) - 1

    def draw(shape, mbits, ebits):
        kind = rng.integers(0, 8, shape)
        field = rng.integers(0, 1 << ebits, shape)
        field = np.where(kind == 0, (1 << ebits) - 1, field)                       # Inf / NaN
        field = np.where(kind == 1, 0, field)                                       # zero / tiny
        field = np.where(kind == 2, rng.integers((1 << ebits) - 6, (1 << ebits) - 1, shape), field)  # huge
        field = np.where(kind == 3, rng.integers(0, 4, shape), field)               # tiny
        mant = rng.integers(0, 1 << mbits, shape)
        mant = np.where((kind == 0) & (rng.random(shape) < 0.6), 0, mant)           # Inf more often than NaN
        mant = np.where((kind == 1) & (rng.random(shape) < 0.7), 0, mant)           # +-0
        sign = rng.integers(0, 2, shape)
        return (sign << (mbits + ebits)) | (field << mbits) | mant

    a = draw((n, k), mb, eb).astype(dt)
    b = draw((n, k), mb, eb).astype(dt)
    if fmt == "xf32":
        a &= dt(0xFFFFE000)
        b &= dt(0xFFFFE000)
    c = draw(n, 23, 8).astype(np.uint32)
    assert emax > 0
    return a, b, c


@pytest.mark.parametrize("fmt,k", [("bf16", 4), ("xf32", 2), ("fp16", 4), ("e4m3", 8), ("e5m2", 8)])
def test_special_operand_mixes(L, fmt, k):
    """Every stream model on sets dense in Inf, NaN, zeros and extreme binades: the
    special result (NaN for a NaN, Inf * 0 or Inf - Inf, else the signed Inf) and the
    finite results around them.  OCP FP8 at K = 8 runs the paired kernel's product
    table, whose special entries (and, for E5M2, the signs of infinite products)
    decide these sets; E4M3's all-ones exponent field is finite but for the NaN
    mantissa."""
    a, b, c = _special_mix(fmt, 50000, k, seed=97)
    for name, spec in block_models(fmt, k).items():
        for out_round in ("rne", "rtz") if name == "ieee_exact" else (None,):
            s = spec if out_round is None else dict(spec, out_round=out_round)
            got = gpu_block(L, s, a, b, c)
            want = oracle.block_fma_parallel(s, a, b, c, threads=8)
            assert np.array_equal(got, want), f"{fmt} {name} {out_round}\n" + mismatches(got, want, a, b, c)


def _dropped_mix(fmt, n, k, seed):
    """c in a high binade, at most one product within 30 binades of it (so the kept sum
    leaves a remainder or none), the other products 112-140 binades below c with random
    signs and nearby exponents: the sign of the dropped terms' sum decides RZ."""
    rng = np.random.default_rng(seed)
    mb = 7 if fmt == "bf16" else 23
    dt = np.uint16 if fmt == "bf16" else np.uint32

    def elem(field, size):
        m = rng.integers(0, 1 << mb, size)
        if fmt == "xf32":
            m &= ~((1 << 13) - 1)
        return ((rng.integers(0, 2, size) << (mb + 8)) | (np.clip(field, 1, 254) << mb) | m).astype(dt)

    fc = rng.integers(150, 250, n)
    # product field sums: the first near c (or far below it), the rest 112-140 binades down
    gap = rng.integers(112, 141, (n, k))
    gap[:, 0] = np.where(rng.random(n) < 0.5, rng.integers(1, 30, n), gap[:, 0])
    gap[:, 1:] = np.minimum(gap[:, 1:], gap[:, 1:2] + rng.integers(0, 3, (n, k - 1)))   # nearby exponents
    s = fc[:, None] + 127 - gap
    fa = np.clip(s // 2, 1, 254)
    fb = np.clip(s - fa, 1, 254)
    a, b = elem(fa, (n, k)), elem(fb, (n, k))
    c = ((rng.integers(0, 2, n) << 31) | (fc << 23) | rng.integers(0, 1 << 23, n)).astype(np.uint32)
    return a, b, c


@pytest.mark.parametrize("fmt,k", [("bf16", 4), ("xf32", 2)])
def test_exact_rz_dropped_terms(L, fmt, k):
    """Exact-then-round, RZ and RNE, where the rounding hinges on terms far below the kept
    sum: their sign alone, or set against a small remainder of the kept sum."""
    a, b, c = _dropped_mix(fmt, 60000, k, seed=89)
    for out_round in ("rtz", "rne"):
        spec = dict(block_models(fmt, k)["ieee_exact"], out_round=out_round)
        got = gpu_block(L, spec, a, b, c)
        want = oracle.block_fma_parallel(spec, a, b, c, threads=8)
        assert np.array_equal(got, want), f"{fmt} {out_round}\n" + mismatches(got, want, a, b, c)


@pytest.mark.parametrize("fmt,k", [("bf16", 4), ("xf32", 2)])
def test_exact_scale_extremes(L, fmt, k):
    """Exact-then-round, RNE and RTZ, on BF16/XF32 sets at the ends of the exponent range,
    where the terms' common rescaling, its limits and the dropped terms decide the result."""
    a, b, c = _scale_extremes(fmt, 60000, k, seed=83)
    for out_round in ("rne", "rtz"):
        spec = dict(block_models(fmt, k)["ieee_exact"], out_round=out_round)
        got = gpu_block(L, spec, a, b, c)
        want = oracle.block_fma_parallel(spec, a, b, c, threads=8)
        assert np.array_equal(got, want), f"{fmt} {out_round}\n" + mismatches(got, want, a, b, c)


F16_OUT = ["b200_fp16_f16", "h100_fp16_f16", "a100_fp16_f16", "b200_fp8_f16", "h100_fp8_f16"]


@pytest.mark.parametrize("name", F16_OUT)
@pytest.mark.parametrize("variant", ["preset", "exact_rne", "rd_flush", "e5m2"])
def test_fp16_output_models(L, name, variant):
    """Table 3's note: fp16 c and d (binary16 in the low half of each word) for fp16 and
    fp8 inputs, e_min^lim -20/-21, RTZ; plus the exact model with RNE, round-down
    alignment with flushed subnormals, and E5M2 operands.  Independent bits with
    specials, and exponent-mantissa sets down at the limit."""
    spec = dict(PRESETS[name])
    if variant == "exact_rne":
        spec.update(arch="exact", out_round="rne")
    elif variant == "rd_flush":
        spec.update(align_round="rd", sub_in_flush=True, sub_out_flush=True)
    elif variant == "e5m2":
        if spec["fmt_a"] != "e4m3":
            pytest.skip("fp16 operands")
        spec.update(fmt_a="e5m2", fmt_b="e5m2")
    fmt, k = spec["fmt_a"], spec["n_fma"]
    rng = np.random.default_rng(80)
    a, b, _ = W.gen_block_fma_set(fmt, 20000, k, seed=81, special_rate=0.01)
    c = W.independent_bits(rng, "fp16", (20000,), "ocp", 0.01).astype(np.uint32)
    sets = [(a, b, c)]
    lo = {"fp16": (-24, -12), "e4m3": (-9, -4), "e5m2": (-16, -8)}[fmt]
    a2, b2, _ = W.gen_exp_mantissa(fmt, 20000, k, lo, (-14, 15), seed=0)
    c2 = W.gen_exp_mantissa("fp16", 20000, 1, (-24, -10), (-14, 15), seed=1)[0].reshape(-1).astype(np.uint32)
    sets.append((a2, b2, c2))
    for a, b, c in sets:
        got = gpu_block(L, spec, a, b, c)
        want = oracle.block_fma_parallel(spec, a, b, c, threads=8)
        assert np.array_equal(got, want), f"{name} {variant}\n" + mismatches(got, want, a, b, c)
        assert (got >> 16).max() == 0

GENERIC_CASES = [
    ("exact", "fp16", 1), ("exact", "bf16", 3), ("ga_early", "bf16", 5), ("ga_late", "fp16", 12),
    ("odd_even", "e4m3", 32), ("ga_early", "e5m2", 32), ("pairwise", "bf16", 8), ("exact", "xf32", 16),
    ("ga_late", "bf16", 16), ("exact", "fp32", 1), ("exact", "fp32", 3), ("ga_early", "fp32", 2),
    ("pairwise", "fp32", 1), ("ga_early", "fp16", 16), ("exact", "e4m3", 32),
]


@pytest.mark.parametrize("arch,fmt,k", GENERIC_CASES)
@pytest.mark.parametrize("variant", ["plain", "flush_rd_fnuz"])
def test_every_architecture_any_block_size(L, arch, fmt, k, variant):
    base = dict(fmt_a=fmt, fmt_b=fmt, arch=arch, n_fma=k, align_frac=24, c_zero_exp=-126,
                prod_overflow=True, nan_bits=0xFFC00000, pair_group=k)
    if arch == "ga_early":
        base.update(align_frac=25, c_zero_exp=None, emin_lim=-133, out_round="rtz")
    if variant == "flush_rd_fnuz":
        base.update(sub_in_flush=True, sub_out_flush=True, fp8_enc="fnuz", xf32_round="rne")
        if arch in ("ga_early",):
            base.update(align_round="rd")
    enc = base.get("fp8_enc", "ocp")
    a, b, c = W.gen_block_fma_set(fmt, 8000, k, seed=31 + k, enc=enc, special_rate=0.02)
    got = gpu_block(L, base, a, b, c)
    want = oracle.block_fma_parallel(base, a, b, c, threads=8)
    assert np.array_equal(got, want), f"{arch} {fmt} k={k} {variant}\n" + mismatches(got, want, a, b, c)


def test_mixed_fp8_operands(L):
    spec = dict(PRESETS["cdna3_fp8"], fmt_b="e5m2")
    a = W.gen_exp_mantissa("e4m3", 20000, 16, (-7, 7), (-126, 127), seed=0, enc="fnuz")[0]
    b, _, c = W.gen_exp_mantissa("e5m2", 20000, 16, (-15, 15), (-126, 127), seed=1, enc="fnuz")
    got = gpu_block(L, spec, a, b, c)
    want = oracle.block_fma_parallel(spec, a, b, c, threads=8)
    assert np.array_equal(got, want), mismatches(got, want)


FP8_ADDENDS = ["0", "-0", "2^-149", "-1", "3*2^-30", "1.5*2^20", "-2^-20", "0.75", "-448", "2^-126"]


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("enc", ["ocp", "fnuz"])
def test_fp8_all_pairs(L, fmt, enc):
    """Every (a, b) pair of the 8-bit format against a set of addends: K = 1 (the general
    evaluator) and K = 8 with the pair among seven zero products (the product-table
    kernel), for truncation, RNE and exact-then-round, and the CDNA 3 Algorithm 2
    preset (K = 16)."""
    codes = np.arange(256, dtype=np.uint8)
    a1 = np.repeat(codes, 256)
    b1 = np.tile(codes, 256)
    n = a1.size
    cs = np.array([W.encode_exact(W.parse_value(x), "fp32") for x in FP8_ADDENDS], np.uint32)
    models = {name: dict(spec, fp8_enc=enc) for name, spec in block_models(fmt, 8).items()}
    models["cdna3"] = dict(PRESETS["cdna3_fp8" if fmt == "e4m3" else "cdna3_bf8"], fp8_enc=enc)
    rng = np.random.default_rng(9)
    for name, spec in models.items():
        for k in (1, spec["n_fma"]):
            s = dict(spec, n_fma=k)
            pos = rng.integers(0, k, n)                       # where the pair sits in the block
            a = np.zeros((n, k), np.uint8)
            b = np.zeros((n, k), np.uint8)
            a[np.arange(n), pos] = a1
            b[np.arange(n), pos] = b1
            for cb in cs:
                c = np.full(n, cb, np.uint32)
                got = gpu_block(L, s, a, b, c)
                want = oracle.block_fma_parallel(s, a, b, c, threads=8)
                assert np.array_equal(got, want), f"{fmt} {enc} {name} k={k} c={cb:#x}\n" + mismatches(got, want)

@pytest.mark.parametrize("sat", [False, True])
@pytest.mark.parametrize("fa,fb", [("int8", "int8"), ("uint8", "uint8"), ("int8", "uint8")])
def test_integer_formats(L, fa, fb, sat):
    rng = np.random.default_rng(3)
    n = 50000
    a = rng.integers(0, 256, (n, 16), dtype=np.uint64).astype(np.uint8)
    b = rng.integers(0, 256, (n, 16), dtype=np.uint64).astype(np.uint8)
    c = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
    c[:100] = 0x7FFFFFF0
    c[100:200] = 0x80000010
    spec = dict(fmt_a=fa, fmt_b=fb, arch="exact", n_fma=16, int_saturate=sat)
    got = gpu_block(L, spec, a, b, c)
    want = oracle.block_fma(spec, a, b, c)
    assert np.array_equal(got, want), mismatches(got, want)


def test_empty_single_and_ragged(L):
    spec = block_models("bf16", 4)["ga_trunc"]
    m = L.Model(spec)
    e = torch.empty(0, dtype=torch.int16, device="cuda")
    d = L.block_fma(m, e, e, torch.empty(0, dtype=torch.int32, device="cuda"))
    assert d.numel() == 0
    for n in (1, 2, 255, 257, 100003):
        a, b, c = W.gen_block_fma_set("bf16", n, 4, seed=n)
        got = gpu_block(L, spec, a, b, c)
        assert np.array_equal(got, oracle.block_fma(spec, a, b, c))


@pytest.mark.parametrize("fmt,k", [("fp16", 4), ("bf16", 4), ("xf32", 2), ("e4m3", 8), ("e5m2", 8)])
@pytest.mark.parametrize("name", ["ga_trunc", "ga_rne", "ieee_exact"])
def test_paired_sets_tails_and_alignment(L, fmt, k, name):
    """The models on 8-byte sets run two sets per thread with 16-byte loads: odd
    counts end with a one-set launch, and operands only 8-byte aligned (or c, d only
    4-byte aligned) take the one-set kernel; every case against the oracle."""
    spec = block_models(fmt, k)[name]
    m = L.Model(spec)
    for n in (2, 3, 63, 64, 65, 100001):
        a, b, c = W.gen_block_fma_set(fmt, n, k, seed=n + 5)
        want = oracle.block_fma(spec, a, b, c)
        for off_ab, off_cd in ((0, 0), (8, 0), (0, 4)):
            def place(x, off):
                raw = np.ascontiguousarray(x).view(np.uint8).reshape(-1)
                buf = torch.zeros(raw.size + 64, dtype=torch.uint8, device="cuda")
                buf[off:off + raw.size] = torch.from_numpy(raw).cuda()
                return buf[off:off + raw.size]
            da, db = place(a, off_ab), place(b, off_ab)
            dc = place(c, off_cd).view(torch.int32)                      # n elements, 4-byte aligned
            dd = place(np.zeros(n, np.uint32), off_cd).view(torch.int32)
            L.block_fma(m, da, db, dc, dd)
            got = dd.cpu().numpy().view(np.uint32)
            assert np.array_equal(got, want), f"{fmt} {name} n={n} offsets {off_ab}/{off_cd}\n" + mismatches(got, want)

@pytest.mark.parametrize("fa,fb", [("int8", "int8"), ("uint8", "uint8"), ("int8", "uint8")])
@pytest.mark.parametrize("sat", [False, True])
def test_int8_pairs_tails_and_alignment(L, fa, fb, sat):
    """INT8 K=16 runs two sets per thread: odd counts, and c, d only 4-byte aligned
    (the one-set kernel), against the integer dot product of the oracle."""
    spec = dict(fmt_a=fa, fmt_b=fb, arch="exact", n_fma=16, int_saturate=sat)
    m = L.Model(spec)
    rng = np.random.default_rng(5)
    for n in (2, 3, 1001, 65536):
        a = rng.integers(0, 256, (n, 16), dtype=np.uint64).astype(np.uint8)
        b = rng.integers(0, 256, (n, 16), dtype=np.uint64).astype(np.uint8)
        c = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
        c[: n // 3] = 0x7FFFFF00
        want = oracle.block_fma(spec, a, b, c)
        for off in (0, 1):                       # c and d 4-byte but not 8-byte aligned: one set per thread
            bufc = torch.zeros(n + 2, dtype=torch.int32, device="cuda")
            bufd = torch.zeros(n + 2, dtype=torch.int32, device="cuda")
            bufc[off:off + n] = torch.from_numpy(c.view(np.int32)).cuda()
            L.block_fma(m, dev(a), dev(b), bufc[off:off + n], bufd[off:off + n])
            got = bufd[off:off + n].cpu().numpy().view(np.uint32)
            assert np.array_equal(got, want), f"{fa}x{fb} sat={sat} n={n} off={off}\n" + mismatches(got, want)

@pytest.mark.parametrize("pinned", [True, False])
def test_host_entry_point(L, pinned):
    """mcemu_block_fma_host on page-locked buffers (read in place by the kernel) and on
    pageable ones (staged through the workspace), against the device entry point."""
    n = 3 * 4_194_304 // 2 + 7                    # crosses the staging chunk size
    for fmt, k in (("bf16", 4), ("e4m3", 8)):
        a, b, c = W.gen_block_fma_set(fmt, n, k, seed=23)
        m = L.Model(block_models(fmt, k)["ga_rne"])
        want = gpu_block(L, block_models(fmt, k)["ga_rne"], a, b, c)

        def host(x):
            x = np.ascontiguousarray(x)
            t = torch.from_numpy(x.view({np.uint16: np.int16, np.uint32: np.int32}.get(x.dtype.type, x.dtype)))
            return t.pin_memory() if pinned else t
        ha, hb, hc = host(a), host(b), host(c)
        hd = torch.empty(n, dtype=torch.int32)
        hd = hd.pin_memory() if pinned else hd
        ws = torch.empty(L.block_fma_host_workspace(m), dtype=torch.uint8, device="cuda")
        L.block_fma_host(m, ha, hb, hc, hd, ws)
        assert np.array_equal(hd.numpy().view(np.uint32), want)


def test_misaligned_pointer_is_rejected(L):
    spec = block_models("fp16", 4)["ga_rne"]
    m = L.Model(spec)
    buf = torch.zeros(4 * 64 + 8, dtype=torch.int16, device="cuda")
    a = buf[1:1 + 4 * 64]                        # 2-byte offset: not 8-byte aligned
    c = torch.zeros(64, dtype=torch.int32, device="cuda")
    with pytest.raises(L.McemuError) as e:
        L.block_fma(m, a, a, c)
    assert e.value.status == 4

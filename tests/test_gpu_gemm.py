"""Emulated GEMMs on the GPU (dense tile GEMM, 2:4 compression and sparse GEMM,
multi-word GEMM), bit for bit against the oracle through the C ABI."""
import os
import threading

import numpy as np
import pytest

import oracle
from oracle.presets import PRESETS, block_models
from bit_exact_emulation_gb300 import workloads as W

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


def host_u32(t):
    return t.cpu().numpy().view(np.uint32)


def all_entries(M, N):
    ii, jj = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    return ii.ravel().astype(np.int32), jj.ravel().astype(np.int32)


def operands(fmt, M, N, K, seed, enc="ocp", special_rate=0.0):
    rng = np.random.default_rng(seed)
    if fmt == "bf16" and special_rate == 0.0:
        A, Bt, C = W.gen_dense_bf16(M, N, K, seed)
        return A, Bt, C
    A = W.independent_bits(rng, fmt, (M, K), enc, special_rate)
    Bt = W.independent_bits(rng, fmt, (N, K), enc, special_rate)
    if fmt in ("int8", "uint8"):
        C = rng.integers(0, 1 << 32, (M, N), dtype=np.uint64).astype(np.uint32)
    else:
        C = rng.standard_normal((M, N), dtype=np.float32).view(np.uint32)
    return A, Bt, C


GEMM_CASES = [  # model, tile K (instruction inner size), input format
    (PRESETS["cdna3_bf16"], 8, "bf16"),                 # 32x32x8 bf16_1k, N_FMA 8
    (PRESETS["cdna3_fp16"], 16, "fp16"),                # 16x16x16 f16
    (PRESETS["cdna3_xf32"], 8, "xf32"),                 # 16x16x8 xf32, N_FMA 4
    (PRESETS["cdna3_fp8"], 32, "e4m3"),                 # 16x16x32 fp8, Algorithm 2
    (PRESETS["cdna1_bf16"], 8, "bf16"),                 # exact, N_FMA 2
    (PRESETS["cdna2_fp16"], 16, "fp16"),                # pair-wise
    (PRESETS["b200_fp16"], 16, "fp16"),
    (block_models("bf16", 4)["ga_trunc"], 8, "bf16"),
    (block_models("bf16", 4)["ga_rne"], 8, "bf16"),
    (block_models("bf16", 4)["ieee_exact"], 8, "bf16"),
    (dict(fmt_a="int8", fmt_b="int8", arch="exact", n_fma=16), 16, "int8"),
    (PRESETS["cdna1_fp16"], 16, "fp16"),                # exact, N_FMA 4, with specials
    (block_models("xf32", 2)["ieee_exact"], 8, "xf32"),
    (block_models("e4m3", 8)["ieee_exact"], 32, "e4m3"),
]


@pytest.mark.parametrize("case", range(len(GEMM_CASES)))
@pytest.mark.parametrize("shape", [(37, 29, 100), (16, 16, 8), (1, 1, 3)])
def test_tile_gemm_full(L, case, shape):
    spec, kt, fmt = GEMM_CASES[case]
    M, N, K = shape
    enc = spec.get("fp8_enc", "ocp")
    A, Bt, C = operands(fmt, M, N, K, seed=case, enc=enc, special_rate=0.01 if fmt != "bf16" else 0.0)
    m = L.Model(spec)
    D = host_u32(L.tile_gemm(m, L.tile(0, 16, 16, kt, 4), dev(A), dev(Bt), dev(C)))
    ii, jj = all_entries(M, N)
    want = oracle.gemm_entries(spec, K, kt, A, Bt, C, ii, jj).reshape(M, N)
    bad = np.argwhere(D != want)
    assert len(bad) == 0, f"{len(bad)} mismatches, first {bad[:5].tolist()}"


EARLY_RANGE_CASES = [  # format, element scale 2^s, addend scale 2^t, model options
    ("bf16", -63, -126, dict(out_round="rne")),                       # results cross into subnormals
    ("bf16", -63, -130, dict(out_round="rtz", sub_in_flush=True)),
    ("bf16", 62, 123, dict(out_round="rne")),                         # results overflow mid-chain
    ("bf16", 62, 125, dict(out_round="rtz")),
    ("bf16", 0, 0, dict(out_round="rne", emin_lim=-133, c_zero_exp=-126)),
    ("fp16", None, None, dict(out_round="rne")),                      # random bit patterns
    ("fp16", -7, -140, dict(out_round="rtz", align_frac=20)),
    ("e4m3", None, None, dict(out_round="rtz", n_fma=8)),
    ("e5m2", -8, -135, dict(out_round="rne", n_fma=8, align_frac=29)),
    ("xf32", 40, 100, dict(out_round="rne", n_fma=2, align_frac=24)),
]


@pytest.mark.parametrize("case", range(len(EARLY_RANGE_CASES)))
def test_early_c_gemm_exponent_ranges(L, case):
    """Early-c global alignment through the fast GEMM kernel with chains whose partial
    results leave the normal fp32 range (overflow, subnormal), subnormal and zero
    addends, exponent limits and flushed inputs, over several CTA tiles with ragged
    edges: every output against the oracle."""
    fmt, s, t, opts = EARLY_RANGE_CASES[case]
    spec = dict(dict(fmt_a=fmt, fmt_b=fmt, arch="ga_early", n_fma=4, align_frac=26), **opts)
    rng = np.random.default_rng(40 + case)
    M, N, K, kt = 70, 67, 200, 2 * spec["n_fma"]
    if s is None:
        A = W.independent_bits(rng, fmt, (M, K), "ocp", 0.0)
        Bt = W.independent_bits(rng, fmt, (N, K), "ocp", 0.0)
        C = W.independent_bits(rng, "fp32", (M, N), "ocp", 0.0)
    else:
        def draw(shape):
            x = rng.standard_normal(shape) * 2.0 ** s
            x[rng.random(shape) < 0.05] = 0.0
            if fmt == "bf16":
                return W.fp32_to_bf16_rne(x.astype(np.float32))
            if fmt == "xf32":
                return x.astype(np.float32).view(np.uint32) & np.uint32(0xFFFFE000)
            return W.nearest_even(x, fmt)
        A, Bt = draw((M, K)), draw((N, K))
        c = (rng.standard_normal((M, N)) * 2.0 ** t).astype(np.float32)
        c[rng.random((M, N)) < 0.1] = 0.0
        C = c.view(np.uint32).copy()
    m = L.Model(spec)
    D = host_u32(L.tile_gemm(m, L.tile(0, 16, 16, kt, 4), dev(A), dev(Bt), dev(C)))
    ii, jj = all_entries(M, N)
    want = oracle.gemm_entries(spec, K, kt, A, Bt, C, ii, jj).reshape(M, N)
    bad = np.argwhere(D != want)
    assert len(bad) == 0, f"{len(bad)} mismatches, first {bad[:5].tolist()}"


GEMM_BOUNDARY = [  # format, model, instruction K
    ("bf16", PRESETS["cdna3_bf16"], 8), ("bf16", block_models("bf16", 4)["ga_rne"], 8),
    ("bf16", block_models("bf16", 4)["ga_trunc"], 8), ("bf16", block_models("bf16", 4)["ieee_exact"], 8),
    ("xf32", PRESETS["cdna3_xf32"], 8), ("xf32", block_models("xf32", 2)["ieee_exact"], 8),
    ("bf16", PRESETS["b200_bf16"], 16),
]


@pytest.mark.parametrize("case", range(len(GEMM_BOUNDARY)))
def test_gemm_subnormal_boundary(L, case):
    """The tile GEMM on sums next to 2^-126: row i of A and of B^T is one boundary
    vector set (with C[i][:] its addend), so every diagonal output is a set that sits
    at or near a tie of the subnormal grid; the off-diagonal ones mix sets.  Every
    output against the oracle (the fast kernels send these chains to the fixup pass)."""
    fmt, spec, kt = GEMM_BOUNDARY[case]
    k = spec["n_fma"]
    n = 96
    a, b, c = W.gen_subnormal_boundary(fmt, n, k, seed=90 + case)
    A, Bt = np.ascontiguousarray(a), np.ascontiguousarray(b)
    C = np.repeat(c.reshape(n, 1), n, axis=1)
    m = L.Model(spec)
    D = host_u32(L.tile_gemm(m, L.tile(0, 16, 16, kt, 4), dev(A), dev(Bt), dev(C)))
    ii, jj = all_entries(n, n)
    want = oracle.gemm_entries(spec, k, kt, A, Bt, C, ii, jj).reshape(n, n)
    bad = np.argwhere(D != want)
    assert len(bad) == 0, f"{len(bad)} mismatches, first {bad[:5].tolist()}"

@pytest.mark.parametrize("name", ["b200_fp16_f16", "a100_fp16_f16", "h100_fp8_f16"])
def test_gemm_fp16_output(L, name):
    """Tile GEMM with the fp16 accumulator: C and D hold binary16 in the low half of
    each 32-bit word, and every block's binary16 result is the next block's addend."""
    spec = PRESETS[name]
    fmt = spec["fmt_a"]
    M, N, K, kt = 37, 29, 96, 2 * spec["n_fma"]
    rng = np.random.default_rng(7)
    A = W.independent_bits(rng, fmt, (M, K), "ocp", 0.005)
    Bt = W.independent_bits(rng, fmt, (N, K), "ocp", 0.005)
    if fmt == "fp16":                                   # keep most chains finite
        A = (A & np.uint16(0xBFFF)).astype(np.uint16)
        Bt = (Bt & np.uint16(0xBFFF)).astype(np.uint16)
    C = W.independent_bits(rng, "fp16", (M, N), "ocp", 0.005).astype(np.uint32)
    m = L.Model(spec)
    D = host_u32(L.tile_gemm(m, L.tile(0, 16, 16, kt, 4), dev(A), dev(Bt), dev(C)))
    ii, jj = all_entries(M, N)
    want = oracle.gemm_entries(spec, K, kt, A, Bt, C, ii, jj).reshape(M, N)
    bad = np.argwhere(D != want)
    assert len(bad) == 0, f"{len(bad)} mismatches, first {bad[:5].tolist()}"
    assert (D >> 16).max() == 0

def test_tile_gemm_specials_and_zero_k(L):
    spec = PRESETS["cdna3_bf16"]
    A, Bt, C = operands("bf16", 20, 20, 64, seed=5, special_rate=0.03)
    m = L.Model(spec)
    D = host_u32(L.tile_gemm(m, L.tile(0, 32, 32, 8, 4), dev(A), dev(Bt), dev(C)))
    ii, jj = all_entries(20, 20)
    assert np.array_equal(D.ravel(), oracle.gemm_entries(spec, 64, 8, A, Bt, C, ii, jj))
    # K = 0: D = C
    A0 = torch.empty((20, 0), dtype=torch.int16, device="cuda")
    D0 = host_u32(L.tile_gemm(m, L.tile(0, 32, 32, 8, 4), A0, A0, dev(C)))
    assert np.array_equal(D0, C)


@pytest.mark.parametrize("fmt", ["bf16", "fp16"])
def test_exact_gemm_cancellation(L, fmt):
    """C is minus the fp32-rounded exact A*B, moved by a few units in the last place:
    every chain ends in heavy cancellation, which the exact kernel's window must either
    round correctly or hand to the general evaluator."""
    M, N, K = 48, 40, 64
    rng = np.random.default_rng(9)
    if fmt == "bf16":
        A, Bt, _ = W.gen_dense_bf16(M, N, K, seed=9)
        fa = (A.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        fb = (Bt.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    else:
        A = rng.standard_normal((M, K)).astype(np.float16).view(np.uint16)
        Bt = rng.standard_normal((N, K)).astype(np.float16).view(np.uint16)
        fa, fb = A.view(np.float16).astype(np.float64), Bt.view(np.float16).astype(np.float64)
    C = (-(fa @ fb.T)).astype(np.float32).view(np.int32) + rng.integers(-2, 3, (M, N)).astype(np.int32)
    C = C.view(np.uint32)
    spec = block_models(fmt, 4)["ieee_exact"]
    m = L.Model(spec)
    D = host_u32(L.tile_gemm(m, L.tile(0, 32, 32, 8, 4), dev(A), dev(Bt), dev(C)))
    ii, jj = all_entries(M, N)
    want = oracle.gemm_entries(spec, K, 8, A, Bt, C, ii, jj).reshape(M, N)
    assert np.array_equal(D, want), f"{int((D != want).sum())} mismatches"


@pytest.mark.parametrize("name", ["cdna3_bf16", "ga_rne", "ieee_exact"])
def test_in_place_accumulation(L, name):
    """D = A*B + D with D the same buffer as C (the general kernel then runs), and D a
    separate buffer (the fast kernels), against the oracle."""
    spec = PRESETS["cdna3_bf16"] if name == "cdna3_bf16" else block_models("bf16", 4)[name]
    M, N, K = 70, 66, 96
    A, Bt, C = operands("bf16", M, N, K, seed=12)
    m = L.Model(spec)
    ii, jj = all_entries(M, N)
    want = oracle.gemm_entries(spec, K, 8, A, Bt, C, ii, jj).reshape(M, N)
    dC = dev(C)
    D_sep = host_u32(L.tile_gemm(m, L.tile(0, 32, 32, 8, 4), dev(A), dev(Bt), dC))
    L.tile_gemm(m, L.tile(0, 32, 32, 8, 4), dev(A), dev(Bt), dC, dC)
    assert np.array_equal(D_sep, want)
    assert np.array_equal(host_u32(dC), want)


def entries_parallel(fn, ii, jj):
    """fn(ii_part, jj_part) over the host's cores: the oracle's C calls release the GIL
    and keep no state between calls."""
    parts = np.array_split(np.arange(len(ii)), max(1, min(os.cpu_count() or 1, 32)))
    out = [None] * len(parts)

    def work(t):
        out[t] = fn(ii[parts[t]], jj[parts[t]])

    ts = [threading.Thread(target=work, args=(t,)) for t in range(len(parts))]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    return np.concatenate(out)


def test_dense_bf16_2048_sampled(L):
    """The dense BF16 GEMM workload: M = N = K = 2048, 32x32x8 bf16 tile semantics;
    2048 sampled outputs per model against the oracle."""
    M = N = K = 2048
    A, Bt, C = W.gen_dense_bf16(M, N, K, seed=3)
    rng = np.random.default_rng(11)
    ii = rng.integers(0, M, 2048).astype(np.int32)
    jj = rng.integers(0, N, 2048).astype(np.int32)
    for spec in (PRESETS["cdna3_bf16"], block_models("bf16", 4)["ga_trunc"], block_models("bf16", 4)["ga_rne"],
                 block_models("bf16", 4)["ieee_exact"]):
        m = L.Model(spec)
        D = host_u32(L.tile_gemm(m, L.tile(0, 32, 32, 8, 4), dev(A), dev(Bt), dev(C)))
        want = entries_parallel(lambda i, j: oracle.gemm_entries(spec, K, 8, A, Bt, C, i, j), ii, jj)
        assert np.array_equal(D[ii, jj], want)


# ---------------------------------------------------------------------------
# 2:4 sparsity
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("fmt,enc", [("e4m3", "ocp"), ("e4m3", "fnuz"), ("fp16", "ocp"), ("bf16", "ocp"),
                                     ("int8", "ocp")])
def test_sparse24_compress_matches_oracle(L, fmt, enc):
    rng = np.random.default_rng(1)
    M, K = 97, 128
    A = W.independent_bits(rng, fmt, (M, K), enc, 0.01)
    # zero out two thirds of the entries so that most groups have <= 2 nonzeros
    A[rng.random((M, K)) < 0.6] = 0
    Ac, meta, viol = L.sparse24_compress(fmt, dev(A), enc)
    rAc, rmeta, rviol = oracle.sparse24_compress(fmt, A, enc)
    assert np.array_equal(Ac.cpu().numpy().view(A.dtype), rAc)
    assert np.array_equal(meta.cpu().numpy(), rmeta)
    assert int(viol.item()) == rviol and rviol > 0


def test_sparse24_violation_raises_not_2_4(L):
    """A group of four with three nonzeros: the device counter reports it, and the
    synchronous check returns MCEMU_ERR_NOT_2_4 (the 2:4 pattern does not hold)."""
    A, _, _ = W.gen_sparse_e4m3(8, 8, 64, seed=4)
    ok_Ac, _, v0 = L.sparse24_compress("e4m3", dev(A), check=True)   # a valid pattern passes
    assert int(v0.item()) == 0
    bad = A.copy()
    g = bad[3, 8:12]
    bad[3, 8:12] = np.where(g == 0, np.uint8(0x38), g)[:4]          # fill the zeros: 4 nonzeros
    bad[5, 20:24] = [0x38, 0x40, 0x48, 0]                            # 3 nonzeros
    Ac, meta, viol = L.sparse24_compress("e4m3", dev(bad))
    torch.cuda.synchronize()
    assert int(viol.item()) == 2
    with pytest.raises(L.McemuError) as e:
        L.sparse24_compress("e4m3", dev(bad), check=True)
    assert e.value.status == 3
    want_Ac, want_meta, want_v = oracle.sparse24_compress("e4m3", bad)
    assert want_v == 2
    assert np.array_equal(Ac.cpu().numpy(), want_Ac) and np.array_equal(meta.cpu().numpy(), want_meta)

def test_sparse24_expand_inverts_compress(L):
    A, Bt, C = W.gen_sparse_e4m3(64, 8, 256, seed=4)
    Ac, meta, viol = L.sparse24_compress("e4m3", dev(A))
    assert int(viol.item()) == 0
    E = L.sparse24_expand("e4m3", Ac, meta, 256)
    assert np.array_equal(E.cpu().numpy(), A)


SPARSE_CASES = [
    dict(fmt_a="e4m3", fmt_b="e4m3", arch="ga_early", n_fma=8, align_frac=26, out_round="rtz"),
    dict(fmt_a="e4m3", fmt_b="e4m3", arch="ga_early", n_fma=8, align_frac=26, out_round="rne"),
    dict(fmt_a="e4m3", fmt_b="e4m3", arch="exact", n_fma=8),
    dict(PRESETS["cdna3_fp8"], fp8_enc="ocp", n_fma=8),
    # blocks of 5 and 3 compressed terms: blocks that end inside a group of four
    dict(fmt_a="e4m3", fmt_b="e4m3", arch="ga_early", n_fma=5, align_frac=26, out_round="rne"),
    dict(PRESETS["cdna3_bf16"], fmt_a="e4m3", fmt_b="e4m3", n_fma=3),
]


@pytest.mark.parametrize("case", range(len(SPARSE_CASES)))
def test_sparse24_gemm_full(L, case):
    spec = SPARSE_CASES[case]
    M, N, K = 45, 33, 160
    A, Bt, C = W.gen_sparse_e4m3(M, N, K, seed=case, c_zero=False)
    Ac, meta, _ = oracle.sparse24_compress("e4m3", A)
    m = L.Model(spec)
    D = host_u32(L.sparse24_gemm(m, L.tile(1, 16, 16, 32, 8), dev(Ac), dev(meta), dev(Bt), dev(C)))
    ii, jj = all_entries(M, N)
    want = oracle.sparse24_entries(spec, K, 32, Ac, meta, Bt, C, ii, jj).reshape(M, N)
    assert np.array_equal(D, want), f"{int((D != want).sum())} mismatches"


@pytest.mark.parametrize("fmt", ["e4m3", "fp16"])
@pytest.mark.parametrize("arch", ["ga_early", "ga_late"])
def test_sparse24_gemm_specials_and_bad_metadata(L, fmt, arch):
    """Specials in Ac and B, metadata with idx0 >= idx1 and a K that is not a multiple
    of the instruction: the outputs that leave the fast path take the compressed chain."""
    rng = np.random.default_rng(21)
    M, N, K = 70, 67, 200
    Ac = W.independent_bits(rng, fmt, (M, K // 2), "ocp", 0.001)
    Bt = W.independent_bits(rng, fmt, (N, K), "ocp", 0.0005)
    pairs = np.array([0b0100, 0b1000, 0b1100, 0b1001, 0b1101, 0b1110], np.uint8)
    meta = pairs[rng.integers(0, 6, (M, K // 4))]
    meta[3, 5] = 0b0101                     # idx0 == idx1
    meta[10, :] = 0b0011                    # idx0 > idx1 along a whole row
    C = rng.standard_normal((M, N), dtype=np.float32).view(np.uint32)
    if arch == "ga_early":
        spec = dict(fmt_a=fmt, fmt_b=fmt, arch="ga_early", n_fma=8, align_frac=26, out_round="rne")
    else:
        spec = dict(PRESETS["cdna3_bf16"], fmt_a=fmt, fmt_b=fmt, n_fma=8)
    m = L.Model(spec)
    D = host_u32(L.sparse24_gemm(m, L.tile(1, 16, 16, 32, 8), dev(Ac), dev(meta), dev(Bt), dev(C)))
    ii, jj = all_entries(M, N)
    want = oracle.sparse24_entries(spec, K, 32, Ac, meta, Bt, C, ii, jj).reshape(M, N)
    assert np.array_equal(D, want), f"{int((D != want).sum())} mismatches"


@pytest.mark.parametrize("case", [0, 1])
def test_sparse_e4m3_4096_sampled(L, case):
    """The 2:4 E4M3 workload at full size (truncation and RNE outputs): A 4096x4096
    compressed to 4096x2048, 16x16x32 tiles."""
    M = N = K = 4096
    A, Bt, C = W.gen_sparse_e4m3(M, N, K, seed=4)
    dA = dev(A)
    Ac, meta, viol = L.sparse24_compress("e4m3", dA)
    assert int(viol.item()) == 0
    spec = SPARSE_CASES[case]
    m = L.Model(spec)
    D = host_u32(L.sparse24_gemm(m, L.tile(1, 16, 16, 32, 8), Ac, meta, dev(Bt), dev(C)))
    rng = np.random.default_rng(12 + case)
    ii = rng.integers(0, M, 2048).astype(np.int32)
    jj = rng.integers(0, N, 2048).astype(np.int32)
    hAc, hmeta = Ac.cpu().numpy(), meta.cpu().numpy()
    want = entries_parallel(lambda i, j: oracle.sparse24_entries(spec, K, 32, hAc, hmeta, Bt, C, i, j), ii, jj)
    assert np.array_equal(D[ii, jj], want)


# ---------------------------------------------------------------------------
# multi-word GEMM
# ---------------------------------------------------------------------------
def test_multiword_split_matches_oracle(L):
    A, _ = W.gen_multiword_fp64(64, 1, 96, seed=5)
    w = L.multiword_split(torch.from_numpy(A).cuda(), 3).cpu().numpy().view(np.uint16)
    assert np.array_equal(w, oracle.split_bf16(A, 3))


@pytest.mark.parametrize("truncated", [False, True])
@pytest.mark.parametrize("word_model", ["cdna3_bf16", "ga_trunc"])
def test_multiword_gemm_full(L, truncated, word_model):
    spec = PRESETS["cdna3_bf16"] if word_model == "cdna3_bf16" else block_models("bf16", 8)["ga_trunc"]
    M, N, K = 19, 23, 72
    A, Bt = W.gen_multiword_fp64(M, N, K, seed=6)
    m = L.Model(spec)
    D = L.multiword_gemm(m, L.tile(0, 32, 32, 8, 4), 3, truncated, torch.from_numpy(A).cuda(),
                         torch.from_numpy(Bt).cuda()).cpu().numpy()
    ii, jj = all_entries(M, N)
    want = oracle.multiword_entries(spec, 8, 3, truncated, A, Bt, ii, jj).reshape(M, N)
    assert np.array_equal(D.view(np.uint64), want.view(np.uint64))


@pytest.mark.parametrize("n_words", [1, 2, 4])
def test_multiword_gemm_word_counts(L, n_words):
    """Every word count the fast word-product path takes, with a ragged tile edge."""
    spec = PRESETS["cdna3_bf16"]
    M, N, K = 66, 65, 40
    A, Bt = W.gen_multiword_fp64(M, N, K, seed=8 + n_words)
    m = L.Model(spec)
    for truncated in (False, True):
        D = L.multiword_gemm(m, L.tile(0, 32, 32, 8, 4), n_words, truncated, torch.from_numpy(A).cuda(),
                             torch.from_numpy(Bt).cuda()).cpu().numpy()
        ii, jj = all_entries(M, N)
        want = oracle.multiword_entries(spec, 8, n_words, truncated, A, Bt, ii, jj).reshape(M, N)
        assert np.array_equal(D.view(np.uint64), want.view(np.uint64))


def test_multiword_fp64_4096_sampled(L):
    """The multi-word workload at full size (4096^3, 3 words, 9 and 6 products, CDNA3 BF16
    word model): sampled entries against the oracle."""
    M = N = K = 4096
    A, Bt = W.gen_multiword_fp64(M, N, K, seed=5)
    m = L.Model(PRESETS["cdna3_bf16"])
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(Bt).cuda()
    rng = np.random.default_rng(13)
    ii = rng.integers(0, M, 256).astype(np.int32)
    jj = rng.integers(0, N, 256).astype(np.int32)
    for truncated in (False, True):
        D = L.multiword_gemm(m, L.tile(0, 32, 32, 8, 4), 3, truncated, dA, dB).cpu().numpy()
        want = entries_parallel(
            lambda i, j: oracle.multiword_entries(PRESETS["cdna3_bf16"], 8, 3, truncated, A, Bt, i, j), ii, jj)
        assert np.array_equal(D[ii, jj].view(np.uint64), want.view(np.uint64))


def test_multiword_error_report(L):
    M, N, K = 64, 48, 256
    A, Bt = W.gen_multiword_fp64(M, N, K, seed=7)
    m = L.Model(PRESETS["cdna3_bf16"])
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(Bt).cuda()
    errs = []
    for truncated in (False, True):
        D = L.multiword_gemm(m, L.tile(0, 32, 32, 8, 4), 3, truncated, dA, dB)
        R = dA @ dB.T
        e2, r2 = L.fro_error(D, R).cpu().numpy()
        errs.append(np.sqrt(e2 / r2))
        ref = np.sqrt(((D.cpu().numpy() - R.cpu().numpy()) ** 2).sum() / (R.cpu().numpy() ** 2).sum())
        assert abs(errs[-1] - ref) <= 1e-12 * max(ref, 1e-300)
    assert errs[0] < 1e-5 and errs[1] < 1e-5

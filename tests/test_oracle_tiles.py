"""Oracle pins for the tile semantics, 2:4 compression and the multi-word split (no GPU)."""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from bit_exact_emulation_gb300 import workloads as W
from _golden import GOLDEN


def _table(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append([c.strip() for c in line.split("|")])
    return rows


def test_block_count_matches_ops_column():
    """blocks = 64 * (elements per lane) / (M*K) reproduces Ops = 2*M*N*K*blocks for every
    builtin of the throughput table (the page's 'packed: blocks = 64/M' rule does not)."""
    rows = _table("mfma_builtins.txt")
    assert len(rows) == 32
    for name, M, N, K, epl, ops, _cyc in rows:
        M, N, K, epl, ops = map(int, (M, N, K, epl, ops))
        blocks, acc = oracle.tile_blocks(0, M, N, K, epl)
        assert ops == 2 * M * N * K * blocks, name
        assert acc == blocks * M * N // 64
    # the printed accumulator sizes: 32x32 two blocks -> 32 accVGPRs, 16x16 four -> 16, 4x4 -> 4
    assert oracle.tile_blocks(0, 32, 32, 1, 1) == (2, 32)
    assert oracle.tile_blocks(0, 16, 16, 1, 1) == (4, 16)
    assert oracle.tile_blocks(0, 4, 4, 1, 1) == (16, 4)
    assert oracle.tile_blocks(1, 16, 16, 32, 8) == (1, 8)


def _span(s):
    if "," in s:
        return [int(x) for x in s.split(",")]
    lo, hi = (int(x) for x in s.split("-")) if "-" in s else (int(s), int(s))
    return list(range(lo, hi + 1))


def test_printed_layout_tables():
    for layout, M, blocks, rows, block, lanes, regs in _table("tile_layouts.txt"):
        M, blocks = int(M), int(blocks)
        rset, bset, lset, gset = _span(rows), _span(block), set(_span(lanes)), set(_span(regs))
        seen_l, seen_g = set(), set()
        for b in bset:
            for i in rset:
                if layout.startswith("swmmac_a"):
                    for j in range(16):
                        lane, g, half = oracle.swmmac_src_pos(0, j, i)
                        seen_l.add(lane); seen_g.add(g)
                    continue
                if layout.startswith("swmmac_b"):
                    for j in range(16):
                        lane, g, half = oracle.swmmac_src_pos(1, j, i)
                        seen_l.add(lane); seen_g.add(g)
                    continue
                family = 1 if layout == "swmmac_d" else 0
                f64 = layout.startswith("f64")
                for j in range(M):
                    lane, g = oracle.tile_acc_pos(family, M, M, blocks, f64, i, j, b)
                    seen_l.add(lane); seen_g.add(g)
        assert seen_l == lset, (layout, rows, block)
        assert seen_g == gset, (layout, rows, block)


@pytest.mark.parametrize("family,M,blocks,f64,lanes", [(0, 32, 2, 0, 64), (0, 32, 1, 0, 64), (0, 16, 4, 0, 64),
                                                        (0, 4, 16, 0, 64), (0, 16, 1, 1, 64), (0, 4, 4, 1, 64),
                                                        (1, 16, 1, 0, 32)])
def test_layout_is_a_bijection(family, M, blocks, f64, lanes):
    """Each (lane, register) holds exactly one output element of one block."""
    seen = set()
    for b in range(blocks):
        for i in range(M):
            for j in range(M):
                lane, g = oracle.tile_acc_pos(family, M, M, blocks, f64, i, j, b)
                assert 0 <= lane < lanes
                seen.add((lane, g))
    assert len(seen) == blocks * M * M


def test_printed_inverse_formulas():
    """32x32: i = (8*floor(G/4)) mod 32 + 4*floor(L/32) + G mod 4, j = L mod 32, b = floor(G/16);
    16x16: i = 4*floor(L/16) + G mod 4, b = floor(G/4); 4x4: i = G, j = L mod 4, b = floor(L/4)."""
    for b in range(2):
        for i in range(32):
            for j in range(32):
                L, G = oracle.tile_acc_pos(0, 32, 32, 2, 0, i, j, b)
                assert (8 * (G // 4)) % 32 + 4 * (L // 32) + G % 4 == i and L % 32 == j and G // 16 == b
    for b in range(4):
        for i in range(16):
            for j in range(16):
                L, G = oracle.tile_acc_pos(0, 16, 16, 4, 0, i, j, b)
                assert 4 * (L // 16) + G % 4 == i and L % 16 == j and G // 4 == b
    for b in range(16):
        for i in range(4):
            for j in range(4):
                L, G = oracle.tile_acc_pos(0, 4, 4, 16, 0, i, j, b)
                assert G % 4 == i and L % 4 == j and L // 4 == b
    for i in range(16):
        for j in range(16):
            L, G = oracle.tile_acc_pos(1, 16, 16, 1, 0, i, j, 0)
            assert (L // 16) * 8 + G == i and L % 16 == j


def test_swmmac_a_and_b_groups_agree():
    """The lane group holding compressed A position k also holds the dense B rows that the
    2:4 index can select for it: rows 4*floor(k/2) .. 4*floor(k/2)+3."""
    for k in range(16):
        la, _, _ = oracle.swmmac_src_pos(0, 0, k)
        for r in range(4 * (k // 2), 4 * (k // 2) + 4):
            lb, _, _ = oracle.swmmac_src_pos(1, 0, r)
            assert la // 16 == lb // 16


# ---------------------------------------------------------------------------
# 2:4 compression
# ---------------------------------------------------------------------------
def test_sparse24_example_pattern():
    """The page's example keeps positions 0 and 2 of every group: metadata 0 | 2 << 2."""
    A = np.array([[0x38, 0, 0x40, 0, 0x44, 0, 0xB8, 0]], np.uint8)
    Ac, meta, v = oracle.sparse24_compress("e4m3", A)
    assert v == 0
    assert list(meta[0]) == [0b1000, 0b1000]
    assert list(Ac[0]) == [0x38, 0x40, 0x44, 0xB8]


def test_sparse24_padding_and_violations():
    A = np.array([[0, 0, 0, 0x38, 0, 0x80, 0x40, 0, 0x38, 0x38, 0x38, 0]], np.uint8)
    Ac, meta, v = oracle.sparse24_compress("e4m3", A)
    assert v == 1                                    # third group holds three nonzeros
    assert meta[0, 0] == (0 | 3 << 2)                # one nonzero at 3, padded with position 0
    assert meta[0, 1] == (0 | 2 << 2)                # -0 (0x80) counts as zero; pad with 0
    assert meta[0, 2] == (0 | 1 << 2)                # first two nonzeros kept
    # FNUZ: 0x80 is NaN, so it is a nonzero
    _, meta2, v2 = oracle.sparse24_compress("e4m3", A, fp8_enc="fnuz")
    assert meta2[0, 1] == (1 | 2 << 2)


def test_sparse24_compress_expand_identity():
    A, Bt, C = W.gen_sparse_e4m3(64, 8, 128, seed=4)
    Ac, meta, v = oracle.sparse24_compress("e4m3", A)
    assert v == 0
    E = np.zeros_like(A)
    for i in range(A.shape[0]):
        for g in range(A.shape[1] // 4):
            m = meta[i, g]
            E[i, 4 * g + (m & 3)] = Ac[i, 2 * g]
            E[i, 4 * g + ((m >> 2) & 3)] = Ac[i, 2 * g + 1]
    assert np.array_equal(E, A)


def test_sparse_gemm_equals_dense_gemm_on_expansion():
    """With one exact block per instruction, the chain over compressed terms equals the chain
    over the dense expansion (the zero products add nothing)."""
    A, Bt, C = W.gen_sparse_e4m3(16, 12, 96, seed=7, c_zero=False)
    Ac, meta, _ = oracle.sparse24_compress("e4m3", A)
    ii, jj = np.meshgrid(np.arange(16), np.arange(12), indexing="ij")
    sp = dict(fmt_a="e4m3", fmt_b="e4m3", arch="exact", n_fma=16, out_round="rne")
    dn = dict(sp, n_fma=32)
    d_sparse = oracle.sparse24_entries(sp, 96, 32, Ac, meta, Bt, C, ii.ravel(), jj.ravel())
    d_dense = oracle.gemm_entries(dn, 96, 32, A, Bt, C, ii.ravel(), jj.ravel())
    assert np.array_equal(d_sparse, d_dense)
    # and a wrong index (B row shifted) changes results
    bad = oracle.sparse24_entries(sp, 96, 32, Ac, (meta ^ 1).astype(np.uint8), Bt, C, ii.ravel(), jj.ravel())
    assert not np.array_equal(bad, d_dense)


# ---------------------------------------------------------------------------
# multi-word split
# ---------------------------------------------------------------------------
def _bf16_value(w):
    import struct
    return Fraction(struct.unpack("<f", struct.pack("<I", int(w) << 16))[0])


def test_multiword_split_is_successive_rne():
    A, _ = W.gen_multiword_fp64(64, 1, 64, seed=5)
    x = A.ravel()
    w = oracle.split_bf16(x, 3)
    for t in range(x.size):
        r = Fraction(float(x[t]))
        for k in range(3):
            v = _bf16_value(w[k, t])
            # v is the bf16 value nearest to r (ties to even significand)
            e = abs(r).numerator.bit_length() - abs(r).denominator.bit_length()
            if Fraction(2) ** e > abs(r):
                e -= 1
            ulp = Fraction(2) ** (max(e, -126) - 7)
            assert abs(r - v) <= ulp / 2
            if abs(r - v) == ulp / 2:
                assert (int(w[k, t]) & 1) == 0
            r -= v
        # x = x1 + x2 + x3 + r with |r| <= 2^-24 |x|
        assert abs(r) <= Fraction(2) ** -24 * abs(Fraction(float(x[t])))


def test_multiword_combine_order_and_products():
    """With an exact word model each word GEMM entry is the correctly rounded exact sum; the
    words are summed in binary64, i+j descending then i ascending; the truncated set keeps
    i+j <= 4."""
    import exact_spec
    A, Bt = W.gen_multiword_fp64(3, 2, 40, seed=6)
    wm = dict(fmt_a="bf16", fmt_b="bf16", arch="exact", n_fma=40, out_round="rne")
    for truncated in (False, True):
        got = oracle.multiword_entries(wm, 0, 3, truncated, A, Bt, [0, 1, 2, 0], [0, 1, 0, 1])
        for e, (i, j) in enumerate([(0, 0), (1, 1), (2, 0), (0, 1)]):
            aw = oracle.split_bf16(A[i], 3)
            bw = oracle.split_bf16(Bt[j], 3)
            D = 0.0
            for s in range(6, 1, -1):
                for wi in range(1, 4):
                    wj = s - wi
                    if not 1 <= wj <= 3 or (truncated and wi + wj > 4):
                        continue
                    exact = sum(_bf16_value(aw[wi - 1, k]) * _bf16_value(bw[wj - 1, k]) for k in range(40))
                    d32 = exact_spec.round_fp32(exact)
                    D = D + float(np.uint32(d32).view(np.float32))
            assert got[e] == D

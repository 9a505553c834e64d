"""The C ABI without a GPU: the library builds, loads, exports every function that
include/mcemu.h declares, validates models, and its host-side tile helpers and presets
agree with the oracle's independent versions."""
import ctypes
import os
import re
import subprocess

import pytest

import oracle
from oracle.presets import PRESETS
from bit_exact_emulation_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mcemu.h")


@pytest.fixture(scope="module")
def L():
    B.build()
    from bit_exact_emulation_gb300 import binding
    return binding


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mcemu_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("mcemu_model_create", "mcemu_block_fma", "mcemu_tile_gemm", "mcemu_sparse24_compress",
                 "mcemu_sparse24_gemm", "mcemu_multiword_gemm"):
        assert must in names


def test_library_exports_every_declared_symbol(L):
    lib = L.lib()
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (mcemu_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert getattr(lib, n) is not None
    assert set(L.SYMBOLS) == set(declared_functions())


def test_status_strings(L):
    lib = L.lib()
    assert lib.mcemu_status_string(0) == b"ok"
    assert lib.mcemu_status_string(3) == b"not 2:4 sparse"
    assert lib.mcemu_version() >= 10000


# presets: the library's copy (C) against the oracle's copy (Python), both from the paper
_FIELD = {"arch": "arch", "n_fma": "block_k", "align_frac": "align_frac_bits"}


@pytest.mark.parametrize("name", [n for n in PRESETS])
def test_presets_agree_with_oracle(L, name):
    got = L.preset_desc(name)
    want = L.desc_from_spec(PRESETS[name])
    for f, _ in L.ModelDesc._fields_:
        if f in ("align_frac_bits", "align_round", "c_frac_bits", "psum_frac_bits", "post_norm_frac_bits",
                 "pair_group") and PRESETS[name]["arch"] in ("exact", "pairwise"):
            continue          # unused by those architectures
        if f == "c_zero_exp" and PRESETS[name]["arch"] in ("exact", "pairwise"):
            continue
        assert getattr(got, f) == getattr(want, f), (name, f)


@pytest.mark.parametrize("name,fmt,k", [("ga_trunc", "fp16", 4), ("ga_rne", "bf16", 4), ("ieee_exact", "e4m3", 8)])
def test_workload_presets(L, name, fmt, k):
    from oracle.presets import block_models
    got = L.preset_desc(name, fmt, k)
    want = L.desc_from_spec(block_models(fmt, k)[name])
    for f in ("fmt_a", "arch", "block_k", "out_round", "c_zero_exp", "emin_lim", "prod_overflow_2p128"):
        assert getattr(got, f) == getattr(want, f), f
    if name != "ieee_exact":
        assert got.align_frac_bits == 26 and got.align_round == 0


def test_model_validation(L):
    good = dict(PRESETS["cdna3_bf16"])
    L.Model(good)
    for bad, status in ((dict(good, n_fma=0), 1), (dict(good, n_fma=33), 1), (dict(good, align_frac=60), 2),
                        (dict(good, c_frac=23), 2), (dict(good, fmt_b="int8"), 1),
                        (dict(good, fmt_b="fp16"), 0), (dict(good, fmt_b="e4m3"), 2)):
        if status == 0:
            L.Model(bad)
            continue
        with pytest.raises(L.McemuError) as e:
            L.Model(bad)
        assert e.value.status == status
    d = L.desc_from_spec(good)
    d.struct_size = 4
    with pytest.raises(L.McemuError):
        L.Model(d)
    d = L.desc_from_spec(good)
    d.acc_sig_bits = 11
    with pytest.raises(L.McemuError) as e:
        L.Model(d)
    assert e.value.status == 2


def test_null_arguments_are_rejected(L):
    lib = L.lib()
    m = L.Model(PRESETS["cdna3_fp16"])
    assert lib.mcemu_block_fma(m.handle, 10, None, None, None, None, None) == 1
    assert lib.mcemu_block_fma(m.handle, 0, None, None, None, None, None) == 0      # n = 0: no-op
    assert lib.mcemu_model_create(None, None) == 1
    t = L.tile(0, 32, 32, 8, 4)
    assert lib.mcemu_tile_gemm(None, ctypes.byref(t), 4, 4, 4, None, 4, None, 4, None, 4, None, 4, None) == 1
    assert lib.mcemu_sparse24_compress(4, 0, 4, 6, None, 6, None, 3, None, 1, None, None) == 1   # K % 4
    assert lib.mcemu_multiword_gemm(m.handle, ctypes.byref(t), 3, 0, 4, 4, 4, None, 4, None, 4, None, 4,
                                    None, 0, None) == 2                                       # fp16 words
    assert lib.mcemu_multiword_workspace(3, 4096, 4096, 4096) == 3 * 2 * 4096 * 4096 * 2 + 4096 * 4096 * 4


def test_tile_info_matches_oracle(L):
    for fam, M, N, K, epl in ((0, 32, 32, 8, 4), (0, 16, 16, 16, 4), (0, 4, 4, 4, 4), (0, 32, 32, 1, 1),
                              (0, 16, 16, 8, 2), (0, 32, 32, 16, 8), (1, 16, 16, 32, 8)):
        assert L.tile_info(L.tile(fam, M, N, K, epl)) == oracle.tile_blocks(fam, M, N, K, epl)


@pytest.mark.parametrize("fam,M,K,epl,f64", [(0, 32, 8, 4, 0), (0, 32, 1, 1, 0), (0, 16, 4, 4, 0), (0, 4, 4, 4, 0),
                                             (0, 16, 4, 1, 1), (0, 4, 4, 1, 1), (1, 16, 32, 8, 0)])
def test_tile_layout_matches_oracle(L, fam, M, K, epl, f64):
    t = L.tile(fam, M, M, K, epl)
    blocks = (4 if M == 4 else 1) if f64 else L.tile_info(t)[0]
    for b in range(blocks):
        for i in range(M):
            for j in range(M):
                lane, reg = L.tile_layout(t, f64, i, j, b)
                assert (lane, reg) == oracle.tile_acc_pos(fam, M, M, blocks, f64, i, j, b)
                assert L.tile_layout_inverse(t, f64, lane, reg) == (i, j, b)


def test_swmmac_src_layout_matches_oracle(L):
    for op, kmax in ((0, 16), (1, 32)):
        for idx in range(16):
            for k in range(kmax):
                assert L.swmmac_src_layout(op, idx, k) == oracle.swmmac_src_pos(op, idx, k)


def test_static_scratch_entry_without_a_device(L):
    """On a host without a GPU the no-allocation multi-word entry point's first call
    (the per-device lookup of its scratch array) returns MCEMU_ERR_CUDA; nothing is
    launched.  Skipped where a GPU is present (these are host buffers)."""
    import numpy as np
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    m = L.Model(PRESETS["cdna3_bf16"])
    A = np.zeros((4, 8))
    B = np.zeros((4, 8))
    D = np.zeros((4, 4))
    t = L.tile(0, 32, 32, 8, 4)
    p = lambda x: ctypes.c_void_p(x.ctypes.data)
    st = L.lib().mcemu_multiword_gemm_static(m.handle, ctypes.byref(t), 3, 0, 4, 4, 8, p(A), 8, p(B), 8, p(D), 4,
                                             None)
    assert st == 5                               # MCEMU_ERR_CUDA

"""CPU oracle for bit-exact matrix-multiplier emulation -- TEST INFRASTRUCTURE ONLY.

A plain, slow, exact model (C source in ``orc.c``) of the block fused
multiply-add d = sum_l a_l*b_l + c of "Accurate Models of AMD Matrix Cores"
(Sec. 2, eq. (1)) and of the tile/2:4/multi-word GEMM drivers built on it.
Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` leg of
``bench.py`` may import this package; the product path never does.  It shares
no code with the CUDA library: models are described to it by name (see
``presets.py``) and translated here into its own C structure.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from .build import build_oracle, LIB_PATH
from . import presets

__all__ = ["Model", "block_fma", "block_fma_parallel", "gemm_entries", "sparse24_compress",
           "sparse24_entries", "split_bf16", "multiword_entries", "tile_blocks",
           "tile_acc_pos", "swmmac_src_pos", "presets", "FORMATS", "ELEM_DTYPE"]

FORMATS = {"fp16": 0, "bf16": 1, "xf32": 2, "fp32": 3, "e4m3": 4, "e5m2": 5, "int8": 6, "uint8": 7}
ELEM_DTYPE = {"fp16": np.uint16, "bf16": np.uint16, "xf32": np.uint32, "fp32": np.uint32,
              "e4m3": np.uint8, "e5m2": np.uint8, "int8": np.uint8, "uint8": np.uint8}
_ARCH = {"exact": 0, "ga_early": 1, "ga_late": 2, "odd_even": 3, "pairwise": 4}
_NO_EXP = -(2 ** 31)


class Model(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "fmt_a", "fmt_b", "fp8_enc", "xf32_round", "arch", "n_fma", "align_frac", "align_round",
        "c_frac", "psum_frac", "post_norm_frac", "out_round", "sub_in", "sub_out",
        "c_zero_exp", "emin_lim", "prod_ovf")] + [("nan_bits", ctypes.c_uint32),
                                                  ("int_sat", ctypes.c_int32),
                                                  ("pair_group", ctypes.c_int32),
                                                  ("acc_fmt", ctypes.c_int32)]

    @classmethod
    def from_spec(cls, spec: dict) -> "Model":
        """Translate a model described by name (see presets.py) into the C struct."""
        m = cls()
        m.fmt_a = FORMATS[spec["fmt_a"]]
        m.fmt_b = FORMATS[spec["fmt_b"]]
        m.fp8_enc = {"ocp": 0, "fnuz": 1}[spec.get("fp8_enc", "ocp")]
        m.xf32_round = {"trunc": 0, "rne": 1}[spec.get("xf32_round", "trunc")]
        m.arch = _ARCH[spec["arch"]]
        m.n_fma = int(spec["n_fma"])
        m.align_frac = int(spec.get("align_frac", 24))
        m.align_round = {"rz": 0, "rd": 1}[spec.get("align_round", "rz")]
        m.c_frac = int(spec.get("c_frac", 24))
        m.psum_frac = int(spec.get("psum_frac", 32))
        m.post_norm_frac = int(spec.get("post_norm_frac", 31))
        m.out_round = {"rne": 0, "rtz": 1}[spec.get("out_round", "rne")]
        m.sub_in = int(bool(spec.get("sub_in_flush", False)))
        m.sub_out = int(bool(spec.get("sub_out_flush", False)))
        cz = spec.get("c_zero_exp", None)
        m.c_zero_exp = _NO_EXP if cz is None else int(cz)
        el = spec.get("emin_lim", None)
        m.emin_lim = _NO_EXP if el is None else int(el)
        m.prod_ovf = int(bool(spec.get("prod_overflow", False)))
        m.nan_bits = int(spec.get("nan_bits", 0x7FC00000))
        m.int_sat = int(bool(spec.get("int_saturate", False)))
        m.pair_group = int(spec.get("pair_group", spec["n_fma"]))
        m.acc_fmt = {"fp32": 0, "fp16": 1}[spec.get("acc_fmt", "fp32")]
        return m


_lib = None
_lib_lock = threading.Lock()


def _load():
    global _lib
    with _lib_lock:
        if _lib is None:
            build_oracle()      # rebuilds only when orc.c is newer than the library
            lib = ctypes.CDLL(LIB_PATH)
            P = ctypes.c_void_p
            i32, i64 = ctypes.c_int32, ctypes.c_int64
            lib.orc_block_fma.argtypes = [P, i64, P, P, P, P]
            lib.orc_block_fma_n.argtypes = [P, i64, i32, P, P, P, P]
            lib.orc_gemm_entries.argtypes = [P, i32, i32, P, i64, P, i64, P, i64, i64, P, P, P]
            lib.orc_sparse24_compress.argtypes = [i32, i32, i32, i32, P, i64, P, i64, P, i64]
            lib.orc_sparse24_compress.restype = i64
            lib.orc_sparse24_entries.argtypes = [P, i32, i32, P, i64, P, i64, P, i64, P, i64, i64,
                                                 P, P, P]
            lib.orc_split_bf16.argtypes = [i64, i32, P, P]
            lib.orc_multiword_entries.argtypes = [P, i32, i32, i32, i32, P, i64, P, i64, i64, P, P, P]
            lib.orc_tile_blocks.argtypes = [i32] * 5 + [P, P]
            lib.orc_tile_acc_pos.argtypes = [i32] * 8 + [P, P]
            lib.orc_swmmac_src_pos.argtypes = [i32] * 3 + [P, P, P]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _model(spec) -> Model:
    return spec if isinstance(spec, Model) else Model.from_spec(spec)


def block_fma(spec, a: np.ndarray, b: np.ndarray, c: np.ndarray, n_terms: int | None = None) -> np.ndarray:
    """One block FMA per row: a, b are [n][n_terms] element bit patterns, c is [n] uint32."""
    m = _model(spec)
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b)
    c = np.ascontiguousarray(c, dtype=np.uint32)
    n = c.shape[0]
    nt = m.n_fma if n_terms is None else int(n_terms)
    assert a.size == n * nt and b.size == n * nt
    d = np.empty(n, dtype=np.uint32)
    rc = _load().orc_block_fma_n(ctypes.byref(m), n, nt, _ptr(a), _ptr(b), _ptr(c), _ptr(d))
    if rc != 0:
        raise ValueError(f"oracle rejected the model or sizes (rc={rc})")
    return d


def block_fma_parallel(spec, a, b, c, threads: int) -> np.ndarray:
    """block_fma split over `threads` host threads (the C call releases the GIL)."""
    n = c.shape[0]
    if threads <= 1 or n < 2 * threads:
        return block_fma(spec, a, b, c)
    out = np.empty(n, dtype=np.uint32)
    bounds = np.linspace(0, n, threads + 1).astype(np.int64)

    def work(t):
        lo, hi = bounds[t], bounds[t + 1]
        out[lo:hi] = block_fma(spec, a[lo:hi], b[lo:hi], c[lo:hi])

    ts = [threading.Thread(target=work, args=(t,)) for t in range(threads)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    return out


def gemm_entries(spec, K, kt, A, Bt, C, ii, jj) -> np.ndarray:
    """Entries D[ii[e], jj[e]] of the emulated GEMM D = A @ B + C (Bt = B^T, [N][K])."""
    m = _model(spec)
    A = np.ascontiguousarray(A)
    Bt = np.ascontiguousarray(Bt)
    C = np.ascontiguousarray(C, dtype=np.uint32)
    ii = np.ascontiguousarray(ii, dtype=np.int32)
    jj = np.ascontiguousarray(jj, dtype=np.int32)
    out = np.empty(ii.shape[0], dtype=np.uint32)
    rc = _load().orc_gemm_entries(ctypes.byref(m), int(K), int(kt), _ptr(A), A.shape[1], _ptr(Bt),
                                  Bt.shape[1], _ptr(C), C.shape[1], ii.shape[0], _ptr(ii), _ptr(jj),
                                  _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle gemm failed (rc={rc})")
    return out


def sparse24_compress(fmt: str, A: np.ndarray, fp8_enc: str = "ocp"):
    """2:4 compression of A [M][K]; returns (Ac [M][K/2], meta [M][K/4] uint8, violations)."""
    A = np.ascontiguousarray(A)
    M, K = A.shape
    Ac = np.zeros((M, K // 2), dtype=A.dtype)
    meta = np.zeros((M, K // 4), dtype=np.uint8)
    v = _load().orc_sparse24_compress(FORMATS[fmt], {"ocp": 0, "fnuz": 1}[fp8_enc], M, K, _ptr(A),
                                      K, _ptr(Ac), K // 2, _ptr(meta), K // 4)
    if v < 0:
        raise ValueError("oracle sparse24_compress rejected the input")
    return Ac, meta, int(v)


def sparse24_entries(spec, K, kt, Ac, meta, Bt, C, ii, jj) -> np.ndarray:
    m = _model(spec)
    Ac = np.ascontiguousarray(Ac)
    meta = np.ascontiguousarray(meta, dtype=np.uint8)
    Bt = np.ascontiguousarray(Bt)
    C = np.ascontiguousarray(C, dtype=np.uint32)
    ii = np.ascontiguousarray(ii, dtype=np.int32)
    jj = np.ascontiguousarray(jj, dtype=np.int32)
    out = np.empty(ii.shape[0], dtype=np.uint32)
    rc = _load().orc_sparse24_entries(ctypes.byref(m), int(K), int(kt), _ptr(Ac), Ac.shape[1],
                                      _ptr(meta), meta.shape[1], _ptr(Bt), Bt.shape[1], _ptr(C),
                                      C.shape[1], ii.shape[0], _ptr(ii), _ptr(jj), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle sparse gemm failed (rc={rc})")
    return out


def split_bf16(x: np.ndarray, n_words: int) -> np.ndarray:
    """Multi-word split of binary64 x into [n_words][x.size] bf16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float64).reshape(-1)
    w = np.empty((n_words, x.size), dtype=np.uint16)
    rc = _load().orc_split_bf16(x.size, n_words, _ptr(x), _ptr(w))
    if rc != 0:
        raise ValueError("oracle split rejected the word count")
    return w


def multiword_entries(spec, kt, n_words, truncated, A, Bt, ii, jj) -> np.ndarray:
    m = _model(spec)
    A = np.ascontiguousarray(A, dtype=np.float64)
    Bt = np.ascontiguousarray(Bt, dtype=np.float64)
    ii = np.ascontiguousarray(ii, dtype=np.int32)
    jj = np.ascontiguousarray(jj, dtype=np.int32)
    out = np.empty(ii.shape[0], dtype=np.float64)
    rc = _load().orc_multiword_entries(ctypes.byref(m), int(kt), int(n_words), int(bool(truncated)),
                                       A.shape[1], _ptr(A), A.shape[1], _ptr(Bt), Bt.shape[1],
                                       ii.shape[0], _ptr(ii), _ptr(jj), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle multiword failed (rc={rc})")
    return out


def tile_blocks(family: int, M: int, N: int, K: int, elems_per_lane: int):
    b, r = ctypes.c_int32(), ctypes.c_int32()
    rc = _load().orc_tile_blocks(family, M, N, K, elems_per_lane, ctypes.byref(b), ctypes.byref(r))
    if rc != 0:
        raise ValueError("oracle: not a valid tile")
    return b.value, r.value


def tile_acc_pos(family: int, M: int, N: int, blocks: int, f64: bool, i: int, j: int, b: int):
    lane, reg = ctypes.c_int32(), ctypes.c_int32()
    rc = _load().orc_tile_acc_pos(family, M, N, blocks, int(f64), i, j, b, ctypes.byref(lane),
                                  ctypes.byref(reg))
    if rc != 0:
        raise ValueError("oracle: no such accumulator position")
    return lane.value, reg.value


def swmmac_src_pos(operand: int, idx: int, k: int):
    """(lane, vgpr, half) of compressed A (operand 0) or dense B (operand 1) element k."""
    lane, vgpr, half = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    rc = _load().orc_swmmac_src_pos(operand, idx, k, ctypes.byref(lane), ctypes.byref(vgpr),
                                    ctypes.byref(half))
    if rc != 0:
        raise ValueError("oracle: no such source position")
    return lane.value, vgpr.value, half.value

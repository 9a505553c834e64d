"""Python binding of libmcemu.so: argument marshalling only.

Every computation happens in the CUDA library (C ABI in include/mcemu.h).  Device
buffers are torch CUDA tensors whose raw bytes are the element bit patterns (any
dtype of the right element size); results are int32 tensors holding fp32/int32 bit
patterns.  Calls run on torch's current CUDA stream.  If the library has not been
built, every entry point raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

FMT = {"fp16": 0, "bf16": 1, "xf32": 2, "fp32": 3, "e4m3": 4, "e5m2": 5, "int8": 6, "uint8": 7}
ELEM_BYTES = {"fp16": 2, "bf16": 2, "xf32": 4, "fp32": 4, "e4m3": 1, "e5m2": 1, "int8": 1, "uint8": 1}
ARCH = {"exact": 0, "ga_early": 1, "ga_late": 2, "odd_even": 3, "pairwise": 4}
NO_EXP = -(2 ** 31)
PRESET = {"cdna3_fp16": 0, "cdna3_bf16": 1, "cdna3_xf32": 2, "cdna3_fp8": 3, "cdna3_bf8": 4,
          "cdna1_fp16": 5, "cdna1_bf16": 6, "cdna1_fp32": 7, "cdna2_fp16": 8, "cdna2_bf16_1k": 9,
          "cdna2_bf16": 10, "b200_fp16": 11, "h100_fp16": 12, "a100_fp16": 13, "b200_bf16": 14,
          "a100_bf16": 15, "b200_tf19": 16, "a100_tf19": 17, "b200_fp8": 18, "h100_fp8": 19,
          "b200_fp16_f16": 20, "h100_fp16_f16": 21, "a100_fp16_f16": 22, "b200_fp8_f16": 23,
          "h100_fp8_f16": 24, "ga_trunc": 100, "ga_rne": 101, "ieee_exact": 102}
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "not 2:4 sparse", 4: "alignment",
          5: "CUDA error", 6: "timeout", 7: "workspace too small"}
FRO_OUT_DOUBLES = 1026
MULTIWORD_STATIC_BYTES = 8 << 20      # MCEMU_MULTIWORD_STATIC_BYTES


class McemuError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: mcemu status {status} ({STATUS.get(status, '?')})")
        self.status = status


class ModelDesc(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_uint32)] + [(n, ctypes.c_int32) for n in (
        "fmt_a", "fmt_b", "fp8_enc", "xf32_round", "arch", "block_k", "align_frac_bits",
        "align_round", "c_frac_bits", "psum_frac_bits", "post_norm_frac_bits", "acc_sig_bits",
        "out_round", "subnormal_in_flush", "subnormal_out_flush", "c_zero_exp", "emin_lim",
        "prod_overflow_2p128")] + [("nan_bits", ctypes.c_uint32), ("int_saturate", ctypes.c_int32),
                                   ("pair_group", ctypes.c_int32)]


class TileDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("family", "M", "N", "K", "elems_per_lane")]


_lib = None
SYMBOLS = {
    # name: (restype, argtypes)
    "mcemu_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "mcemu_version": (ctypes.c_int, []),
    "mcemu_model_preset": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
    "mcemu_model_create": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "mcemu_model_destroy": (None, [ctypes.c_void_p]),
    "mcemu_model_get_desc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "mcemu_block_fma": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t] + [ctypes.c_void_p] * 5),
    "mcemu_block_fma_host": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t] + [ctypes.c_void_p] * 5
                             + [ctypes.c_size_t, ctypes.c_void_p]),
    "mcemu_block_fma_host_workspace": (ctypes.c_size_t, [ctypes.c_void_p]),
    "mcemu_tile_info": (ctypes.c_int, [ctypes.c_void_p] * 3),
    "mcemu_tile_layout": (ctypes.c_int, [ctypes.c_void_p] + [ctypes.c_int] * 4 + [ctypes.c_void_p] * 2),
    "mcemu_tile_layout_inverse": (ctypes.c_int, [ctypes.c_void_p] + [ctypes.c_int] * 3 + [ctypes.c_void_p] * 3),
    "mcemu_swmmac_src_layout": (ctypes.c_int, [ctypes.c_int] * 3 + [ctypes.c_void_p] * 3),
    "mcemu_tile_gemm": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p] + [ctypes.c_int] * 3
                        + [ctypes.c_void_p, ctypes.c_int64] * 4 + [ctypes.c_void_p]),
    "mcemu_sparse24_compress": (ctypes.c_int, [ctypes.c_int] * 4 + [ctypes.c_void_p, ctypes.c_int64] * 3
                                + [ctypes.c_void_p, ctypes.c_void_p]),
    "mcemu_sparse24_check": (ctypes.c_int, [ctypes.c_void_p] * 3),
    "mcemu_sparse24_expand": (ctypes.c_int, [ctypes.c_int] * 3 + [ctypes.c_void_p, ctypes.c_int64] * 3
                              + [ctypes.c_void_p]),
    "mcemu_sparse24_gemm": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p] + [ctypes.c_int] * 3
                            + [ctypes.c_void_p, ctypes.c_int64] * 5 + [ctypes.c_void_p]),
    "mcemu_multiword_split": (ctypes.c_int, [ctypes.c_int, ctypes.c_size_t] + [ctypes.c_void_p] * 3),
    "mcemu_multiword_workspace": (ctypes.c_size_t, [ctypes.c_int] * 4),
    "mcemu_multiword_gemm": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p] + [ctypes.c_int] * 5
                             + [ctypes.c_void_p, ctypes.c_int64] * 3
                             + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "mcemu_multiword_gemm_static": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p] + [ctypes.c_int] * 5
                                    + [ctypes.c_void_p, ctypes.c_int64] * 3 + [ctypes.c_void_p]),
    "mcemu_fro_error": (ctypes.c_int, [ctypes.c_int] * 2 + [ctypes.c_void_p, ctypes.c_int64] * 2
                        + [ctypes.c_void_p, ctypes.c_void_p]),
}


def lib():
    """The loaded library; raises when it has not been built (no fallback exists)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with bit_exact_emulation_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SYMBOLS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(st: int, where: str):
    if st != 0:
        raise McemuError(st, where)


# ---------------------------------------------------------------------------
# models
# ---------------------------------------------------------------------------
def desc_from_spec(spec: dict) -> ModelDesc:
    """Model description from the named-feature dict used across the project
    (keys: fmt_a, fmt_b, fp8_enc, xf32_round, arch, n_fma, align_frac, align_round,
    c_frac, psum_frac, post_norm_frac, out_round, sub_in_flush, sub_out_flush,
    c_zero_exp, emin_lim, prod_overflow, nan_bits, int_saturate, pair_group, acc_fmt)."""
    d = ModelDesc()
    d.struct_size = ctypes.sizeof(ModelDesc)
    d.fmt_a, d.fmt_b = FMT[spec["fmt_a"]], FMT[spec["fmt_b"]]
    d.fp8_enc = {"ocp": 0, "fnuz": 1}[spec.get("fp8_enc", "ocp")]
    d.xf32_round = {"trunc": 0, "rne": 1}[spec.get("xf32_round", "trunc")]
    d.arch = ARCH[spec.get("arch", "exact")]
    d.block_k = int(spec["n_fma"])
    d.align_frac_bits = int(spec.get("align_frac", 24))
    d.align_round = {"rz": 0, "rd": 1}[spec.get("align_round", "rz")]
    d.c_frac_bits = int(spec.get("c_frac", 24))
    d.psum_frac_bits = int(spec.get("psum_frac", 32))
    d.post_norm_frac_bits = int(spec.get("post_norm_frac", 31))
    d.acc_sig_bits = {"fp32": 24, "fp16": 11}[spec.get("acc_fmt", "fp32")]
    d.out_round = {"rne": 0, "rtz": 1}[spec.get("out_round", "rne")]
    d.subnormal_in_flush = int(bool(spec.get("sub_in_flush", False)))
    d.subnormal_out_flush = int(bool(spec.get("sub_out_flush", False)))
    cz = spec.get("c_zero_exp", None)
    d.c_zero_exp = NO_EXP if cz is None else int(cz)
    el = spec.get("emin_lim", None)
    d.emin_lim = NO_EXP if el is None else int(el)
    d.prod_overflow_2p128 = int(bool(spec.get("prod_overflow", False)))
    d.nan_bits = int(spec.get("nan_bits", 0x7FC00000))
    d.int_saturate = int(bool(spec.get("int_saturate", False)))
    d.pair_group = int(spec.get("pair_group", spec["n_fma"]))
    return d


def preset_desc(name: str, fmt: str | None = None, k: int = 0) -> ModelDesc:
    d = ModelDesc()
    _check(lib().mcemu_model_preset(PRESET[name], FMT[fmt] if fmt else -1, k, ctypes.byref(d)),
           f"preset {name}")
    return d


class Model:
    """A validated model handle (owned by the library, freed with the object)."""

    def __init__(self, spec_or_desc):
        desc = spec_or_desc if isinstance(spec_or_desc, ModelDesc) else desc_from_spec(spec_or_desc)
        h = ctypes.c_void_p()
        _check(lib().mcemu_model_create(ctypes.byref(desc), ctypes.byref(h)), "mcemu_model_create")
        self.handle = h
        self.desc = desc

    def __del__(self):
        h = getattr(self, "handle", None)
        if h and _lib is not None:
            _lib.mcemu_model_destroy(h)
            self.handle = None


# ---------------------------------------------------------------------------
# compute entry points (torch CUDA tensors)
# ---------------------------------------------------------------------------
def _stream():
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def block_fma(model: Model, a, b, c, d=None):
    """d[v] = model(a[v], b[v], c[v]); a, b [n][k] elements, c [n] 32-bit patterns."""
    import torch
    n = c.numel()
    if d is None:
        d = torch.empty(n, dtype=torch.int32, device=c.device)
    _check(lib().mcemu_block_fma(model.handle, n, _p(a), _p(b), _p(c), _p(d), _stream()), "mcemu_block_fma")
    return d


def block_fma_host(model: Model, a, b, c, d, workspace):
    """Host-buffer variant: a, b, c, d are CPU tensors (pinned for overlap); synchronous."""
    ws = workspace
    _check(lib().mcemu_block_fma_host(model.handle, c.numel(), _p(a), _p(b), _p(c), _p(d), _p(ws),
                                      ws.numel() * ws.element_size(), _stream()), "mcemu_block_fma_host")
    return d


def block_fma_host_workspace(model: Model) -> int:
    return int(lib().mcemu_block_fma_host_workspace(model.handle))


def tile(family: int, M: int, N: int, K: int, elems_per_lane: int = 4) -> TileDesc:
    return TileDesc(family, M, N, K, elems_per_lane)


def tile_gemm(model: Model, t: TileDesc, A, Bt, C, D=None):
    """D = A @ B + C (Bt = B^T [N][K]); 32-bit patterns in C and D."""
    import torch
    M, K = A.shape
    N = Bt.shape[0]
    if D is None:
        D = torch.empty((M, N), dtype=torch.int32, device=A.device)
    _check(lib().mcemu_tile_gemm(model.handle, ctypes.byref(t), M, N, K, _p(A), A.stride(0), _p(Bt),
                                 Bt.stride(0), _p(C), C.stride(0), _p(D), D.stride(0), _stream()),
           "mcemu_tile_gemm")
    return D


def sparse24_compress(fmt: str, A, fp8_enc: str = "ocp", check: bool = False):
    """(Ac [M][K/2], meta [M][K/4] uint8, violations int64 tensor on the device).
    With check=True the call waits for the stream and raises McemuError with status
    MCEMU_ERR_NOT_2_4 (3) when a group of four held more than two nonzeros."""
    import torch
    M, K = A.shape
    Ac = torch.empty((M, K // 2), dtype=A.dtype, device=A.device)
    meta = torch.empty((M, K // 4), dtype=torch.uint8, device=A.device)
    viol = torch.zeros(1, dtype=torch.int64, device=A.device)
    _check(lib().mcemu_sparse24_compress(FMT[fmt], {"ocp": 0, "fnuz": 1}[fp8_enc], M, K, _p(A), A.stride(0),
                                         _p(Ac), Ac.stride(0), _p(meta), meta.stride(0), _p(viol),
                                         _stream()), "mcemu_sparse24_compress")
    if check:
        _check(lib().mcemu_sparse24_check(_p(viol), None, _stream()), "mcemu_sparse24_check")
    return Ac, meta, viol


def sparse24_expand(fmt: str, Ac, meta, K: int):
    import torch
    M = Ac.shape[0]
    A = torch.empty((M, K), dtype=Ac.dtype, device=Ac.device)
    _check(lib().mcemu_sparse24_expand(FMT[fmt], M, K, _p(Ac), Ac.stride(0), _p(meta), meta.stride(0), _p(A),
                                       A.stride(0), _stream()), "mcemu_sparse24_expand")
    return A


def sparse24_gemm(model: Model, t: TileDesc, Ac, meta, Bt, C, D=None):
    import torch
    M = Ac.shape[0]
    K = Ac.shape[1] * 2
    N = Bt.shape[0]
    if D is None:
        D = torch.empty((M, N), dtype=torch.int32, device=Ac.device)
    _check(lib().mcemu_sparse24_gemm(model.handle, ctypes.byref(t), M, N, K, _p(Ac), Ac.stride(0), _p(meta),
                                     meta.stride(0), _p(Bt), Bt.stride(0), _p(C), C.stride(0), _p(D),
                                     D.stride(0), _stream()), "mcemu_sparse24_gemm")
    return D


def multiword_split(x, n_words: int):
    import torch
    w = torch.empty((n_words, x.numel()), dtype=torch.int16, device=x.device)
    _check(lib().mcemu_multiword_split(n_words, x.numel(), _p(x), _p(w), _stream()), "mcemu_multiword_split")
    return w


def multiword_workspace(n_words: int, M: int, N: int, K: int) -> int:
    return int(lib().mcemu_multiword_workspace(n_words, M, N, K))


def multiword_gemm(model: Model, t: TileDesc, n_words: int, truncated: bool, A, Bt, D=None, workspace=None):
    import torch
    M, K = A.shape
    N = Bt.shape[0]
    if D is None:
        D = torch.empty((M, N), dtype=torch.float64, device=A.device)
    if workspace is None:
        workspace = torch.empty(multiword_workspace(n_words, M, N, K), dtype=torch.uint8, device=A.device)
    _check(lib().mcemu_multiword_gemm(model.handle, ctypes.byref(t), n_words, int(bool(truncated)), M, N, K,
                                      _p(A), A.stride(0), _p(Bt), Bt.stride(0), _p(D), D.stride(0),
                                      _p(workspace), workspace.numel() * workspace.element_size(),
                                      _stream()), "mcemu_multiword_gemm")
    return D


def multiword_gemm_static(model: Model, t: TileDesc, n_words: int, truncated: bool, A, Bt, D=None):
    """mcemu_multiword_gemm_static: the multi-word GEMM with the library's fixed scratch."""
    import torch
    M, K = A.shape
    N = Bt.shape[0]
    if D is None:
        D = torch.empty((M, N), dtype=torch.float64, device=A.device)
    _check(lib().mcemu_multiword_gemm_static(model.handle, ctypes.byref(t), n_words, int(bool(truncated)), M, N,
                                             K, _p(A), A.stride(0), _p(Bt), Bt.stride(0), _p(D), D.stride(0),
                                             _stream()), "mcemu_multiword_gemm_static")
    return D


def fro_error(D, R, out=None):
    """Device tensor [2]: sum (D-R)^2 and sum R^2 (binary64, fixed summation order)."""
    import torch
    if out is None:
        out = torch.empty(FRO_OUT_DOUBLES, dtype=torch.float64, device=D.device)
    M, N = D.shape
    _check(lib().mcemu_fro_error(M, N, _p(D), D.stride(0), _p(R), R.stride(0), _p(out), _stream()),
           "mcemu_fro_error")
    return out[:2]


# ---------------------------------------------------------------------------
# tile semantics helpers (host)
# ---------------------------------------------------------------------------
def tile_info(t: TileDesc):
    b, r = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().mcemu_tile_info(ctypes.byref(t), ctypes.byref(b), ctypes.byref(r)), "mcemu_tile_info")
    return b.value, r.value


def tile_layout(t: TileDesc, f64: bool, i: int, j: int, b: int):
    lane, reg = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().mcemu_tile_layout(ctypes.byref(t), int(f64), i, j, b, ctypes.byref(lane), ctypes.byref(reg)),
           "mcemu_tile_layout")
    return lane.value, reg.value


def tile_layout_inverse(t: TileDesc, f64: bool, lane: int, reg: int):
    i, j, b = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check(lib().mcemu_tile_layout_inverse(ctypes.byref(t), int(f64), lane, reg, ctypes.byref(i),
                                           ctypes.byref(j), ctypes.byref(b)), "mcemu_tile_layout_inverse")
    return i.value, j.value, b.value


def swmmac_src_layout(operand: int, idx: int, k: int):
    lane, vgpr, half = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check(lib().mcemu_swmmac_src_layout(operand, idx, k, ctypes.byref(lane), ctypes.byref(vgpr),
                                         ctypes.byref(half)), "mcemu_swmmac_src_layout")
    return lane.value, vgpr.value, half.value

"""Named model configurations for the oracle (test infrastructure only).

Each preset is a plain dict of features, written from "Accurate Models of AMD
Matrix Cores": Sec. 4.1 (CDNA 1), Sec. 4.2 (CDNA 2), Sec. 4.3 with Algorithms
1-2 (CDNA 3) and Table 3 (NVIDIA columns, early c).  The three block-FMA models
of the randomized-validation workload (truncate, round-to-nearest-even, exact)
are the global-alignment early-c model with F_p = 23 + 3 extra alignment bits
and the correctly rounded model.  Keys (all optional except fmt/arch/n_fma):

  fmt_a, fmt_b      fp16 | bf16 | xf32 | fp32 | e4m3 | e5m2 | int8 | uint8
  fp8_enc           ocp | fnuz              xf32_round   trunc | rne
  arch              exact | ga_early | ga_late | odd_even | pairwise
  n_fma             N_FMA, products per multi-term addition
  align_frac        F_p, fraction bits kept after aligning to e_max
  align_round       rz | rd                 out_round    rne | rtz
  c_frac, psum_frac, post_norm_frac         late-c widths (24, 32, 31 on CDNA 3)
  sub_in_flush, sub_out_flush               bool
  c_zero_exp        exponent given to c = 0, None = c discarded (e_{c=0} = -inf)
  emin_lim          lower limit of the alignment exponent or None
  prod_overflow     |p| >= 2^128 gives Inf
  nan_bits          fp32 bit pattern of every NaN result
  int_saturate      integer formats: clamp the int32 result instead of wrapping
  acc_fmt           fp32 | fp16: format of c and d (fp16 in the low half of each 32-bit word)
"""

CDNA_NAN = 0xFFC00000     # "the resulting NaN carries a negative sign" (Secs. 4.1-4.3)
GENERIC_NAN = 0x7FC00000
GENERIC_NAN16 = 0x7E00    # the quiet NaN of binary16 (fp16-output models)


def _cdna3(fmt, n_fma, **kw):
    d = dict(fmt_a=fmt, fmt_b=fmt, arch="ga_late", n_fma=n_fma, align_frac=24, align_round="rz",
             c_frac=24, psum_frac=32, post_norm_frac=31, out_round="rne", sub_in_flush=False,
             sub_out_flush=False, c_zero_exp=-126, emin_lim=None, prod_overflow=True,
             nan_bits=CDNA_NAN)
    d.update(kw)
    return d


def _exact(fmt, n_fma, **kw):
    d = dict(fmt_a=fmt, fmt_b=fmt, arch="exact", n_fma=n_fma, out_round="rne", sub_in_flush=False,
             sub_out_flush=False, prod_overflow=False, nan_bits=CDNA_NAN)
    d.update(kw)
    return d


def _early(fmt, n_fma, align_frac, out_round, emin_lim=None, **kw):
    d = dict(fmt_a=fmt, fmt_b=fmt, arch="ga_early", n_fma=n_fma, align_frac=align_frac,
             align_round="rz", out_round=out_round, sub_in_flush=False, sub_out_flush=False,
             c_zero_exp=None, emin_lim=emin_lim, prod_overflow=False, nan_bits=GENERIC_NAN)
    d.update(kw)
    return d


PRESETS = {
    # CDNA 3 (MI300A/X), Algorithm 1: N_FMA 8 for fp16/bf16 (Sec. 4.3.1), 4 for tf19 (Sec. 4.3.3)
    "cdna3_fp16": _cdna3("fp16", 8),
    "cdna3_bf16": _cdna3("bf16", 8),
    "cdna3_xf32": _cdna3("xf32", 4, xf32_round="trunc"),
    # CDNA 3 binary8, Algorithm 2: FMA size 16 = 8 odd + 8 even products, FNUZ encodings
    "cdna3_fp8": _cdna3("e4m3", 16, arch="odd_even", fp8_enc="fnuz"),
    "cdna3_bf8": _cdna3("e5m2", 16, arch="odd_even", fp8_enc="fnuz"),
    # CDNA 1 (MI100): correctly rounded, N_FMA 4 (fp16), 2 (bf16), SFMA for fp32
    "cdna1_fp16": _exact("fp16", 4),
    "cdna1_bf16": _exact("bf16", 2),
    "cdna1_fp32": _exact("fp32", 1),
    # CDNA 2 (MI210/250): pair-wise sums of fp32-rounded products, subnormals flushed
    "cdna2_fp16": dict(fmt_a="fp16", fmt_b="fp16", arch="pairwise", n_fma=4, pair_group=4,
                       out_round="rne", sub_in_flush=True, sub_out_flush=True,
                       prod_overflow=False, nan_bits=CDNA_NAN),
    "cdna2_bf16_1k": dict(fmt_a="bf16", fmt_b="bf16", arch="pairwise", n_fma=4, pair_group=4,
                          out_round="rne", sub_in_flush=True, sub_out_flush=True,
                          prod_overflow=False, nan_bits=CDNA_NAN),
    "cdna2_bf16": dict(fmt_a="bf16", fmt_b="bf16", arch="pairwise", n_fma=2, pair_group=2,
                       out_round="rne", sub_in_flush=True, sub_out_flush=True,
                       prod_overflow=False, nan_bits=CDNA_NAN),
    # Table 3, NVIDIA columns (early c, RTZ output, c = 0 discarded)
    "b200_fp16": _early("fp16", 16, 25, "rtz", emin_lim=-133),
    "h100_fp16": _early("fp16", 16, 25, "rtz", emin_lim=-133),
    "a100_fp16": _early("fp16", 8, 24, "rtz", emin_lim=-132),
    "b200_bf16": _early("bf16", 16, 25, "rtz", emin_lim=-133),
    "a100_bf16": _early("bf16", 8, 24, "rtz", emin_lim=-132),
    "b200_tf19": _early("xf32", 8, 25, "rtz", emin_lim=-133),
    "a100_tf19": _early("xf32", 4, 24, "rtz", emin_lim=-132),
    "b200_fp8": _early("e4m3", 32, 25, "rtz"),
    "h100_fp8": _early("e4m3", 32, 13, "rtz"),
    # Table 3's note: fp16 output for fp16 and fp8 inputs, e_min^lim -20 (A100) / -21 (H100, B200)
    "b200_fp16_f16": _early("fp16", 16, 25, "rtz", emin_lim=-21, acc_fmt="fp16", nan_bits=GENERIC_NAN16),
    "h100_fp16_f16": _early("fp16", 16, 25, "rtz", emin_lim=-21, acc_fmt="fp16", nan_bits=GENERIC_NAN16),
    "a100_fp16_f16": _early("fp16", 8, 24, "rtz", emin_lim=-20, acc_fmt="fp16", nan_bits=GENERIC_NAN16),
    "b200_fp8_f16": _early("e4m3", 32, 25, "rtz", emin_lim=-21, acc_fmt="fp16", nan_bits=GENERIC_NAN16),
    "h100_fp8_f16": _early("e4m3", 32, 13, "rtz", emin_lim=-21, acc_fmt="fp16", nan_bits=GENERIC_NAN16),
}


def block_models(fmt: str, k: int):
    """The three models of the randomized block-FMA workload for one format and K:
    global alignment with 3 extra bits and truncation (RTZ output), the same with
    an RNE output, and the correctly rounded (exact-then-round) model."""
    if fmt in ("int8", "uint8"):
        return {"int": dict(fmt_a=fmt, fmt_b=fmt, arch="exact", n_fma=k, int_saturate=False)}
    return {
        "ga_trunc": _early(fmt, k, 26, "rtz"),
        "ga_rne": _early(fmt, k, 26, "rne"),
        "ieee_exact": _exact(fmt, k, nan_bits=GENERIC_NAN),
    }

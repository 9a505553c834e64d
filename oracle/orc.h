/*
 * orc.h -- interface of the CPU oracle for bit-exact matrix-multiplier emulation.
 *
 * TEST INFRASTRUCTURE ONLY.  This header and orc.c form a plain, slow, exact
 * CPU model of the block fused multiply-add
 *
 *     d = sum_{l=1..k} a_l * b_l + c                 ("Accurate Models of AMD
 *                                                      Matrix Cores", Sec. 2, eq. (1))
 *
 * and of the GEMM, 2:4-sparse GEMM and multi-word GEMM drivers built on it.
 * It shares no code, header, table or constant with the CUDA library; only
 * the test-suite, the package smoke check and the benchmark's CPU-baseline
 * leg may load it.  Nothing in the product path may call it.
 *
 * All arithmetic is exact: every value is held as a signed big integer times
 * 2^-ORC_FIX (see orc.c), and every rounding step of a model is an explicit
 * "round this exact value to a multiple of 2^g" call.
 */
#ifndef ORC_H
#define ORC_H
#include <stdint.h>

/* Input formats ("Accurate Models of AMD Matrix Cores", Table 1). */
enum { ORC_FP16 = 0, ORC_BF16 = 1, ORC_XF32 = 2, ORC_FP32 = 3,
       ORC_E4M3 = 4, ORC_E5M2 = 5, ORC_INT8 = 6, ORC_UINT8 = 7 };
/* fp8 encodings: OCP (IEEE-like, E5M2 has Inf) or FNUZ (0x80 = NaN, no Inf, no -0). */
enum { ORC_OCP = 0, ORC_FNUZ = 1 };
/* How an fp32 input is reduced to the 10-bit XF32 mantissa (Sec. 4.3.3 measures truncation). */
enum { ORC_XF32_TRUNC = 0, ORC_XF32_RNE = 1 };
/* Multi-term adder architectures (Sec. 7 names the four MATLAB configurations). */
enum { ORC_EXACT = 0,          /* correct_rounding: Kulisch-like, CDNA1 (Sec. 4.1)      */
       ORC_GA_EARLY = 1,       /* global alignment, c aligned with the products (Table 3) */
       ORC_GA_LATE = 2,        /* global alignment, late c: Algorithm 1 (CDNA3)          */
       ORC_ODD_EVEN = 3,       /* odd-even grouping, late c: Algorithm 2 (CDNA3 binary8) */
       ORC_PAIRWISE = 4 };     /* pair-wise sum of fl() results (CDNA2, Sec. 4.2)        */
enum { ORC_RZ = 0, ORC_RD = 1 };        /* alignment rounding of shifted terms        */
enum { ORC_RNE = 0, ORC_RTZ = 1 };      /* final rounding to the fp32 output          */
#define ORC_NO_EXP INT32_MIN            /* "minus infinity": c=0 discarded / no limit */

typedef struct {
  int32_t fmt_a, fmt_b;      /* ORC_FP16 ... ORC_UINT8                                   */
  int32_t fp8_enc;           /* ORC_OCP or ORC_FNUZ                                      */
  int32_t xf32_round;        /* ORC_XF32_TRUNC or ORC_XF32_RNE                           */
  int32_t arch;              /* ORC_EXACT ...                                            */
  int32_t n_fma;             /* N_FMA: products per multi-term addition                  */
  int32_t align_frac;        /* F_p: fraction bits kept when products are aligned        */
  int32_t align_round;       /* ORC_RZ or ORC_RD for the product alignment               */
  int32_t c_frac;            /* late c: frac bits of the shifted c (24 on CDNA3)         */
  int32_t psum_frac;         /* late c: frac bits of the shifted product sum (32)        */
  int32_t post_norm_frac;    /* late c: frac bits after the normalisation (31)           */
  int32_t out_round;         /* ORC_RNE or ORC_RTZ                                       */
  int32_t sub_in;            /* 1 = subnormal inputs are flushed to zero                 */
  int32_t sub_out;           /* 1 = subnormal results are flushed to zero                */
  int32_t c_zero_exp;        /* exponent given to c = 0, or ORC_NO_EXP (c discarded)     */
  int32_t emin_lim;          /* lower limit of the alignment exponent, or ORC_NO_EXP     */
  int32_t prod_ovf;          /* 1 = a product with |p| >= 2^128 becomes +-Inf            */
  uint32_t nan_bits;         /* fp32 pattern returned for every NaN result               */
  int32_t int_sat;           /* INT inputs: 1 = saturate the int32 result, 0 = wrap      */
  int32_t pair_group;        /* pairwise arch: products per group (4 or 2)               */
  int32_t acc_fmt;           /* c and d: ORC_ACC_FP32, or ORC_ACC_FP16 (binary16 in the  */
                             /* low half of each 32-bit c and d word; Table 3 note)      */
} orc_model;

/* Accumulator (c and d) formats.  Table 3's note in "Accurate Models of AMD Matrix
 * Cores": NVIDIA tensor cores also write fp16 for fp8 and fp16 inputs, with
 * e_min^lim = -20 (A100) or -21 (H100/B200).  Taken with the EXACT and GA_EARLY
 * architectures and fp16/fp8 inputs only. */
enum { ORC_ACC_FP32 = 0, ORC_ACC_FP16 = 1 };

#ifdef __cplusplus
extern "C" {
#endif
/* Element size in bytes of an input format (1, 2 or 4). */
int orc_elem_bytes(int32_t fmt);
/* One block FMA per vector: a, b are [n][m->n_fma] packed little-endian elements,
 * c and d are [n] fp32 (int32 for integer formats) bit patterns. Returns 0 or <0. */
int orc_block_fma(const orc_model *m, int64_t n, const void *a, const void *b,
                  const uint32_t *c, uint32_t *d);
/* The same with vectors of n_terms (< n_fma allowed: missing products are zeros). */
int orc_block_fma_n(const orc_model *m, int64_t n, int32_t n_terms, const void *a,
                    const void *b, const uint32_t *c, uint32_t *d);
/* Entries D[ii[e]][jj[e]] of the emulated GEMM D = A*B + C.  A is [M][K] (row
 * stride lda elements), Bt is B transposed, [N][K] (row stride ldb), C is [M][N]
 * (ldc).  kt is the instruction K: the chain restarts its N_FMA blocks at every
 * multiple of kt. */
int orc_gemm_entries(const orc_model *m, int32_t K, int32_t kt, const void *A, int64_t lda,
                     const void *Bt, int64_t ldb, const uint32_t *C, int64_t ldc,
                     int64_t n_entries, const int32_t *ii, const int32_t *jj, uint32_t *out);
/* 2:4 compression of A [M][K] along K; returns the number of groups of four
 * that hold more than two nonzeros (their first two nonzeros are kept). */
int64_t orc_sparse24_compress(int32_t fmt, int32_t fp8_enc, int32_t M, int32_t K,
                              const void *A, int64_t lda, void *Ac, int64_t ldac,
                              uint8_t *meta, int64_t ldm);
/* Entries of the sparse GEMM D = expand(Ac, meta) * B + C; K is the dense K and
 * kt the dense instruction K (the chain runs over compressed terms). */
int orc_sparse24_entries(const orc_model *m, int32_t K, int32_t kt, const void *Ac,
                         int64_t ldac, const uint8_t *meta, int64_t ldm, const void *Bt,
                         int64_t ldb, const uint32_t *C, int64_t ldc, int64_t n_entries,
                         const int32_t *ii, const int32_t *jj, uint32_t *out);
/* Multi-word split of binary64 values into n_words bf16 words (RNE, successive residuals). */
int orc_split_bf16(int64_t n, int32_t n_words, const double *x, uint16_t *words /* [n_words][n] */);
/* Entries of the multi-word GEMM: word products (i,j) with i+j <= n_words+1 when
 * truncated, else all; each an emulated bf16 GEMM with C = 0; combined in binary64. */
int orc_multiword_entries(const orc_model *word_model, int32_t kt, int32_t n_words,
                          int32_t truncated, int32_t K, const double *A, int64_t lda,
                          const double *Bt, int64_t ldb, int64_t n_entries,
                          const int32_t *ii, const int32_t *jj, double *out);
/* MFMA / SWMMAC tile facts.  family 0 = CDNA3 MFMA (wave64), 1 = RDNA4 SWMMAC (wave32). */
int orc_tile_blocks(int32_t family, int32_t M, int32_t N, int32_t K, int32_t elems_per_lane,
                    int32_t *blocks, int32_t *acc_regs);
/* Accumulator position of output (i, j) of block b.  f64 selects the FP64 layouts. */
int orc_tile_acc_pos(int32_t family, int32_t M, int32_t N, int32_t blocks, int32_t f64,
                     int32_t i, int32_t j, int32_t b, int32_t *lane, int32_t *reg);
/* SWMMAC 16x16x32 source fragment position of A (operand 0, compressed k) or B (1, dense k). */
int orc_swmmac_src_pos(int32_t operand, int32_t idx, int32_t k, int32_t *lane, int32_t *vgpr,
                       int32_t *half);
#ifdef __cplusplus
}
#endif
#endif

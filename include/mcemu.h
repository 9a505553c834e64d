/*
 * mcemu.h -- C ABI of the GB300 (sm_103a) bit-exact matrix-multiplier emulator.
 *
 * The library evaluates block fused multiply-adds
 *
 *     d = sum_{l=1..k} a_l * b_l + c                                  (1)
 *
 * ("Accurate Models of AMD Matrix Cores", Sec. 2, eq. (1)) under a
 * parameterised model of a hardware multi-term adder, and builds emulated
 * GEMMs on them with the tile semantics of the CDNA3 dense MFMA builtins and
 * the RDNA4 sparse (2:4) WMMA builtins.  Every result is an fp32 (or int32)
 * bit pattern that the model defines exactly.
 *
 * Conventions
 *  - Every function returns an mcemu_status (MCEMU_OK = 0); nothing aborts or
 *    throws across the ABI.  mcemu_status_string() names a status.
 *  - Device buffers and the CUDA stream belong to the caller.  Compute calls
 *    are enqueued on `stream` and return before the work finishes; their
 *    argument checks are synchronous.  A launch failure returns
 *    MCEMU_ERR_CUDA (cudaGetLastError() holds the CUDA error).
 *  - Model handles belong to the library (mcemu_model_create/destroy).
 *  - Element data move as raw little-endian bit patterns: 8-bit formats one
 *    byte, FP16/BF16 two bytes, XF32/FP32 four bytes; results are uint32
 *    fp32 (int32 for the integer formats) patterns.
 *  - Row-major matrices with leading dimensions in elements.  B is passed
 *    transposed, Bt = [N][K] (K contiguous), so both operand panels of a GEMM
 *    are read along K.
 *  - `stream` is a cudaStream_t passed as void* (0 = legacy default stream).
 */
#ifndef MCEMU_H
#define MCEMU_H
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------- */
typedef enum {
  MCEMU_OK = 0,
  MCEMU_ERR_INVALID_ARG = 1,   /* null/negative/inconsistent argument            */
  MCEMU_ERR_UNSUPPORTED = 2,   /* valid request this library does not implement  */
  MCEMU_ERR_NOT_2_4 = 3,       /* an A group of four holds more than 2 nonzeros  */
  MCEMU_ERR_ALIGNMENT = 4,     /* pointer or leading dimension not aligned       */
  MCEMU_ERR_CUDA = 5,          /* a CUDA runtime call or launch failed           */
  MCEMU_ERR_TIMEOUT = 6,       /* reserved: a bounded device wait gave up        */
  MCEMU_ERR_WORKSPACE = 7      /* caller workspace smaller than required         */
} mcemu_status;

const char *mcemu_status_string(int status);
/* Library version as 10000*major + 100*minor + patch. */
int mcemu_version(void);

/* ---- formats, encodings and model features --------------------------- */
/* Input formats of "Accurate Models of AMD Matrix Cores", Table 1, plus the
 * integer inputs of the MFMA/SWMMAC INT8 builtins.  XF32 (tf19) is an fp32
 * container whose mantissa the unit reduces to 10 bits (Sec. 4.3.3). */
enum { MCEMU_FP16 = 0, MCEMU_BF16 = 1, MCEMU_XF32 = 2, MCEMU_FP32 = 3,
       MCEMU_E4M3 = 4, MCEMU_E5M2 = 5, MCEMU_INT8 = 6, MCEMU_UINT8 = 7 };
/* fp8 encodings: OCP (E4M3: NaN = S.1111.111, no Inf; E5M2: IEEE-like) and
 * FNUZ (bias one larger, 0x80 is the only NaN, no Inf, no negative zero). */
enum { MCEMU_FP8_OCP = 0, MCEMU_FP8_FNUZ = 1 };
/* XF32 mantissa reduction: truncation (measured on CDNA3, Sec. 4.3.3) or RNE. */
enum { MCEMU_XF32_TRUNC = 0, MCEMU_XF32_RNE = 1 };
/* Multi-term adder architectures (the four configurations of Sec. 7):
 *  EXACT     correct rounding of the exact sum (CDNA 1, Sec. 4.1);
 *  GA_EARLY  global alignment with c aligned together with the products,
 *            the NVIDIA-like columns of Table 3;
 *  GA_LATE   Algorithm 1: products aligned and truncated, then c merged with
 *            the (24, 32, RD) rule and a normalised RD to 31 bits (CDNA 3);
 *  ODD_EVEN  Algorithm 2: odd- and even-indexed products aligned separately
 *            (CDNA 3 binary8);
 *  PAIRWISE  fl(c + fl(fl(p1+p2) + fl(p3+p4))) with products rounded to fp32
 *            (CDNA 2, Sec. 4.2). */
enum { MCEMU_ARCH_EXACT = 0, MCEMU_ARCH_GA_EARLY = 1, MCEMU_ARCH_GA_LATE = 2,
       MCEMU_ARCH_ODD_EVEN = 3, MCEMU_ARCH_PAIRWISE = 4 };
enum { MCEMU_ALIGN_RZ = 0, MCEMU_ALIGN_RD = 1 };   /* rounding of aligned products */
enum { MCEMU_OUT_RNE = 0, MCEMU_OUT_RTZ = 1 };     /* rounding of the fp32 result  */
#define MCEMU_NO_EXP INT32_MIN                      /* "minus infinity" exponent   */

/* A model: the feature vector of Table 3 plus the knobs of Secs. 4.1-4.3. */
typedef struct {
  uint32_t struct_size;          /* sizeof(mcemu_model_desc): ABI versioning         */
  int32_t fmt_a, fmt_b;          /* MCEMU_FP16 ... MCEMU_UINT8 (same class for a, b) */
  int32_t fp8_enc;               /* MCEMU_FP8_OCP or MCEMU_FP8_FNUZ                  */
  int32_t xf32_round;            /* MCEMU_XF32_TRUNC or MCEMU_XF32_RNE               */
  int32_t arch;                  /* MCEMU_ARCH_*                                     */
  int32_t block_k;               /* N_FMA: products per multi-term addition (1..32)  */
  int32_t align_frac_bits;       /* F_p: fraction bits kept after alignment to e_max */
  int32_t align_round;           /* MCEMU_ALIGN_RZ (truncate) or MCEMU_ALIGN_RD      */
  int32_t c_frac_bits;           /* GA_LATE/ODD_EVEN: shifted c kept to this (24)    */
  int32_t psum_frac_bits;        /* GA_LATE/ODD_EVEN: shifted product sum (32)      */
  int32_t post_norm_frac_bits;   /* GA_LATE/ODD_EVEN: after normalisation (31)       */
  int32_t acc_sig_bits;          /* significand of c and d: 24 (binary32), or 11     */
                                 /* (binary16 in the low half of each 32-bit c and d */
                                 /* word; GA_EARLY or EXACT with FP16/FP8 inputs)    */
  int32_t out_round;             /* MCEMU_OUT_RNE or MCEMU_OUT_RTZ                   */
  int32_t subnormal_in_flush;    /* 1: subnormal inputs (a, b, c) count as zero      */
  int32_t subnormal_out_flush;   /* 1: subnormal results become zero                 */
  int32_t c_zero_exp;            /* exponent of c = 0 (-126 on CDNA 3) or NO_EXP     */
  int32_t emin_lim;              /* GA_EARLY: floor of e_max (Table 3) or NO_EXP     */
  int32_t prod_overflow_2p128;   /* 1: a product with |p| >= 2^128 becomes +-Inf     */
  uint32_t nan_bits;             /* pattern of every NaN result (binary16 for 11)    */
  int32_t int_saturate;          /* INT formats: clamp the int32 sum instead of wrap */
  int32_t pair_group;            /* PAIRWISE: products per group (= block_k)         */
} mcemu_model_desc;

/* Named configurations.  Hardware presets fix format and N_FMA (pass fmt = -1,
 * block_k = 0); the three workload models take the format and K:
 *   GA_TRUNC   GA_EARLY, F_p = 23 + 3, truncated alignment, RTZ result;
 *   GA_RNE     the same with an RNE result;
 *   IEEE_EXACT correctly rounded (exact-then-round). */
enum {
  MCEMU_PRESET_CDNA3_FP16 = 0,   /* Algorithm 1, N_FMA 8  (Sec. 4.3.1)               */
  MCEMU_PRESET_CDNA3_BF16 = 1,   /* Algorithm 1, N_FMA 8  (Sec. 4.3.2)               */
  MCEMU_PRESET_CDNA3_XF32 = 2,   /* Algorithm 1, N_FMA 4, truncation (Sec. 4.3.3)    */
  MCEMU_PRESET_CDNA3_FP8 = 3,    /* Algorithm 2, E4M3 FNUZ, N_FMA 16 (Sec. 4.3.4)    */
  MCEMU_PRESET_CDNA3_BF8 = 4,    /* Algorithm 2, E5M2 FNUZ, N_FMA 16                 */
  MCEMU_PRESET_CDNA1_FP16 = 5,   /* exact, N_FMA 4 (Sec. 4.1.2)                      */
  MCEMU_PRESET_CDNA1_BF16 = 6,   /* exact, N_FMA 2 (Sec. 4.1.3)                      */
  MCEMU_PRESET_CDNA1_FP32 = 7,   /* SFMA: exact, N_FMA 1 (Sec. 4.1.1)                */
  MCEMU_PRESET_CDNA2_FP16 = 8,   /* pair-wise, groups of 4, no subnormals (4.2.1)    */
  MCEMU_PRESET_CDNA2_BF16_1K = 9,/* pair-wise, groups of 4 (Sec. 4.2.2)              */
  MCEMU_PRESET_CDNA2_BF16 = 10,  /* pair-wise, groups of 2 (Sec. 4.2.2)              */
  MCEMU_PRESET_B200_FP16 = 11,   /* Table 3: early c, (2,25), N_FMA 16, RTZ, -133    */
  MCEMU_PRESET_H100_FP16 = 12,
  MCEMU_PRESET_A100_FP16 = 13,   /* (2,24), N_FMA 8, -132                            */
  MCEMU_PRESET_B200_BF16 = 14,
  MCEMU_PRESET_A100_BF16 = 15,
  MCEMU_PRESET_B200_TF19 = 16,   /* (2,25), N_FMA 8                                  */
  MCEMU_PRESET_A100_TF19 = 17,   /* (2,24), N_FMA 4                                  */
  MCEMU_PRESET_B200_FP8 = 18,    /* (2,25), N_FMA 32, no e_min limit                 */
  MCEMU_PRESET_H100_FP8 = 19,    /* (2,13), N_FMA 32                                 */
  /* Table 3's note: fp16 output (acc_sig_bits 11) for fp16 and fp8 inputs, with
   * e_min^lim -21 (H100, B200) or -20 (A100); c and d are binary16 */
  MCEMU_PRESET_B200_FP16_F16 = 20, /* as B200_FP16, fp16 c and d, e_min^lim -21      */
  MCEMU_PRESET_H100_FP16_F16 = 21,
  MCEMU_PRESET_A100_FP16_F16 = 22, /* as A100_FP16, fp16 c and d, e_min^lim -20      */
  MCEMU_PRESET_B200_FP8_F16 = 23,  /* as B200_FP8, fp16 c and d, e_min^lim -21       */
  MCEMU_PRESET_H100_FP8_F16 = 24,
  MCEMU_PRESET_GA_TRUNC = 100,
  MCEMU_PRESET_GA_RNE = 101,
  MCEMU_PRESET_IEEE_EXACT = 102
};
/* Fill *out with a named configuration.  INVALID_ARG for an unknown preset or
 * a format/K that the preset does not take. */
int mcemu_model_preset(int preset, int fmt, int block_k, mcemu_model_desc *out);

typedef struct mcemu_model *mcemu_model_t;
/* Validate a description and create a model handle (host memory, owned by the
 * library until mcemu_model_destroy).  UNSUPPORTED for valid features outside
 * what the kernels implement (e.g. acc_sig_bits != 24, F_p > 56). */
int mcemu_model_create(const mcemu_model_desc *desc, mcemu_model_t *out);
void mcemu_model_destroy(mcemu_model_t model);
/* Copy the (validated) description of a model. */
int mcemu_model_get_desc(mcemu_model_t model, mcemu_model_desc *out);

/* ---- stream of block FMAs (eq. (1), one per vector set) ---------------- */
/* d[v] = model(a[v][0..k-1], b[v][0..k-1], c[v]) for v < n, k = block_k.
 * a, b: device, [n][k] packed elements of fmt_a / fmt_b; c, d: device [n]
 * fp32 (int32) patterns.  a, b, c, d must be 4-byte aligned (16-byte
 * alignment gives the vectorised path).  n = 0 is a no-op. */
int mcemu_block_fma(mcemu_model_t model, size_t n, const void *a, const void *b,
                    const uint32_t *c, uint32_t *d, void *stream);
/* The same from host memory: a, b, c and d are HOST buffers.  When all four are
 * page-locked and mapped into the device's address space (cudaHostAlloc memory
 * under unified addressing), the kernels read and write them in place over the
 * host link; otherwise the library streams them through the caller's device
 * workspace in chunks, overlapping copies with compute.  Either way the call
 * returns after d has been written (synchronous).  ws_bytes must be at least
 * mcemu_block_fma_host_workspace(model, ...). */
int mcemu_block_fma_host(mcemu_model_t model, size_t n, const void *a, const void *b,
                         const uint32_t *c, uint32_t *d, void *workspace, size_t ws_bytes,
                         void *stream);
size_t mcemu_block_fma_host_workspace(mcemu_model_t model);

/* ---- MFMA / SWMMAC tile semantics -------------------------------------- */
/* family 0: CDNA3 MFMA (wave64); family 1: RDNA4 SWMMAC (wave32, 2:4 sparse A,
 * K counts dense positions).  elems_per_lane: A elements one lane supplies
 * (1 for FP32/FP64, 4 for v4half/v4bfloat and packed INT8, 2 for XF32, 8 for
 * FP8/BF8 and the wide INT8 builtins). */
typedef struct {
  int32_t family;
  int32_t M, N, K;
  int32_t elems_per_lane;
} mcemu_tile_desc;
/* Blocks (independent M x N tiles per instruction) and accumulator registers
 * per lane.  CDNA3: blocks = 64 * elems_per_lane / (M*K), which reproduces the
 * Ops column of the builtin table (Ops = 2*M*N*K*blocks); accVGPRs =
 * blocks * M*N / 64 ("Accumulator layout").  SWMMAC: 1 block, M*N/32 VGPRs. */
int mcemu_tile_info(const mcemu_tile_desc *tile, int32_t *blocks, int32_t *acc_regs);
/* Lane and register that hold output (i, j) of block b ("Accumulator layout"
 * formulas for 32x32, 16x16, 4x4 and, with f64 = 1, the FP64 16x16 and 4x4
 * layouts; the SWMMAC 16x16 accumulator layout for family 1). */
int mcemu_tile_layout(const mcemu_tile_desc *tile, int f64, int i, int j, int b,
                      int32_t *lane, int32_t *reg);
/* Inverse of mcemu_tile_layout. */
int mcemu_tile_layout_inverse(const mcemu_tile_desc *tile, int f64, int lane, int reg,
                              int32_t *i, int32_t *j, int32_t *b);
/* SWMMAC 16x16x32 source fragments ("srcA (sparse)", "srcB (dense)"):
 * operand 0 = compressed A element k (0..15) of row idx; operand 1 = dense B
 * row k (0..31) of column idx; two 16-bit values share a VGPR (half 0/1). */
int mcemu_swmmac_src_layout(int operand, int idx, int k, int32_t *lane, int32_t *vgpr,
                            int32_t *half);

/* ---- emulated GEMMs ------------------------------------------------------ */
/* D = A*B + C, M x N x K, with the instruction inner size tile->K: each output
 * is a chain over K in instructions of tile->K, each instruction made of
 * ceil(tile->K / block_k) block FMAs over consecutive k, the fp32 accumulator
 * carried as the next c (MFMA builtins: "Each instruction processes one K
 * step; the caller loops over K").  A [M][K] (lda), Bt [N][K] (ldb), C and D
 * [M][N] (ldc, ldd); C may equal D.  Ragged M, N, K are allowed. */
int mcemu_tile_gemm(mcemu_model_t model, const mcemu_tile_desc *tile, int M, int N, int K,
                    const void *A, int64_t lda, const void *Bt, int64_t ldb,
                    const uint32_t *C, int64_t ldc, uint32_t *D, int64_t ldd, void *stream);

/* 2:4 compression along K ("Structured sparsity (2:4 pattern)"): for every row
 * and group of four, Ac keeps two values and meta one byte idx0 | idx1 << 2
 * (idx0 < idx1).  A group with fewer than two nonzeros is padded with its
 * lowest zero positions; -0 is zero, NaN is nonzero.  A group with more than
 * two nonzeros keeps its first two and adds 1 to *d_violations (device
 * int64, accumulated: zero it first).  K % 4 == 0. */
int mcemu_sparse24_compress(int fmt, int fp8_enc, int M, int K, const void *A, int64_t lda,
                            void *Ac, int64_t ldac, uint8_t *meta, int64_t ldm,
                            int64_t *d_violations, void *stream);
/* Synchronous check of a compression: waits for `stream`, reads the device
 * counter *d_violations into *h_count (when not NULL) and returns
 * MCEMU_ERR_NOT_2_4 when some group held more than two nonzeros (the pattern of
 * "Structured sparsity (2:4 pattern)" does not hold), MCEMU_OK otherwise. */
int mcemu_sparse24_check(const int64_t *d_violations, int64_t *h_count, void *stream);
/* Inverse: A = expand(Ac, meta), zeros elsewhere. */
int mcemu_sparse24_expand(int fmt, int M, int K, const void *Ac, int64_t ldac,
                          const uint8_t *meta, int64_t ldm, void *A, int64_t lda, void *stream);
/* D = expand(Ac, meta) * B + C with SWMMAC tile semantics: the chain runs over
 * the compressed terms in order, tile->K/2 of them per instruction, in blocks
 * of block_k; the product of compressed term kc is Ac[i][kc] *
 * B[4*(kc/2) + idx(kc)][j].  K is the dense inner size (K % 4 == 0). */
int mcemu_sparse24_gemm(mcemu_model_t model, const mcemu_tile_desc *tile, int M, int N, int K,
                        const void *Ac, int64_t ldac, const uint8_t *meta, int64_t ldm,
                        const void *Bt, int64_t ldb, const uint32_t *C, int64_t ldc,
                        uint32_t *D, int64_t ldd, void *stream);

/* ---- multi-word GEMM (Sec. 8.1) ------------------------------------------ */
enum { MCEMU_WORDS_ALL = 0, MCEMU_WORDS_TRUNCATED = 1 };
/* Split binary64 x[n] into n_words BF16 words: w_1 = RNE_bf16(x), w_{i+1} =
 * RNE_bf16 of the exact residual x - w_1 - ... - w_i.  words: [n_words][n]. */
int mcemu_multiword_split(int n_words, size_t n, const double *x, uint16_t *words,
                          void *stream);
/* D = sum over word pairs (i, j) of fp64(D_ij), D_ij = emulated BF16 GEMM of
 * the words A_i, B_j with C = 0 and fp32 output, under word_model (fmt BF16).
 * All n_words^2 pairs, or with MCEMU_WORDS_TRUNCATED those with
 * i + j <= n_words + 1.  The binary64 sum runs over i+j descending, then i
 * ascending.  A [M][K] (lda), Bt [N][K] (ldb) binary64; D [M][N] binary64.
 * workspace: device, >= mcemu_multiword_workspace(n_words, M, N, K) bytes: the
 * BF16 words of A and B and one fp32 word product. */
int mcemu_multiword_gemm(mcemu_model_t word_model, const mcemu_tile_desc *tile, int n_words,
                         int product_set, int M, int N, int K, const double *A, int64_t lda,
                         const double *Bt, int64_t ldb, double *D, int64_t ldd,
                         void *workspace, size_t ws_bytes, void *stream);
size_t mcemu_multiword_workspace(int n_words, int M, int N, int K);
/* ---- multi-word GEMM with no allocation (library addition) ----------------
 * The paper has no counterpart to this call: it is a convenience of this
 * library.  It computes exactly what mcemu_multiword_gemm computes (same
 * kernels, same results bit for bit), but takes no workspace argument: its
 * workspace (the BF16 words of A and B and one fp32 word product) is a fixed
 * array in the library's own device memory, MCEMU_MULTIWORD_STATIC_BYTES long.  It is meant for callers
 * that cannot allocate device memory where they call it: a host program that
 * only holds device buffers handed to it, or a loop whose device memory was
 * budgeted up front and must not grow.  The call itself allocates nothing.
 * Set-up: the first call on each device (the caller's current device) looks up
 * the array's device address once; make that first call before any stream
 * capture.  Limit: mcemu_multiword_workspace(n_words, M, N, K) must not exceed
 * MCEMU_MULTIWORD_STATIC_BYTES, else MCEMU_ERR_WORKSPACE and nothing runs.
 * Nothing in the array has to start at zero (everything in it is written
 * before it is read).  The array is shared by all calls on a device: two calls whose
 * kernels may overlap (other streams, other host threads) race on it; order
 * them on one stream.  Other arguments and errors as mcemu_multiword_gemm;
 * MCEMU_ERR_CUDA when the address look-up fails. */
#define MCEMU_MULTIWORD_STATIC_BYTES ((size_t)8 << 20)
int mcemu_multiword_gemm_static(mcemu_model_t word_model, const mcemu_tile_desc *tile, int n_words,
                                int product_set, int M, int N, int K, const double *A, int64_t lda,
                                const double *Bt, int64_t ldb, double *D, int64_t ldd, void *stream);
/* Relative norm-wise error ||D - R||_F / ||R||_F pieces (Sec. 8.1 reports this
 * error): out[0] = sum (D-R)^2, out[1] = sum R^2, summed in a fixed order.
 * out: device, MCEMU_FRO_OUT_DOUBLES doubles; out[2..] is scratch. */
#define MCEMU_FRO_OUT_DOUBLES 1026
int mcemu_fro_error(int M, int N, const double *D, int64_t ldd, const double *R, int64_t ldr,
                    double *out, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* MCEMU_H */

// model.h -- the model description as the kernels see it, and the host-side
// launchers that the C ABI (api.cu) calls.  Built only into libmcemu.so.
#pragma once
#include <cstddef>
#include <cstdint>

#include "../../include/mcemu.h"

namespace mcemu {

// Exponent used for "no exponent": zero elements, a discarded c = 0, no limit.
constexpr int32_t kNegE = -4096;

// One input format as the decoder needs it (all runtime values, so one kernel
// serves every format of a container size).
struct FmtDev {
  uint32_t mbits;       // stored mantissa bits (23 for the fp32 container of XF32)
  uint32_t emask;       // exponent field mask after shifting by mbits
  uint32_t sshift;      // position of the sign bit
  int32_t bias;         // exponent bias (normal: E = field - bias; subnormal: 1 - bias)
  uint32_t top_special; // exponent field of Inf/NaN, 0xFFFFFFFF when the format has none
  uint32_t nan_pat;     // extra NaN encoding: (bits & nan_mask) == nan_pat
  uint32_t nan_mask;    //   (0, 0xFFFFFFFF: none)
  uint32_t sub_keep;    // mantissa mask applied to subnormals (0 = flushed to zero)
  uint32_t xf32;        // fp32 container reduced to 10 bits: 0 no, 1 truncate, 2 RNE
  uint32_t sig_rshift;  // 13 for XF32 (low mantissa bits dropped), else 0
  int32_t m_eff;        // significand fraction bits after the reduction
  uint32_t is_int;      // 1 = INT8/UINT8
  uint32_t is_signed;   // INT8
  // SWAR special-value detection on a 32-bit word of packed elements:
  // special lanes have ((w & sw_mask) + sw_add) & sw_hi != 0, or (FNUZ) a 0x80 byte.
  uint32_t sw_mask, sw_add, sw_hi, sw_fnuz;
};

struct DevModel {
  FmtDev fa, fb;
  int32_t arch, k;
  int32_t F;              // alignment fraction bits F_p
  int32_t align_rd;       // 1 = RD (floor), 0 = RZ
  int32_t c_frac, psum_frac, post_norm_frac;
  int32_t rne;            // 1 = RNE result, 0 = RTZ
  int32_t sub_out_flush;
  uint32_t c_sub_keep;    // 0x7FFFFF, or 0 when subnormal inputs are flushed
  int32_t c_zero_exp;     // kNegE when c = 0 is discarded
  int32_t emin_lim;       // kNegE when none
  int32_t prod_ovf;
  uint32_t nan_bits;
  int32_t int_sat;
  // derived
  int32_t mab;            // m_eff(a) + m_eff(b): fraction bits of a product significand
  int32_t P0, R0;         // product significand pre-shift left / extra right shift (F - mab)
  int32_t P0c, R0c;       // the same for c (F - 23)
  int32_t bias_sum;       // bias_a + bias_b (products carry biased exponents)
  int32_t wide;           // 1 when sums need 64-bit integers
  uint32_t p0mul, p0cmul; // 2^P0 and 2^P0c (32-bit sums): the pre-shifts as multiplies
  int32_t acc16;          // 1: c and d are binary16 (low half of the 32-bit words)
};

struct Model {
  mcemu_model_desc desc;
  DevModel dev;
};

// launchers (stream.cu, gemm.cu, sparse.cu, multiword.cu)
int launch_block_fma(const DevModel &m, size_t n, const void *a, const void *b, const uint32_t *c,
                     uint32_t *d, void *stream);
bool f8_stream_ok(const DevModel &m, int id);
int launch_block_fma_f8(const DevModel &m, int id, size_t n, const void *a, const void *b, const uint32_t *c,
                        uint32_t *d, void *stream);
int launch_tile_gemm(const DevModel &m, int kt, int M, int N, int K, const void *A, int64_t lda,
                     const void *Bt, int64_t ldb, const uint32_t *C, int64_t ldc, uint32_t *D,
                     int64_t ldd, void *stream);
bool gemm_fast_ok(const DevModel &m);
int launch_tile_gemm_fast(const DevModel &m, int kt, int M, int N, int K, const void *A, int64_t lda,
                          const void *Bt, int64_t ldb, const uint32_t *C, int64_t ldc, uint32_t *D, int64_t ldd,
                          void *stream);
bool sparse_fast_ok(const DevModel &m, int kt);
bool gemm_exact_ok(const DevModel &m);
int launch_tile_gemm_exact(const DevModel &m, int kt, int M, int N, int K, const void *A, int64_t lda,
                           const void *Bt, int64_t ldb, const uint32_t *C, int64_t ldc, uint32_t *D, int64_t ldd,
                           void *stream);
int launch_sparse24_gemm_exact(const DevModel &m, int kt, int M, int N, int K, const void *Ac, int64_t ldac,
                               const uint8_t *meta, int64_t ldm, const void *Bt, int64_t ldb, const uint32_t *C,
                               int64_t ldc, uint32_t *D, int64_t ldd, void *stream);
int launch_sparse24_gemm_fast(const DevModel &m, int kt, int M, int N, int K, const void *Ac, int64_t ldac,
                              const uint8_t *meta, int64_t ldm, const void *Bt, int64_t ldb, const uint32_t *C,
                              int64_t ldc, uint32_t *D, int64_t ldd, void *stream);
int launch_sparse24_compress(const FmtDev &f, int elem_bytes, int M, int K, const void *A,
                             int64_t lda, void *Ac, int64_t ldac, uint8_t *meta, int64_t ldm,
                             int64_t *viol, void *stream);
int launch_sparse24_expand(int elem_bytes, int M, int K, const void *Ac, int64_t ldac,
                           const uint8_t *meta, int64_t ldm, void *A, int64_t lda, void *stream);
int launch_sparse24_gemm(const DevModel &m, int kt, int M, int N, int K, const void *Ac,
                         int64_t ldac, const uint8_t *meta, int64_t ldm, const void *Bt,
                         int64_t ldb, const uint32_t *C, int64_t ldc, uint32_t *D, int64_t ldd,
                         void *stream);
int launch_multiword_split(int n_words, size_t n, const double *x, int64_t ldx, int rows,
                           uint16_t *words, int64_t word_stride, void *stream);
int launch_multiword_gemm(const DevModel &m, int kt, int n_words, int truncated, int M, int N,
                          int K, const double *A, int64_t lda, const double *Bt, int64_t ldb,
                          double *D, int64_t ldd, void *ws, size_t ws_bytes, void *stream);
int launch_multiword_gemm_static(const DevModel &m, int kt, int n_words, int truncated, int M, int N, int K,
                                 const double *A, int64_t lda, const double *Bt, int64_t ldb, double *D,
                                 int64_t ldd, void *stream);
int launch_fro_error(int M, int N, const double *D, int64_t ldd, const double *R, int64_t ldr,
                     double *out, void *stream);

}  // namespace mcemu

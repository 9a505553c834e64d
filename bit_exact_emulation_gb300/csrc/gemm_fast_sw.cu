// gemm_fast_sw.cu -- the global-alignment tile GEMM for the 2:4-sparse GEMM and for
// the word products of the multi-word GEMM (kernel in gemm_fast.cuh).
#include "gemm_fast.cuh"

namespace mcemu {

// One word-pair product of the multi-word GEMM: BF16 words, C = 0, the fp32 results
// added into the binary64 D (or written as 0 + result when `first`).
int launch_tile_gemm_fast_acc64(const DevModel &m, int kt, int M, int N, int K, const uint16_t *Aw, int64_t lda,
                                const uint16_t *Bw, int64_t ldb, double *D, int64_t ldd, int first, void *stream) {
  cudaStream_t s = (cudaStream_t)stream;
  if (kt > 64 || (int)(m.fa.sshift + 1) / 8 != 2) return MCEMU_ERR_UNSUPPORTED;
  if (m.arch == MCEMU_ARCH_GA_EARLY)
    return run_fast<MCEMU_ARCH_GA_EARLY, 2, 1>(m, kt, M, N, K, Aw, lda, Bw, ldb, nullptr, 0, nullptr, ldd, s, D, first);
  return run_fast<MCEMU_ARCH_GA_LATE, 2, 1>(m, kt, M, N, K, Aw, lda, Bw, ldb, nullptr, 0, nullptr, ldd, s, D, first);
}

// 2:4-sparse tile GEMM through the dense fast kernel (expansion while staging);
// kt and K are the dense instruction and inner sizes.
bool sparse_fast_ok(const DevModel &m, int kt) {
  // an even N_FMA keeps every group of four inside one block
  return gemm_fast_ok(m) && m.k % 2 == 0 && 2 * m.k <= 32 && kt <= 64 && (int)(m.fa.sshift + 1) / 8 <= 2;
}

int launch_sparse24_gemm_fast(const DevModel &m, int kt, int M, int N, int K, const void *Ac, int64_t ldac,
                              const uint8_t *meta, int64_t ldm, const void *Bt, int64_t ldb, const uint32_t *C,
                              int64_t ldc, uint32_t *D, int64_t ldd, void *stream) {
  cudaStream_t s = (cudaStream_t)stream;
  const int eb = (int)(m.fa.sshift + 1) / 8;
  if (!sparse_fast_ok(m, kt)) return MCEMU_ERR_UNSUPPORTED;
  if (m.arch == MCEMU_ARCH_GA_EARLY) {
    if (eb == 1)
      return run_fast<MCEMU_ARCH_GA_EARLY, 1, 0, 1>(m, kt, M, N, K, Ac, ldac, Bt, ldb, C, ldc, D, ldd, s, nullptr, 0,
                                                    meta, ldm);
    return run_fast<MCEMU_ARCH_GA_EARLY, 2, 0, 1>(m, kt, M, N, K, Ac, ldac, Bt, ldb, C, ldc, D, ldd, s, nullptr, 0,
                                                  meta, ldm);
  }
  if (eb == 1)
    return run_fast<MCEMU_ARCH_GA_LATE, 1, 0, 1>(m, kt, M, N, K, Ac, ldac, Bt, ldb, C, ldc, D, ldd, s, nullptr, 0,
                                                 meta, ldm);
  return run_fast<MCEMU_ARCH_GA_LATE, 2, 0, 1>(m, kt, M, N, K, Ac, ldac, Bt, ldb, C, ldc, D, ldd, s, nullptr, 0,
                                               meta, ldm);
}

}  // namespace mcemu

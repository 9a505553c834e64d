// gemm_fast.cu -- dense instantiations of the global-alignment tile GEMM
// (kernel in gemm_fast.cuh).
#include "gemm_fast.cuh"

namespace mcemu {

// true when the fast kernel implements the model (else the general kernel runs)
bool gemm_fast_ok(const DevModel &m) {
  if (m.fa.is_int || m.fb.is_int || m.acc16) return false;
  if (m.arch != MCEMU_ARCH_GA_EARLY && m.arch != MCEMU_ARCH_GA_LATE) return false;
  if (m.wide || m.align_rd || m.sub_out_flush) return false;
  if (m.mab > 22) return false;                          // binary32 significands: 48-bit products
  if (m.k > 32) return false;
  return true;
}

int launch_tile_gemm_fast(const DevModel &m, int kt, int M, int N, int K, const void *A, int64_t lda,
                          const void *Bt, int64_t ldb, const uint32_t *C, int64_t ldc, uint32_t *D, int64_t ldd,
                          void *stream) {
  cudaStream_t s = (cudaStream_t)stream;
  const int eb = (int)(m.fa.sshift + 1) / 8;
  if (kt > 64) return MCEMU_ERR_UNSUPPORTED;
  if (m.arch == MCEMU_ARCH_GA_EARLY) {
    if (eb == 1) return run_fast<MCEMU_ARCH_GA_EARLY, 1>(m, kt, M, N, K, A, lda, Bt, ldb, C, ldc, D, ldd, s);
    if (eb == 2) return run_fast<MCEMU_ARCH_GA_EARLY, 2>(m, kt, M, N, K, A, lda, Bt, ldb, C, ldc, D, ldd, s);
    return run_fast<MCEMU_ARCH_GA_EARLY, 4>(m, kt, M, N, K, A, lda, Bt, ldb, C, ldc, D, ldd, s);
  }
  if (eb == 1) return run_fast<MCEMU_ARCH_GA_LATE, 1>(m, kt, M, N, K, A, lda, Bt, ldb, C, ldc, D, ldd, s);
  if (eb == 2) return run_fast<MCEMU_ARCH_GA_LATE, 2>(m, kt, M, N, K, A, lda, Bt, ldb, C, ldc, D, ldd, s);
  return run_fast<MCEMU_ARCH_GA_LATE, 4>(m, kt, M, N, K, A, lda, Bt, ldb, C, ldc, D, ldd, s);
}

}  // namespace mcemu

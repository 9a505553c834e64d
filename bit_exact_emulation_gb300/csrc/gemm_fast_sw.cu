// gemm_fast_sw.cu -- the global-alignment tile GEMM for the 2:4-sparse GEMM (kernel
// in gemm_fast.cuh).
#include "gemm_fast.cuh"

namespace mcemu {

// 2:4-sparse tile GEMM through the fast kernels in their gather form: the chain runs
// over the compressed terms, each reading B at the row its metadata index names; kt
// and K are the dense instruction and inner sizes.
bool sparse_fast_ok(const DevModel &m, int kt) {
  // any N_FMA: a block of compressed terms may end inside a group of four
  return gemm_fast_ok(m) && kt <= 64 && (int)(m.fa.sshift + 1) / 8 <= 2;
}

int launch_sparse24_gemm_fast(const DevModel &m, int kt, int M, int N, int K, const void *Ac, int64_t ldac,
                              const uint8_t *meta, int64_t ldm, const void *Bt, int64_t ldb, const uint32_t *C,
                              int64_t ldc, uint32_t *D, int64_t ldd, void *stream) {
  cudaStream_t s = (cudaStream_t)stream;
  const int eb = (int)(m.fa.sshift + 1) / 8;
  if (!sparse_fast_ok(m, kt)) return MCEMU_ERR_UNSUPPORTED;
  if (m.arch == MCEMU_ARCH_GA_EARLY) {
    if (eb == 1)
      return run_fast<MCEMU_ARCH_GA_EARLY, 1, 1>(m, kt, M, N, K, Ac, ldac, Bt, ldb, C, ldc, D, ldd, s, meta, ldm);
    return run_fast<MCEMU_ARCH_GA_EARLY, 2, 1>(m, kt, M, N, K, Ac, ldac, Bt, ldb, C, ldc, D, ldd, s, meta, ldm);
  }
  if (eb == 1)
    return run_fast<MCEMU_ARCH_GA_LATE, 1, 1>(m, kt, M, N, K, Ac, ldac, Bt, ldb, C, ldc, D, ldd, s, meta, ldm);
  return run_fast<MCEMU_ARCH_GA_LATE, 2, 1>(m, kt, M, N, K, Ac, ldac, Bt, ldb, C, ldc, D, ldd, s, meta, ldm);
}

}  // namespace mcemu

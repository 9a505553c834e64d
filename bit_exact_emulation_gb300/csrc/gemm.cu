// gemm.cu -- emulated GEMMs with MFMA / SWMMAC tile semantics.
//
// Each output d_ij is the chain over K that an MFMA instruction sequence
// performs ("Each instruction processes one K step; the caller loops over K",
// CDNA3 dense MFMA page): instructions of kt products, each split into
// ceil(kt / N_FMA) block FMAs over consecutive k, the fp32 accumulator carried
// as the next c.  The chain is sequential in k, so work is parallel only over
// outputs; K is never split.
//
// Tiling: a CTA owns a BM x BN tile of D; the A rows and B columns it needs are
// staged through shared memory kt-aligned chunk by chunk (blocks never cross a
// chunk), and each thread evaluates the block FMAs of its TM x TN outputs.
#include <cuda_runtime.h>

#include "core.cuh"

namespace mcemu {

constexpr int kT = 16;                 // CTA tile: kT x kT outputs, one per thread

template <int ESZ>
__device__ __forceinline__ uint32_t ld_elem(const uint8_t *base, int64_t idx) {
  if constexpr (ESZ == 1) return base[idx];
  else if constexpr (ESZ == 2) return reinterpret_cast<const uint16_t *>(base)[idx];
  else return reinterpret_cast<const uint32_t *>(base)[idx];
}

// chunk length: a multiple of the instruction K, about 64 elements
__host__ __device__ __forceinline__ int chunk_len(int kt) { return kt >= 64 ? kt : kt * (64 / kt); }

// Dense tile GEMM, any model.  Shared memory: A chunk [kT][KC] and B chunk
// [kT][KC] raw bit patterns (as 32-bit words).
template <int ESZ>
__global__ void __launch_bounds__(kT *kT) gemm_generic_kernel(const DevModel m, int kt, int M, int N, int K,
                                                              const uint8_t *__restrict__ A, int64_t lda,
                                                              const uint8_t *__restrict__ Bt, int64_t ldb,
                                                              const uint32_t *C, int64_t ldc, uint32_t *D,
                                                              int64_t ldd) {
  extern __shared__ uint32_t smem[];
  const int KC = chunk_len(kt);
  uint32_t *As = smem;                 // [kT][KC]
  uint32_t *Bs = smem + kT * KC;       // [kT][KC]
  const int i0 = blockIdx.y * kT, j0 = blockIdx.x * kT;
  const int tid = threadIdx.y * kT + threadIdx.x;
  const int i = i0 + threadIdx.y, j = j0 + threadIdx.x;
  uint32_t acc = (i < M && j < N) ? C[(int64_t)i * ldc + j] : 0u;
  for (int k0 = 0; k0 < K; k0 += KC) {
    const int kc = min(KC, K - k0);
    __syncthreads();
    for (int e = tid; e < kT * KC; e += kT * kT) {
      int r = e / KC, q = e % KC;
      As[e] = (i0 + r < M && q < kc) ? ld_elem<ESZ>(A, (int64_t)(i0 + r) * lda + k0 + q) : 0u;
      Bs[e] = (j0 + r < N && q < kc) ? ld_elem<ESZ>(Bt, (int64_t)(j0 + r) * ldb + k0 + q) : 0u;
    }
    __syncthreads();
    // instruction steps of kt inside the chunk, N_FMA blocks inside each step
    for (int s0 = 0; s0 < kc; s0 += kt) {
      const int send = min(s0 + kt, kc);
      for (int b0 = s0; b0 < send; b0 += m.k) {
        const int nt = min(m.k, send - b0);
        acc = block_eval_generic(m, As + threadIdx.y * KC + b0, Bs + threadIdx.x * KC + b0, nt, acc);
      }
    }
  }
  if (i < M && j < N) D[(int64_t)i * ldd + j] = acc;
}

// 2:4 sparse GEMM (RDNA4 SWMMAC semantics): the chain runs over compressed
// terms; term kc multiplies Ac[i][kc] with B[4*(kc/2) + idx(kc)][j].
template <int ESZ>
__global__ void __launch_bounds__(kT *kT) sparse_generic_kernel(
    const DevModel m, int ktc, int M, int N, int Kc, const uint8_t *__restrict__ Ac, int64_t ldac,
    const uint8_t *__restrict__ meta, int64_t ldm, const uint8_t *__restrict__ Bt, int64_t ldb,
    const uint32_t *C, int64_t ldc, uint32_t *D, int64_t ldd) {
  extern __shared__ uint32_t smem[];
  const int KC = chunk_len(ktc);          // compressed chunk (even)
  uint32_t *As = smem;                     // [kT][KC] compressed A
  uint32_t *Ms = smem + kT * KC;           // [kT][KC] dense offset 4*(kc/2)+idx of each term
  uint32_t *Bs = Ms + kT * KC;             // [kT][2*KC] dense B rows of the chunk
  const int i0 = blockIdx.y * kT, j0 = blockIdx.x * kT;
  const int tid = threadIdx.y * kT + threadIdx.x;
  const int i = i0 + threadIdx.y, j = j0 + threadIdx.x;
  uint32_t acc = (i < M && j < N) ? C[(int64_t)i * ldc + j] : 0u;
  for (int k0 = 0; k0 < Kc; k0 += KC) {
    const int kc = min(KC, Kc - k0);
    __syncthreads();
    for (int e = tid; e < kT * KC; e += kT * kT) {
      int r = e / KC, q = e % KC;
      bool ok = i0 + r < M && q < kc;
      As[e] = ok ? ld_elem<ESZ>(Ac, (int64_t)(i0 + r) * ldac + k0 + q) : 0u;
      uint32_t mb = ok ? meta[(int64_t)(i0 + r) * ldm + (k0 + q) / 2] : 0u;
      Ms[e] = 4u * (uint32_t)(q / 2) + (((k0 + q) & 1) ? ((mb >> 2) & 3u) : (mb & 3u));
    }
    for (int e = tid; e < kT * 2 * KC; e += kT * kT) {
      int r = e / (2 * KC), q = e % (2 * KC);
      Bs[e] = (j0 + r < N && q < 2 * kc) ? ld_elem<ESZ>(Bt, (int64_t)(j0 + r) * ldb + 2 * k0 + q) : 0u;
    }
    __syncthreads();
    for (int s0 = 0; s0 < kc; s0 += ktc) {
      const int send = min(s0 + ktc, kc);
      for (int b0 = s0; b0 < send; b0 += m.k) {
        const int nt = min(m.k, send - b0);
        uint32_t ea[32], eb[32];
        for (int l = 0; l < nt; l++) {
          ea[l] = As[threadIdx.y * KC + b0 + l];
          eb[l] = Bs[threadIdx.x * 2 * KC + Ms[threadIdx.y * KC + b0 + l]];
        }
        acc = block_eval_generic(m, ea, eb, nt, acc);
      }
    }
  }
  if (i < M && j < N) D[(int64_t)i * ldd + j] = acc;
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
// do the M x N u32 matrices at C (ldc) and D (ldd) share any bytes?
static bool overlaps(const uint32_t *C, int64_t ldc, const uint32_t *D, int64_t ldd, int M, int N) {
  if (M <= 0 || N <= 0) return false;
  const uintptr_t c0 = (uintptr_t)C, c1 = (uintptr_t)(C + (int64_t)(M - 1) * ldc + N);
  const uintptr_t d0 = (uintptr_t)D, d1 = (uintptr_t)(D + (int64_t)(M - 1) * ldd + N);
  return c0 < d1 && d0 < c1;
}

static int elem_size(const DevModel &m) { return m.fa.is_int ? 1 : (int)(m.fa.sshift + 1) / 8; }

template <class Kern>
static int set_smem(Kern kern, size_t shm) {
  if (shm <= 48 * 1024) return MCEMU_OK;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)shm) == cudaSuccess
             ? MCEMU_OK : MCEMU_ERR_UNSUPPORTED;
}

int launch_tile_gemm(const DevModel &m, int kt, int M, int N, int K, const void *A, int64_t lda,
                     const void *Bt, int64_t ldb, const uint32_t *C, int64_t ldc, uint32_t *D,
                     int64_t ldd, void *stream) {
  cudaStream_t s = (cudaStream_t)stream;
  if (kt > 1024) return MCEMU_ERR_UNSUPPORTED;
  // the fast kernels leave some outputs to a second pass that reads C again, so an
  // in-place accumulation (C overlapping D) takes the general kernel
  const bool alias = C && overlaps(C, ldc, D, ldd, M, N);
  if (!alias && gemm_fast_ok(m) && kt <= 64)
    return launch_tile_gemm_fast(m, kt, M, N, K, A, lda, Bt, ldb, C, ldc, D, ldd, stream);
  if (!alias && gemm_exact_ok(m) && kt <= 64)
    return launch_tile_gemm_exact(m, kt, M, N, K, A, lda, Bt, ldb, C, ldc, D, ldd, stream);
  const size_t shm = (size_t)2 * kT * chunk_len(kt) * 4;
  dim3 grid((N + kT - 1) / kT, (M + kT - 1) / kT), block(kT, kT);
  const uint8_t *a = (const uint8_t *)A, *b = (const uint8_t *)Bt;
  int st;
  switch (elem_size(m)) {
    case 1:
      if ((st = set_smem(gemm_generic_kernel<1>, shm)) != MCEMU_OK) return st;
      gemm_generic_kernel<1><<<grid, block, shm, s>>>(m, kt, M, N, K, a, lda, b, ldb, C, ldc, D, ldd);
      break;
    case 2:
      if ((st = set_smem(gemm_generic_kernel<2>, shm)) != MCEMU_OK) return st;
      gemm_generic_kernel<2><<<grid, block, shm, s>>>(m, kt, M, N, K, a, lda, b, ldb, C, ldc, D, ldd);
      break;
    default:
      if ((st = set_smem(gemm_generic_kernel<4>, shm)) != MCEMU_OK) return st;
      gemm_generic_kernel<4><<<grid, block, shm, s>>>(m, kt, M, N, K, a, lda, b, ldb, C, ldc, D, ldd);
      break;
  }
  return cudaGetLastError() == cudaSuccess ? MCEMU_OK : MCEMU_ERR_CUDA;
}

int launch_sparse24_gemm(const DevModel &m, int kt, int M, int N, int K, const void *Ac, int64_t ldac,
                         const uint8_t *meta, int64_t ldm, const void *Bt, int64_t ldb,
                         const uint32_t *C, int64_t ldc, uint32_t *D, int64_t ldd, void *stream) {
  cudaStream_t s = (cudaStream_t)stream;
  if (kt > 1024) return MCEMU_ERR_UNSUPPORTED;
  const bool alias = C && overlaps(C, ldc, D, ldd, M, N);
  if (!alias && sparse_fast_ok(m, kt))
    return launch_sparse24_gemm_fast(m, kt, M, N, K, Ac, ldac, meta, ldm, Bt, ldb, C, ldc, D, ldd, stream);
  if (!alias && gemm_exact_ok(m) && m.k % 2 == 0 && 2 * m.k <= 32 && kt <= 64 && elem_size(m) <= 2)
    return launch_sparse24_gemm_exact(m, kt, M, N, K, Ac, ldac, meta, ldm, Bt, ldb, C, ldc, D, ldd, stream);
  const int Kc = K / 2, ktc = kt / 2;
  const size_t shm = (size_t)4 * kT * chunk_len(ktc) * 4;
  dim3 grid((N + kT - 1) / kT, (M + kT - 1) / kT), block(kT, kT);
  const uint8_t *a = (const uint8_t *)Ac, *b = (const uint8_t *)Bt;
  int st;
  switch (elem_size(m)) {
    case 1:
      if ((st = set_smem(sparse_generic_kernel<1>, shm)) != MCEMU_OK) return st;
      sparse_generic_kernel<1><<<grid, block, shm, s>>>(m, ktc, M, N, Kc, a, ldac, meta, ldm, b, ldb, C, ldc, D, ldd);
      break;
    case 2:
      if ((st = set_smem(sparse_generic_kernel<2>, shm)) != MCEMU_OK) return st;
      sparse_generic_kernel<2><<<grid, block, shm, s>>>(m, ktc, M, N, Kc, a, ldac, meta, ldm, b, ldb, C, ldc, D, ldd);
      break;
    default:
      if ((st = set_smem(sparse_generic_kernel<4>, shm)) != MCEMU_OK) return st;
      sparse_generic_kernel<4><<<grid, block, shm, s>>>(m, ktc, M, N, Kc, a, ldac, meta, ldm, b, ldb, C, ldc, D, ldd);
      break;
  }
  return cudaGetLastError() == cudaSuccess ? MCEMU_OK : MCEMU_ERR_CUDA;
}

}  // namespace mcemu

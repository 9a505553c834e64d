// sparse.cu -- 2:4 structured sparsity along K (RDNA4 sparse WMMA page,
// "Structured sparsity (2:4 pattern)"): compression of A into two values and
// one index byte per group of four, and the inverse expansion.
#include <cuda_runtime.h>

#include "core.cuh"

namespace mcemu {

template <int ESZ>
__device__ __forceinline__ uint32_t ld_e(const uint8_t *base, int64_t idx) {
  if constexpr (ESZ == 1) return base[idx];
  else if constexpr (ESZ == 2) return reinterpret_cast<const uint16_t *>(base)[idx];
  else return reinterpret_cast<const uint32_t *>(base)[idx];
}
template <int ESZ>
__device__ __forceinline__ void st_e(uint8_t *base, int64_t idx, uint32_t v) {
  if constexpr (ESZ == 1) base[idx] = (uint8_t)v;
  else if constexpr (ESZ == 2) reinterpret_cast<uint16_t *>(base)[idx] = (uint16_t)v;
  else reinterpret_cast<uint32_t *>(base)[idx] = v;
}

// One thread per (row, group of four).  Zero test: -0 is zero, NaN is nonzero.
// A group with fewer than two nonzeros is padded with its lowest zero positions;
// more than two: the first two are kept and the group is counted.
template <int ESZ>
__global__ void compress_kernel(const FmtDev f, int M, int G, const uint8_t *__restrict__ A, int64_t lda,
                                uint8_t *__restrict__ Ac, int64_t ldac, uint8_t *__restrict__ meta,
                                int64_t ldm, unsigned long long *viol) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (int64_t)M * G) return;
  const int i = (int)(t / G), g = (int)(t % G);
  uint32_t v[4];
  uint32_t nzmask = 0;
#pragma unroll
  for (int q = 0; q < 4; q++) {
    v[q] = ld_e<ESZ>(A, (int64_t)i * lda + 4 * g + q);
    bool zero = f.is_int ? (v[q] & 0xFFu) == 0u : is_zero_elem(f, v[q]);
    nzmask |= (zero ? 0u : 1u) << q;
  }
  int nnz = __popc(nzmask);
  uint32_t keep = nzmask;
  if (nnz > 2) {
    atomicAdd(viol, 1ull);
    keep = nzmask & ~(1u << (31 - __clz(nzmask)));        // drop the highest until two remain
    if (__popc(keep) > 2) keep &= ~(1u << (31 - __clz(keep)));
  }
  uint32_t zeros = ~nzmask & 0xFu;
  while (__popc(keep) < 2) {                               // pad with the lowest zero position
    uint32_t low = zeros & (0u - zeros);
    keep |= low;
    zeros &= ~low;
  }
  int idx0 = __ffs(keep) - 1;
  int idx1 = 31 - __clz(keep);
  st_e<ESZ>(Ac, (int64_t)i * ldac + 2 * g, v[idx0]);
  st_e<ESZ>(Ac, (int64_t)i * ldac + 2 * g + 1, v[idx1]);
  meta[(int64_t)i * ldm + g] = (uint8_t)(idx0 | (idx1 << 2));
}

template <int ESZ>
__global__ void expand_kernel(int M, int G, const uint8_t *__restrict__ Ac, int64_t ldac,
                              const uint8_t *__restrict__ meta, int64_t ldm, uint8_t *__restrict__ A,
                              int64_t lda) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (int64_t)M * G) return;
  const int i = (int)(t / G), g = (int)(t % G);
  uint32_t mb = meta[(int64_t)i * ldm + g];
  uint32_t x0 = ld_e<ESZ>(Ac, (int64_t)i * ldac + 2 * g), x1 = ld_e<ESZ>(Ac, (int64_t)i * ldac + 2 * g + 1);
#pragma unroll
  for (int q = 0; q < 4; q++) {
    uint32_t v = 0;
    if ((int)(mb & 3u) == q) v = x0;
    if ((int)((mb >> 2) & 3u) == q) v = x1;
    st_e<ESZ>(A, (int64_t)i * lda + 4 * g + q, v);
  }
}

int launch_sparse24_compress(const FmtDev &f, int eb, int M, int K, const void *A, int64_t lda, void *Ac,
                             int64_t ldac, uint8_t *meta, int64_t ldm, int64_t *viol, void *stream) {
  cudaStream_t s = (cudaStream_t)stream;
  const int G = K / 4;
  const int64_t total = (int64_t)M * G;
  const int grid = (int)((total + 255) / 256);
  auto *vp = reinterpret_cast<unsigned long long *>(viol);
  if (eb == 1) compress_kernel<1><<<grid, 256, 0, s>>>(f, M, G, (const uint8_t *)A, lda, (uint8_t *)Ac, ldac, meta, ldm, vp);
  else if (eb == 2) compress_kernel<2><<<grid, 256, 0, s>>>(f, M, G, (const uint8_t *)A, lda, (uint8_t *)Ac, ldac, meta, ldm, vp);
  else compress_kernel<4><<<grid, 256, 0, s>>>(f, M, G, (const uint8_t *)A, lda, (uint8_t *)Ac, ldac, meta, ldm, vp);
  return cudaGetLastError() == cudaSuccess ? MCEMU_OK : MCEMU_ERR_CUDA;
}

int launch_sparse24_expand(int eb, int M, int K, const void *Ac, int64_t ldac, const uint8_t *meta, int64_t ldm,
                           void *A, int64_t lda, void *stream) {
  cudaStream_t s = (cudaStream_t)stream;
  const int G = K / 4;
  const int64_t total = (int64_t)M * G;
  const int grid = (int)((total + 255) / 256);
  if (eb == 1) expand_kernel<1><<<grid, 256, 0, s>>>(M, G, (const uint8_t *)Ac, ldac, meta, ldm, (uint8_t *)A, lda);
  else if (eb == 2) expand_kernel<2><<<grid, 256, 0, s>>>(M, G, (const uint8_t *)Ac, ldac, meta, ldm, (uint8_t *)A, lda);
  else expand_kernel<4><<<grid, 256, 0, s>>>(M, G, (const uint8_t *)Ac, ldac, meta, ldm, (uint8_t *)A, lda);
  return cudaGetLastError() == cudaSuccess ? MCEMU_OK : MCEMU_ERR_CUDA;
}

}  // namespace mcemu

// gemm_exact.cu -- tile GEMM for the exact-then-round model (CDNA 1, "Accurate Models
// of AMD Matrix Cores", Secs. 4.1.1-4.1.3): every block FMA of the chain is the
// correctly rounded value of c + sum a_l * b_l.
//
// Same CTA layout as the global-alignment kernels (64 x KC panels in shared memory,
// 4 x 4 outputs per thread), but the panels hold each element's exact fp32 value and
// the block FMA runs on the FP32 pipe: with every element within 2^(+-60), products of
// at most 22 significant bits are exact normal fp32 values, and Knuth's TwoSum carries
// the accumulator c through the block error-free.  The errors are summed by TwoSum as
// well, so S = s + E + sum f exactly, and the leftovers f give the bound: it is 0 when
// the error sum is exact, which decides the exact ties that few-bit products (BF16)
// often produce.  exact_fp32_round then decides the rounding as in the stream kernels.  An element outside
// that range, an Inf/NaN, a rounding the bound leaves undecided or a result below
// 2^-124 or above the fp32 range marks the output, and the fixup pass evaluates its
// whole chain with the general evaluator.
#include "gemm_fast.cuh"

namespace mcemu {

// An element's exact fp32 value, or true (and 0) for an Inf/NaN or a nonzero value
// outside [2^-60, 2^61).
__device__ __forceinline__ bool stage_float(const FmtDev &f, uint32_t x, float &v) {
  uint32_t S, neg;
  int32_t E;
  decode(f, x, S, E, neg);                           // value = S * 2^(E - m_eff), S < 2^24
  const bool bad = classify(f, x) != 0u || (S != 0u && (E < -60 || E > 60));
  const float w = __fmul_rn(__uint2float_rn(S), __uint_as_float((uint32_t)(E - f.m_eff + 127) << 23));
  v = (bad || S == 0u) ? 0.0f : (neg ? -w : w);
  return bad;
}

// Stage one K-chunk of the CTA's A rows and B columns as fp32 values, element (r, q)
// at [q][r]; a row or column with an element stage_float rejects (or, for SPARSE,
// invalid metadata) is flagged.
template <int ESZ, int SPARSE>
__device__ __forceinline__ void stage_chunk_f(const DevModel &m, int i0, int j0, int k0, int kc, int KC, int M,
                                              int N, const uint8_t *__restrict__ A, int64_t lda,
                                              const uint8_t *__restrict__ meta, int64_t ldm,
                                              const uint8_t *__restrict__ Bt, int64_t ldb, float *aF, float *bF,
                                              uint8_t *aSpec, uint8_t *bSpec) {
  for (int e = threadIdx.x; e < kFB * KC; e += blockDim.x) {
    const int r = e / KC, q = e % KC;
    float v = 0.0f;
    if constexpr (SPARSE) {
      if (i0 + r < M && q < kc) {
        const int kd = k0 + q, g = kd >> 2, p = kd & 3;
        const uint32_t mb = meta[(int64_t)(i0 + r) * ldm + g];
        const uint32_t idx0 = mb & 3u, idx1 = (mb >> 2) & 3u;
        if (idx0 >= idx1) aSpec[r] = 1;                  // not a valid 2:4 pattern
        const int t = (p == (int)idx0) ? 0 : (p == (int)idx1) ? 1 : -1;
        if (t >= 0 && stage_float(m.fa, fld<ESZ>(A, (int64_t)(i0 + r) * lda + 2 * g + t), v)) aSpec[r] = 1;
      }
    } else {
      if (i0 + r < M && q < kc && stage_float(m.fa, fld<ESZ>(A, (int64_t)(i0 + r) * lda + k0 + q), v))
        aSpec[r] = 1;
    }
    aF[q * kFS + r] = v;
    v = 0.0f;
    if (j0 + r < N && q < kc && stage_float(m.fb, fld<ESZ>(Bt, (int64_t)(j0 + r) * ldb + k0 + q), v))
      bSpec[r] = 1;
    bF[q * kFS + r] = v;
  }
}

template <int ESZ, int SPARSE, int RM>
__global__ void __launch_bounds__(kFThreads, 2) gemm_exact_kernel(const __grid_constant__ DevModel m, int kt,
                                                                int kblk, int M, int N, int K,
                                                                const uint8_t *__restrict__ A, int64_t lda,
                                                                const uint8_t *__restrict__ meta, int64_t ldm,
                                                                const uint8_t *__restrict__ Bt, int64_t ldb,
                                                                const uint32_t *C, int64_t ldc, uint32_t *D,
                                                                int64_t ldd) {
  extern __shared__ float xsm[];
  const int KC = fast_chunk(kt);
  float *aF = xsm, *bF = aF + KC * kFS;                // [KC][kFS]
  uint8_t *aSpec = reinterpret_cast<uint8_t *>(bF + KC * kFS);
  uint8_t *bSpec = aSpec + kFB;
  const int i0 = blockIdx.y * kFB, j0 = blockIdx.x * kFB;
  const int tid = threadIdx.x;
  const int ti = (tid / (kFB / kFT)) * kFT, tj = (tid % (kFB / kFT)) * kFT;

  float acc[kFT][kFT];
  uint32_t redo = 0;
#pragma unroll
  for (int a = 0; a < kFT; a++)
#pragma unroll
    for (int b = 0; b < kFT; b++) {
      const int i = i0 + ti + a, j = j0 + tj + b;
      uint32_t cb = (C && i < M && j < N) ? C[(int64_t)i * ldc + j] : 0u;
      if ((cb & 0x7F800000u) == 0x7F800000u) redo |= 1u << (a * kFT + b);
      if (m.c_sub_keep == 0u && (cb & 0x7F800000u) == 0u) cb &= 0x80000000u;   // flushed subnormal c
      acc[a][b] = __uint_as_float(cb);
    }

  for (int k0 = 0; k0 < K; k0 += KC) {
    const int kc = min(KC, K - k0);
    __syncthreads();
    if (tid < kFB) { aSpec[tid] = 0; bSpec[tid] = 0; }
    __syncthreads();
    stage_chunk_f<ESZ, SPARSE>(m, i0, j0, k0, kc, KC, M, N, A, lda, meta, ldm, Bt, ldb, aF, bF, aSpec, bSpec);
    __syncthreads();
#pragma unroll
    for (int a = 0; a < kFT; a++)
      if (aSpec[ti + a]) redo |= 0xFu << (a * kFT);
#pragma unroll
    for (int b = 0; b < kFT; b++)
      if (bSpec[tj + b]) redo |= 0x1111u << b;

    for (int s0 = 0; s0 < kc; s0 += kt) {
      const int send = min(s0 + kt, kc);
      for (int b0 = s0; b0 < send; b0 += kblk) {
        const int nt = min(kblk, send - b0);
        // ---- the block's products, each added to c by TwoSum; the errors summed by
        // TwoSum, with the leftovers' magnitudes rounded upward into the bound
        float es[kFT][kFT], ea[kFT][kFT];
#pragma unroll
        for (int a = 0; a < kFT; a++)
#pragma unroll
          for (int b = 0; b < kFT; b++) es[a][b] = ea[a][b] = 0.0f;
        for (int q = b0; q < b0 + nt; q++) {
          const float4 fa = *reinterpret_cast<const float4 *>(aF + q * kFS + ti);
          const float4 fb = *reinterpret_cast<const float4 *>(bF + q * kFS + tj);
          const float xa[4] = {fa.x, fa.y, fa.z, fa.w}, xb[4] = {fb.x, fb.y, fb.z, fb.w};
#pragma unroll
          for (int a = 0; a < kFT; a++)
#pragma unroll
            for (int b = 0; b < kFT; b++) {
              float e, f;
              two_sum(acc[a][b], __fmul_rn(xa[a], xb[b]), acc[a][b], e);
              two_sum(es[a][b], e, es[a][b], f);
              ea[a][b] = __fadd_ru(ea[a][b], fabsf(f));
            }
        }
        // ---- the correctly rounded block result
#pragma unroll
        for (int a = 0; a < kFT; a++)
#pragma unroll
          for (int b = 0; b < kFT; b++) {
            uint32_t r = 0u;
            if (exact_fp32_round(acc[a][b], es[a][b], ea[a][b], RM, r)) redo |= 1u << (a * kFT + b);
            acc[a][b] = __uint_as_float(r);
          }
      }
    }
  }
  // flagged outputs get the mark; gemm_fixup_kernel recomputes them afterwards
#pragma unroll
  for (int a = 0; a < kFT; a++)
#pragma unroll
    for (int b = 0; b < kFT; b++) {
      const int i = i0 + ti + a, j = j0 + tj + b;
      if (i < M && j < N)
        D[(int64_t)i * ldd + j] = ((redo >> (a * kFT + b)) & 1u) ? redo_mark(m) : __float_as_uint(acc[a][b]);
    }
}

// Whole chains of the outputs gemm_exact_kernel marked, one output per thread.  Each
// block FMA is first evaluated as in that kernel (exact fp32 values, TwoSum with an
// error-free error sum); only a block that path does not decide (an element outside
// 2^(+-60), an Inf/NaN, a flushed subnormal c, an undecided rounding) takes the general
// evaluator.  A marked output thus costs about one fast chain instead of a general
// one.  SPARSE chains run over the compressed terms (kt, K dense sizes).
template <int ESZ, int SPARSE>
__global__ void __launch_bounds__(256) gemm_exact_fixup_kernel(const __grid_constant__ DevModel m, int kt, int M,
                                                               int N, int K, const uint8_t *__restrict__ A,
                                                               int64_t lda, const uint8_t *__restrict__ meta,
                                                               int64_t ldm, const uint8_t *__restrict__ Bt,
                                                               int64_t ldb, const uint32_t *C, int64_t ldc,
                                                               uint32_t *D, int64_t ldd) {
  const int64_t tix = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (tix >= (int64_t)M * N) return;
  const int i = (int)(tix / N), j = (int)(tix % N);
  if (D[(int64_t)i * ldd + j] != redo_mark(m)) return;
  const int Kc = SPARSE ? K / 2 : K, ktc = SPARSE ? kt / 2 : kt;
  uint32_t ea[32], eb[32];
  uint32_t acc = C ? C[(int64_t)i * ldc + j] : 0u;
  for (int s0 = 0; s0 < Kc; s0 += ktc) {
    const int send = min(s0 + ktc, Kc);
    for (int b0 = s0; b0 < send; b0 += m.k) {
      const int nt = min(m.k, send - b0);
      bool ok = (acc & 0x7F800000u) != 0x7F800000u &&
                !(m.c_sub_keep == 0u && (acc & 0x7F800000u) == 0u && (acc & 0x7FFFFFu) != 0u);
      float sv = __uint_as_float(acc), es = 0.0f, bnd = 0.0f;
      for (int l = 0; l < nt; l++) {
        const int kc = b0 + l;
        if constexpr (SPARSE) {
          const uint32_t mb = meta[(int64_t)i * ldm + kc / 2];
          const uint32_t idx = (kc & 1) ? ((mb >> 2) & 3u) : (mb & 3u);
          ea[l] = fld<ESZ>(A, (int64_t)i * lda + kc);
          eb[l] = fld<ESZ>(Bt, (int64_t)j * ldb + 4 * (kc / 2) + idx);
          if ((mb & 3u) >= ((mb >> 2) & 3u)) ok = false;   // not a valid 2:4 pattern
        } else {
          ea[l] = fld<ESZ>(A, (int64_t)i * lda + kc);
          eb[l] = fld<ESZ>(Bt, (int64_t)j * ldb + kc);
        }
        float va, vb, e, f;
        if (stage_float(m.fa, ea[l], va) || stage_float(m.fb, eb[l], vb)) ok = false;
        two_sum(sv, __fmul_rn(va, vb), sv, e);
        two_sum(es, e, es, f);
        bnd = __fadd_ru(bnd, fabsf(f));
      }
      uint32_t r = 0u;
      if (!ok || exact_fp32_round(sv, es, bnd, m.rne, r)) r = block_eval_generic(m, ea, eb, nt, acc);
      acc = r;
    }
  }
  D[(int64_t)i * ldd + j] = acc;
}

// true when the exact kernel implements the model (float operands of at most 11
// significand bits, so that products have at most 22)
bool gemm_exact_ok(const DevModel &m) {
  if (m.fa.is_int || m.fb.is_int || m.arch != MCEMU_ARCH_EXACT || m.acc16) return false;
  return m.mab <= 22 && m.k <= 32;
}

template <int ESZ, int SPARSE>
static int run_exact(const DevModel &m, int kt, int kblk, int M, int N, int K, const void *A, int64_t lda,
                     const uint8_t *meta, int64_t ldm, const void *Bt, int64_t ldb, const uint32_t *C, int64_t ldc,
                     uint32_t *D, int64_t ldd, cudaStream_t s) {
  const size_t shm = (size_t)2 * fast_chunk(kt) * kFS * 4 + 2 * kFB;
  auto kern = m.rne ? gemm_exact_kernel<ESZ, SPARSE, 1> : gemm_exact_kernel<ESZ, SPARSE, 0>;
  if (shm > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)shm) != cudaSuccess)
    return MCEMU_ERR_UNSUPPORTED;
  dim3 grid((N + kFB - 1) / kFB, (M + kFB - 1) / kFB);
  kern<<<grid, kFThreads, shm, s>>>(m, kt, kblk, M, N, K, (const uint8_t *)A, lda, meta, ldm,
                                    (const uint8_t *)Bt, ldb, C, ldc, D, ldd);
  if (cudaGetLastError() != cudaSuccess) return MCEMU_ERR_CUDA;
  const int64_t total = (int64_t)M * N;
  gemm_exact_fixup_kernel<ESZ, SPARSE><<<(unsigned)((total + 255) / 256), 256, 0, s>>>(
      m, kt, M, N, K, (const uint8_t *)A, lda, meta, ldm, (const uint8_t *)Bt, ldb, C, ldc, D, ldd);
  return cudaGetLastError() == cudaSuccess ? MCEMU_OK : MCEMU_ERR_CUDA;
}

int launch_tile_gemm_exact(const DevModel &m, int kt, int M, int N, int K, const void *A, int64_t lda,
                           const void *Bt, int64_t ldb, const uint32_t *C, int64_t ldc, uint32_t *D, int64_t ldd,
                           void *stream) {
  cudaStream_t s = (cudaStream_t)stream;
  if (kt > 64 || !gemm_exact_ok(m)) return MCEMU_ERR_UNSUPPORTED;
  const int eb = (int)(m.fa.sshift + 1) / 8;
  if (eb == 1) return run_exact<1, 0>(m, kt, m.k, M, N, K, A, lda, nullptr, 0, Bt, ldb, C, ldc, D, ldd, s);
  if (eb == 2) return run_exact<2, 0>(m, kt, m.k, M, N, K, A, lda, nullptr, 0, Bt, ldb, C, ldc, D, ldd, s);
  return run_exact<4, 0>(m, kt, m.k, M, N, K, A, lda, nullptr, 0, Bt, ldb, C, ldc, D, ldd, s);
}

// 2:4-sparse chain through the same kernel (A expanded while staging, blocks of
// 2 N_FMA dense positions; the expansion's zero products add nothing to an exact sum)
int launch_sparse24_gemm_exact(const DevModel &m, int kt, int M, int N, int K, const void *Ac, int64_t ldac,
                               const uint8_t *meta, int64_t ldm, const void *Bt, int64_t ldb, const uint32_t *C,
                               int64_t ldc, uint32_t *D, int64_t ldd, void *stream) {
  cudaStream_t s = (cudaStream_t)stream;
  const int eb = (int)(m.fa.sshift + 1) / 8;
  if (kt > 64 || !gemm_exact_ok(m) || m.k % 2 != 0 || 2 * m.k > 32 || eb > 2) return MCEMU_ERR_UNSUPPORTED;
  if (eb == 1) return run_exact<1, 1>(m, kt, 2 * m.k, M, N, K, Ac, ldac, meta, ldm, Bt, ldb, C, ldc, D, ldd, s);
  return run_exact<2, 1>(m, kt, 2 * m.k, M, N, K, Ac, ldac, meta, ldm, Bt, ldb, C, ldc, D, ldd, s);
}

}  // namespace mcemu

// gemm_exact.cu -- tile GEMM for the exact-then-round model (CDNA 1, "Accurate Models
// of AMD Matrix Cores", Secs. 4.1.1-4.1.3): every block FMA of the chain is the
// correctly rounded value of c + sum a_l * b_l.
//
// Same CTA layout as the global-alignment kernel (decoded 64 x KC panels in shared
// memory, 4 x 4 outputs per thread).  Per block and output, T bounds the top bit of
// every term; the terms are floored into a 64-bit window of units 2^L, L = T - 61 +
// ceil(log2(terms)), by one arithmetic shift each.  When no term lost bits the window
// holds the exact sum and one rounding finishes the block.  Otherwise the true sum
// lies in [W, W + terms) units; when |W| >= 2^26 the rounding boundaries of that
// range are multiples of 4 units and the rounding of 4W and 4(W + terms) - 1 (units
// of 2^(L-2)) brackets it: equal results are the correctly rounded sum.  Anything else
// (a special value, heavy cancellation, a subnormal result) marks the output, and the
// fixup pass evaluates its whole chain with the general evaluator.
#include "gemm_fast.cuh"

namespace mcemu {

template <int ESZ, int SPARSE>
__global__ void __launch_bounds__(kFThreads, 2) gemm_exact_kernel(const __grid_constant__ DevModel m, int kt,
                                                                int kblk, int logk, int M, int N, int K,
                                                                const uint8_t *__restrict__ A, int64_t lda,
                                                                const uint8_t *__restrict__ meta, int64_t ldm,
                                                                const uint8_t *__restrict__ Bt, int64_t ldb,
                                                                const uint32_t *C, int64_t ldc, uint32_t *D,
                                                                int64_t ldd) {
  extern __shared__ int32_t fsm[];
  const int KC = fast_chunk(kt);
  int32_t *aS = fsm, *aE = aS + KC * kFS, *aG = aE + KC * kFS;
  int32_t *bS = aG + KC * kFS, *bE = bS + KC * kFS, *bG = bE + KC * kFS;
  uint8_t *aSpec = reinterpret_cast<uint8_t *>(bG + KC * kFS);
  uint8_t *bSpec = aSpec + kFB;
  const int i0 = blockIdx.y * kFB, j0 = blockIdx.x * kFB;
  const int tid = threadIdx.x;
  const int ti = (tid / (kFB / kFT)) * kFT, tj = (tid % (kFB / kFT)) * kFT;
  // B significands pre-shifted so that S_a * S_b' = U * 2^(28 - mab) < 2^30 and a
  // product placed in the high word of a 64-bit value is U * 2^(60 - mab)
  const int qs = 28 - m.mab;

  uint32_t acc[kFT][kFT];
#pragma unroll
  for (int a = 0; a < kFT; a++)
#pragma unroll
    for (int b = 0; b < kFT; b++) {
      const int i = i0 + ti + a, j = j0 + tj + b;
      acc[a][b] = (C && i < M && j < N) ? C[(int64_t)i * ldc + j] : 0u;
    }

  uint32_t redo = 0;
  for (int k0 = 0; k0 < K; k0 += KC) {
    const int kc = min(KC, K - k0);
    __syncthreads();
    if (tid < kFB) { aSpec[tid] = 0; bSpec[tid] = 0; }
    __syncthreads();
    stage_chunk<ESZ, SPARSE>(m, qs, i0, j0, k0, kc, KC, M, N, A, lda, meta, ldm, Bt, ldb, aS, aE, aG, bS, bE, bG,
                             aSpec, bSpec);
    __syncthreads();
    uint32_t rowsp = 0, colsp = 0;
#pragma unroll
    for (int a = 0; a < kFT; a++) rowsp |= (uint32_t)aSpec[ti + a] << a;
#pragma unroll
    for (int b = 0; b < kFT; b++) colsp |= (uint32_t)bSpec[tj + b] << b;

    for (int s0 = 0; s0 < kc; s0 += kt) {
      const int send = min(s0 + kt, kc);
      for (int b0 = s0; b0 < send; b0 += kblk) {
        const int nt = min(kblk, send - b0);
        // ---- pass 1: the largest product exponent E_a + E_b
        int32_t T[kFT][kFT];
#pragma unroll
        for (int a = 0; a < kFT; a++)
#pragma unroll
          for (int b = 0; b < kFT; b++) T[a][b] = kNegE;
        for (int q = b0; q < b0 + nt; q++) {
          const int4 ea = *reinterpret_cast<const int4 *>(aE + q * kFS + ti);
          const int4 eb = *reinterpret_cast<const int4 *>(bE + q * kFS + tj);
          const int32_t xa[4] = {ea.x, ea.y, ea.z, ea.w}, xb[4] = {eb.x, eb.y, eb.z, eb.w};
#pragma unroll
          for (int a = 0; a < kFT; a++)
#pragma unroll
            for (int b = 0; b < kFT; b++) T[a][b] = __viaddmax_s32(xa[a], xb[b], T[a][b]);
        }
        // ---- the window of each output, with c placed in it
        int64_t W[kFT][kFT];
        int32_t C1[kFT][kFT];
        uint32_t st[kFT][kFT];                               // nonzero once a term lost bits
        uint32_t nzm = 0;                                    // outputs with a nonzero product or c
        uint32_t ovm = 0;                                    // outputs whose products may reach 2^128
#pragma unroll
        for (int a = 0; a < kFT; a++)
#pragma unroll
          for (int b = 0; b < kFT; b++) {
            uint32_t cS, cneg;
            int32_t cE;
            decode_c(m, acc[a][b], cS, cE, cneg);
            if (T[a][b] > -1024 || cS) nzm |= 1u << (a * kFT + b);
            if (m.prod_ovf && T[a][b] >= 126) ovm |= 1u << (a * kFT + b);   // CDNA 3 product overflow
            int32_t top = T[a][b] + 2;                       // products: |p| < 2^(E_a + E_b + 2)
            if (cS) top = max(top, cE + 1);
            const int32_t L = top - 61 + logk;
            T[a][b] = L;
            C1[a][b] = 60 + L;
            W[a][b] = 0;
            st[a][b] = 0;
            if (cS) {
              const int32_t sv = cneg ? -(int32_t)cS : (int32_t)cS;
              const uint32_t hv = (uint32_t)sv << 6;
              const int32_t r = 61 - cE + L;
              W[a][b] = ((int64_t)((uint64_t)hv << 32)) >> min(r, 63);   // c * 2^38, floored
              st[a][b] = shl_clamp(hv, (uint32_t)max(64 - r, 0));
            }
          }
        // ---- pass 2: the products, floored into the window
        for (int q = b0; q < b0 + nt; q++) {
          const int4 sa = *reinterpret_cast<const int4 *>(aS + q * kFS + ti);
          const int4 ea = *reinterpret_cast<const int4 *>(aE + q * kFS + ti);
          const int4 ga = *reinterpret_cast<const int4 *>(aG + q * kFS + ti);
          const int4 sb = *reinterpret_cast<const int4 *>(bS + q * kFS + tj);
          const int4 eb = *reinterpret_cast<const int4 *>(bE + q * kFS + tj);
          const int4 gb = *reinterpret_cast<const int4 *>(bG + q * kFS + tj);
          const int32_t SA[4] = {sa.x, sa.y, sa.z, sa.w}, EA[4] = {ea.x, ea.y, ea.z, ea.w}, GA[4] = {ga.x, ga.y, ga.z, ga.w};
          const int32_t SB[4] = {sb.x, sb.y, sb.z, sb.w}, EB[4] = {eb.x, eb.y, eb.z, eb.w}, GB[4] = {gb.x, gb.y, gb.z, gb.w};
#pragma unroll
          for (int a = 0; a < kFT; a++)
#pragma unroll
            for (int b = 0; b < kFT; b++) {
              const int32_t r = C1[a][b] - EA[a] - EB[b];
              const int32_t v = SA[a] * SB[b] * (GA[a] * GB[b]);
              W[a][b] += ((int64_t)((uint64_t)(uint32_t)v << 32)) >> min(r, 63);
              // the bits dropped are the low r - 32 of v (all of v once r >= 64)
              st[a][b] |= shl_clamp((uint32_t)v, (uint32_t)max(64 - r, 0));
            }
        }
        // ---- rounding of the bracket
#pragma unroll
        for (int a = 0; a < kFT; a++)
#pragma unroll
          for (int b = 0; b < kFT; b++) {
            const int64_t w = W[a][b];
            const int32_t L = T[a][b];
            uint32_t lo = 0, hi = 1;
            bool ok = !((((rowsp >> a) | (colsp >> b)) & 1u) || (acc[a][b] & 0x7F800000u) == 0x7F800000u ||
                        ((ovm >> (a * kFT + b)) & 1u)) &&
                      L > kNegE / 2;
            if (st[a][b] == 0u && w == 0)                    // exact zero: +0 unless every term is zero
              ok = ok && ((nzm >> (a * kFT + b)) & 1u);
            else if (st[a][b] == 0u)                         // the window holds the exact sum
              ok = ok && hw_round64_1(w, L, m.rne, lo);
            else
              ok = ok && (w >= (1ll << 26) || w <= -(1ll << 26)) && hw_round64_1(4 * w, L - 2, m.rne, lo) &&
                   hw_round64_1(4 * (w + nt + 1) - 1, L - 2, m.rne, hi) && lo == hi;
            if (!ok) redo |= 1u << (a * kFT + b);
            acc[a][b] = lo;
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
      if (i < M && j < N) D[(int64_t)i * ldd + j] = ((redo >> (a * kFT + b)) & 1u) ? redo_mark(m) : acc[a][b];
    }
}

// true when the exact kernel implements the model (float operands of at most 11
// significand bits, so that products have at most 22)
bool gemm_exact_ok(const DevModel &m) {
  if (m.fa.is_int || m.fb.is_int || m.arch != MCEMU_ARCH_EXACT) return false;
  return m.mab <= 22 && m.k <= 32;
}

template <int ESZ, int SPARSE>
static int run_exact(const DevModel &m, int kt, int kblk, int M, int N, int K, const void *A, int64_t lda,
                     const uint8_t *meta, int64_t ldm, const void *Bt, int64_t ldb, const uint32_t *C, int64_t ldc,
                     uint32_t *D, int64_t ldd, cudaStream_t s) {
  const size_t shm = (size_t)6 * fast_chunk(kt) * kFS * 4 + 2 * kFB;
  auto kern = gemm_exact_kernel<ESZ, SPARSE>;
  if (shm > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)shm) != cudaSuccess)
    return MCEMU_ERR_UNSUPPORTED;
  int logk = 0;
  while ((1 << logk) < kblk + 1) logk++;                 // ceil(log2(products + c))
  dim3 grid((N + kFB - 1) / kFB, (M + kFB - 1) / kFB);
  kern<<<grid, kFThreads, shm, s>>>(m, kt, kblk, logk, M, N, K, (const uint8_t *)A, lda, meta, ldm,
                                    (const uint8_t *)Bt, ldb, C, ldc, D, ldd);
  if (cudaGetLastError() != cudaSuccess) return MCEMU_ERR_CUDA;
  return run_fixup<ESZ, SPARSE>(m, kt, M, N, K, A, lda, meta, ldm, Bt, ldb, C, ldc, D, ldd, s);
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

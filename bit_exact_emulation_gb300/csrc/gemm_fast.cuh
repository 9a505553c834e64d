// gemm_fast.cuh -- tile GEMM for the global-alignment architectures (early c as in
// Table 3, late c as in Algorithm 1 of "Accurate Models of AMD Matrix Cores").
//
// Same chain as gemm.cu (instructions of kt products, N_FMA blocks, the fp32
// accumulator carried as c), organised for the GB300 integer pipes:
//  - a CTA stages a 64 x KC panel of A and of B^T and decodes every element once
//    into shared memory as (significand S, exponent E, sign +-1);
//  - each thread owns a 4 x 4 register tile of outputs; per block FMA it makes two
//    passes over the block's k: the first takes e_max = max(E_a + E_b) with the
//    fused add-max instruction, the second aligns and accumulates the products
//    (IADD3 shift amount, IMAD product, funnel shift, IMAD signed accumulate);
//  - the per-output merge with c and the rounding use the integer helpers of
//    core.cuh with the hardware int->fp32 rounding.
// An output whose chain meets an Inf/NaN input, an Inf/NaN accumulator, a possible
// product overflow, an exact zero sum or a subnormal result is flagged and its
// whole chain is evaluated again at the end with the general evaluator (rare; the
// result is the same model).
#pragma once
#include <cuda_runtime.h>

#include "core.cuh"

namespace mcemu {

constexpr int kFB = 64;                 // CTA tile: kFB x kFB outputs
constexpr int kFT = 4;                  // thread tile: kFT x kFT outputs
constexpr int kFThreads = (kFB / kFT) * (kFB / kFT);
constexpr int32_t kZeroE = -2048;       // exponent of a zero element: never the maximum
constexpr int kFS = kFB + 4;            // panel row stride in words (int4-aligned, fewer bank conflicts)

__host__ __device__ __forceinline__ int fast_chunk(int kt) { return kt >= 32 ? kt : kt * (32 / kt); }

template <int ESZ>
__device__ __forceinline__ uint32_t fld(const uint8_t *base, int64_t idx) {
  if constexpr (ESZ == 1) return base[idx];
  else if constexpr (ESZ == 2) return reinterpret_cast<const uint16_t *>(base)[idx];
  else return reinterpret_cast<const uint32_t *>(base)[idx];
}

// decode one element into the panel; returns 1 when it is Inf/NaN
__device__ __forceinline__ uint32_t stage_elem(const FmtDev &f, uint32_t x, int32_t &S, int32_t &E, int32_t &G) {
  uint32_t s, neg;
  int32_t e;
  decode(f, x, s, e, neg);
  S = (int32_t)s;
  E = s ? e : kZeroE;
  G = neg ? -1 : 1;
  return classify(f, x) != 0u ? 1u : 0u;
}

// Stage one K-chunk of the CTA's A rows and B columns into shared memory, decoded:
// element (r, q) of the chunk goes to [q][r] as significand, exponent (kZeroE for a
// zero) and sign +-1; B significands are shifted left by bshift.  A row or column
// that holds an Inf/NaN (or, for SPARSE, invalid metadata) is flagged.
template <int ESZ, int SPARSE>
__device__ __forceinline__ void stage_chunk(const DevModel &m, int bshift, int i0, int j0, int k0, int kc, int KC,
                                            int M, int N, const uint8_t *__restrict__ A, int64_t lda,
                                            const uint8_t *__restrict__ meta, int64_t ldm,
                                            const uint8_t *__restrict__ Bt, int64_t ldb, int32_t *aS, int32_t *aE,
                                            int32_t *aG, int32_t *bS, int32_t *bE, int32_t *bG, uint8_t *aSpec,
                                            uint8_t *bSpec) {
  for (int e = threadIdx.x; e < kFB * KC; e += blockDim.x) {
    const int r = e / KC, q = e % KC;
    int32_t S = 0, E = kZeroE, G = 1;
    if constexpr (SPARSE) {
      if (i0 + r < M && q < kc) {
        const int kd = k0 + q, g = kd >> 2, p = kd & 3;
        const uint32_t mb = meta[(int64_t)(i0 + r) * ldm + g];
        const uint32_t idx0 = mb & 3u, idx1 = (mb >> 2) & 3u;
        if (idx0 >= idx1) aSpec[r] = 1;                  // not a valid 2:4 pattern
        const int t = (p == (int)idx0) ? 0 : (p == (int)idx1) ? 1 : -1;
        if (t >= 0 && stage_elem(m.fa, fld<ESZ>(A, (int64_t)(i0 + r) * lda + 2 * g + t), S, E, G)) aSpec[r] = 1;
      }
    } else {
      if (i0 + r < M && q < kc && stage_elem(m.fa, fld<ESZ>(A, (int64_t)(i0 + r) * lda + k0 + q), S, E, G))
        aSpec[r] = 1;
    }
    aS[q * kFS + r] = S; aE[q * kFS + r] = E; aG[q * kFS + r] = G;
    S = 0; E = kZeroE; G = 1;
    if (j0 + r < N && q < kc && stage_elem(m.fb, fld<ESZ>(Bt, (int64_t)(j0 + r) * ldb + k0 + q), S, E, G))
      bSpec[r] = 1;
    bS[q * kFS + r] = S << bshift; bE[q * kFS + r] = E; bG[q * kFS + r] = G;
  }
}

// The whole chain of one output with the general evaluator, reading raw operands
// from global memory (outputs that met a case the fast path leaves out); C == nullptr
// stands for C = 0.
template <int ESZ>
__device__ __noinline__ uint32_t chain_generic(const DevModel &m, int kt, int K, const uint8_t *A, int64_t lda,
                                               const uint8_t *Bt, int64_t ldb, int i, int j, const uint32_t *C,
                                               int64_t ldc) {
  uint32_t ea[32], eb[32];
  uint32_t acc = C ? C[(int64_t)i * ldc + j] : 0u;
  for (int s0 = 0; s0 < K; s0 += kt) {
    const int send = min(s0 + kt, K);
    for (int b0 = s0; b0 < send; b0 += m.k) {
      const int nt = min(m.k, send - b0);
      for (int l = 0; l < nt; l++) {
        ea[l] = fld<ESZ>(A, (int64_t)i * lda + b0 + l);
        eb[l] = fld<ESZ>(Bt, (int64_t)j * ldb + b0 + l);
      }
      acc = block_eval_generic(m, ea, eb, nt, acc);
    }
  }
  return acc;
}

// The same for the 2:4-sparse chain: compressed term kc of row i multiplies
// Ac[i][kc] with B[4 (kc / 2) + idx(kc)][j]; blocks of N_FMA compressed terms.
template <int ESZ>
__device__ __noinline__ uint32_t chain_sparse_generic(const DevModel &m, int ktc, int Kc, const uint8_t *Ac,
                                                      int64_t ldac, const uint8_t *meta, int64_t ldm,
                                                      const uint8_t *Bt, int64_t ldb, int i, int j,
                                                      const uint32_t *C, int64_t ldc) {
  uint32_t ea[32], eb[32];
  uint32_t acc = C ? C[(int64_t)i * ldc + j] : 0u;
  for (int s0 = 0; s0 < Kc; s0 += ktc) {
    const int send = min(s0 + ktc, Kc);
    for (int b0 = s0; b0 < send; b0 += m.k) {
      const int nt = min(m.k, send - b0);
      for (int l = 0; l < nt; l++) {
        const int kc = b0 + l;
        const uint32_t mb = meta[(int64_t)i * ldm + kc / 2];
        const uint32_t idx = (kc & 1) ? ((mb >> 2) & 3u) : (mb & 3u);
        ea[l] = fld<ESZ>(Ac, (int64_t)i * ldac + kc);
        eb[l] = fld<ESZ>(Bt, (int64_t)j * ldb + 4 * (kc / 2) + idx);
      }
      acc = block_eval_generic(m, ea, eb, nt, acc);
    }
  }
  return acc;
}

// Early-c merge of one output: S (products and c, aligned and truncated) rounded in
// hardware.  A zero sum is +0 when some term is nonzero; false for a zero sum of zero
// terms (its sign needs the inputs) or a subnormal result.
__device__ __forceinline__ bool merge_early(const DevModel &m, int32_t S, int32_t emax, bool have_nz, uint32_t &r) {
  if (S == 0) {
    r = 0u;
    return have_nz;
  }
  return hw_round32_1(S, emax - m.F, m.rne, r);
}

// Algorithm 1, lines 5-15, for one output with hardware rounding.  A zero sum is +0
// when some product or c is nonzero; false for a zero sum of zero terms or a
// subnormal result (the general evaluator then decides).
__device__ __forceinline__ bool merge_late(const DevModel &m, int32_t Sp, int32_t emax, uint32_t cb, uint32_t &r) {
  uint32_t cS, cneg;
  int32_t cE;
  decode_c(m, cb, cS, cE, cneg);
  const bool have_p = emax > -1024;                      // zero products sit below -1900
  const int32_t ec = cS ? cE : m.c_zero_exp;
  const bool have_c = ec > kNegE / 2;
  if (!have_p && !have_c) return false;
  if (have_p && (!have_c || emax >= ec)) {
    int32_t sc = 0;                                      // line 7: RD to c_frac (= F_p) bits
    if (cS) {
      const int32_t v = cneg ? -(int32_t)cS : (int32_t)cS;
      const int32_t sh = emax - ec + 23 - m.c_frac;
      sc = sh >= 0 ? sar32(v, sh) : v * (1 << (-sh));
    }
    const int32_t Sacc = Sp + sc;                       // line 8
    if (Sacc == 0) {                                     // a nonzero product cancelled: +0
      r = 0u;
      return true;
    }
    return hw_round32_1(Sacc, emax - m.F, m.rne, r);      // line 15
  }
  // line 10: S_p on c's grid with RD (floor) at psum_frac fraction bits; in this branch
  // e_max < e_c, so the shift is at least 1 - (psum_frac - F_p) >= -8 and the product
  // sum, pre-shifted by 16, is floored by one arithmetic shift
  int64_t Sacc = have_p ? (((int64_t)Sp << 16) >> min(ec - emax - (m.psum_frac - m.F) + 16, 63)) : 0;
  const int64_t vc = cneg ? -(int64_t)cS : (int64_t)cS;
  Sacc += vc * ((int64_t)1 << (m.psum_frac - 23));       // line 11
  if (Sacc == 0) {
    r = 0u;
    return have_p || cS != 0u;
  }
  // lines 12-13: normalise (exponent floored at -126) and RD to post_norm_frac bits.
  // The leading bit of |S| is found from S xor its sign: one place lower only when
  // |S| is a power of two, where every lower bit is zero and the RD is exact anyway.
  int32_t lsb = ec - m.psum_frac;
  const int32_t p = 63 - __clzll((long long)(Sacc ^ (Sacc >> 63)));
  const int32_t rsh = max(p + lsb, -126) - m.post_norm_frac - lsb;
  if (rsh > 0) {
    Sacc >>= min(rsh, 63);                               // floor = RD for either sign
    lsb += rsh;
  }
  return hw_round64_1(Sacc, lsb, m.rne, r);                // line 15
}

// A NaN pattern no model returns (their NaN results are always nan_bits): it marks
// an output the fast kernel left to the general evaluator.
__host__ __device__ __forceinline__ uint32_t redo_mark(const DevModel &m) {
  return m.nan_bits == 0x7FFFFFFFu ? 0xFFFFFFFFu : 0x7FFFFFFFu;
}

// C == nullptr stands for C = 0.
//
// SPARSE = 1: A is given 2:4-compressed (Ac [M][K/2], meta [M][K/4]) and is expanded
// into the dense panel while staging; kt and K are then dense sizes and a block spans
// kblk = 2 N_FMA dense positions.  A block of N_FMA compressed terms covers exactly
// those positions (groups of four never straddle blocks), and the positions the
// expansion fills with zeros add zero products, which take no part in e_max and add
// nothing to the aligned sum: the result is the compressed chain's.  The cases where
// that argument needs finite operands, a nonzero sum or valid metadata (idx0 < idx1)
// are the ones sent to the general evaluator of the compressed chain.
template <int ARCH, int ESZ, int SPARSE>
__global__ void __launch_bounds__(kFThreads, 2) gemm_fast_kernel(const __grid_constant__ DevModel m, int kt, int kblk,
                                                               int M, int N, int K, const uint8_t *__restrict__ A,
                                                               int64_t lda, const uint8_t *__restrict__ meta,
                                                               int64_t ldm, const uint8_t *__restrict__ Bt,
                                                               int64_t ldb, const uint32_t *C, int64_t ldc,
                                                               uint32_t *D, int64_t ldd) {
  extern __shared__ int32_t fsm[];
  const int KC = fast_chunk(kt);
  int32_t *aS = fsm, *aE = aS + KC * kFS, *aG = aE + KC * kFS;         // [KC][kFS]
  int32_t *bS = aG + KC * kFS, *bE = bS + KC * kFS, *bG = bE + KC * kFS;  // B significands << P0
  uint8_t *aSpec = reinterpret_cast<uint8_t *>(bG + KC * kFS);          // [kFB] per row
  uint8_t *bSpec = aSpec + kFB;
  const int i0 = blockIdx.y * kFB, j0 = blockIdx.x * kFB;
  const int tid = threadIdx.x;
  const int ti = (tid / (kFB / kFT)) * kFT, tj = (tid % (kFB / kFT)) * kFT;

  uint32_t acc[kFT][kFT];
#pragma unroll
  for (int a = 0; a < kFT; a++)
#pragma unroll
    for (int b = 0; b < kFT; b++) {
      const int i = i0 + ti + a, j = j0 + tj + b;
      acc[a][b] = (C && i < M && j < N) ? C[(int64_t)i * ldc + j] : 0u;
    }

  uint32_t redo = 0;                     // outputs to recompute with the general evaluator
  for (int k0 = 0; k0 < K; k0 += KC) {
    const int kc = min(KC, K - k0);
    __syncthreads();
    if (tid < kFB) { aSpec[tid] = 0; bSpec[tid] = 0; }
    __syncthreads();
    stage_chunk<ESZ, SPARSE>(m, m.P0, i0, j0, k0, kc, KC, M, N, A, lda, meta, ldm, Bt, ldb, aS, aE, aG, bS, bE, bG,
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
        // ---- pass 1: e_max of the products (c joins for the early-c model)
        int32_t emax[kFT][kFT];
#pragma unroll
        for (int a = 0; a < kFT; a++)
#pragma unroll
          for (int b = 0; b < kFT; b++) emax[a][b] = kNegE;
        for (int q = b0; q < b0 + nt; q++) {
          const int4 ea = *reinterpret_cast<const int4 *>(aE + q * kFS + ti);
          const int4 eb = *reinterpret_cast<const int4 *>(bE + q * kFS + tj);
          const int32_t xa[4] = {ea.x, ea.y, ea.z, ea.w}, xb[4] = {eb.x, eb.y, eb.z, eb.w};
#pragma unroll
          for (int a = 0; a < kFT; a++)
#pragma unroll
            for (int b = 0; b < kFT; b++) emax[a][b] = __viaddmax_s32(xa[a], xb[b], emax[a][b]);
        }
        uint32_t hpm = 0;
        // ---- c's exponent (early c) and the shift base
        int32_t base[kFT][kFT];
        int32_t Sp[kFT][kFT];
#pragma unroll
        for (int a = 0; a < kFT; a++)
#pragma unroll
          for (int b = 0; b < kFT; b++) {
            int32_t em = emax[a][b];
            Sp[a][b] = 0;
            if constexpr (ARCH == MCEMU_ARCH_GA_EARLY) {
              // c joins e_max and is aligned here, so the sum starts with its term
              uint32_t cS, cneg;
              int32_t cE;
              decode_c(m, acc[a][b], cS, cE, cneg);
              const int32_t ec = cS ? cE : m.c_zero_exp;
              em = max(max(em, ec), m.emin_lim);
              if (emax[a][b] > -1024 || cS) hpm |= 1u << (a * kFT + b);   // a nonzero term
              emax[a][b] = em;
              if (cS)                                     // truncation (the kernel takes no RD model)
                Sp[a][b] = (int32_t)shr32(cS * m.p0cmul, em + m.R0c - cE) * (1 - 2 * (int32_t)cneg);
            }
            base[a][b] = em + m.R0;
          }
        // ---- pass 2: aligned, truncated products
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
              const int32_t sh = base[a][b] - EA[a] - EB[b];
              const uint32_t U = (uint32_t)(SA[a] * SB[b]);
              const int32_t t = (int32_t)shr32(U, sh);
              Sp[a][b] += t * (GA[a] * GB[b]);
            }
        }
        // ---- merge with c and round; outputs that leave the fast path are redone
#pragma unroll
        for (int a = 0; a < kFT; a++)
#pragma unroll
          for (int b = 0; b < kFT; b++) {
            const uint32_t cb = acc[a][b];
            uint32_t r = 0;
            bool ok = !((((rowsp >> a) | (colsp >> b)) & 1u) || (cb & 0x7F800000u) == 0x7F800000u ||
                        (m.prod_ovf && emax[a][b] >= 126));
            if (ok) {
              if constexpr (ARCH == MCEMU_ARCH_GA_EARLY)
                ok = merge_early(m, Sp[a][b], emax[a][b], (hpm >> (a * kFT + b)) & 1u, r);
              else ok = merge_late(m, Sp[a][b], emax[a][b], cb, r);
            }
            if (!ok) redo |= 1u << (a * kFT + b);
            acc[a][b] = r;
          }
      }
    }
  }
  // flagged outputs get the mark; gemm_fixup_kernel recomputes them afterwards (C
  // does not alias D on this path).  Keeping the general evaluator out of this kernel
  // keeps its register allocation free of a call.
#pragma unroll
  for (int a = 0; a < kFT; a++)
#pragma unroll
    for (int b = 0; b < kFT; b++) {
      const int i = i0 + ti + a, j = j0 + tj + b;
      if (i < M && j < N) D[(int64_t)i * ldd + j] = ((redo >> (a * kFT + b)) & 1u) ? redo_mark(m) : acc[a][b];
    }
}

// Whole chains of the outputs a fast kernel marked, one output per thread.
template <int ESZ, int SPARSE>
__global__ void __launch_bounds__(256) gemm_fixup_kernel(const __grid_constant__ DevModel m, int kt, int M, int N,
                                                         int K, const uint8_t *__restrict__ A, int64_t lda,
                                                         const uint8_t *__restrict__ meta, int64_t ldm,
                                                         const uint8_t *__restrict__ Bt, int64_t ldb,
                                                         const uint32_t *C, int64_t ldc, uint32_t *D, int64_t ldd) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (int64_t)M * N) return;
  const int i = (int)(t / N), j = (int)(t % N);
  if (D[(int64_t)i * ldd + j] != redo_mark(m)) return;
  uint32_t r;
  if constexpr (SPARSE) r = chain_sparse_generic<ESZ>(m, kt / 2, K / 2, A, lda, meta, ldm, Bt, ldb, i, j, C, ldc);
  else r = chain_generic<ESZ>(m, kt, K, A, lda, Bt, ldb, i, j, C, ldc);
  D[(int64_t)i * ldd + j] = r;
}

template <int ESZ, int SPARSE>
static int run_fixup(const DevModel &m, int kt, int M, int N, int K, const void *A, int64_t lda,
                     const uint8_t *meta, int64_t ldm, const void *Bt, int64_t ldb, const uint32_t *C, int64_t ldc,
                     uint32_t *D, int64_t ldd, cudaStream_t s) {
  const int64_t total = (int64_t)M * N;
  gemm_fixup_kernel<ESZ, SPARSE><<<(unsigned)((total + 255) / 256), 256, 0, s>>>(
      m, kt, M, N, K, (const uint8_t *)A, lda, meta, ldm, (const uint8_t *)Bt, ldb, C, ldc, D, ldd);
  return cudaGetLastError() == cudaSuccess ? MCEMU_OK : MCEMU_ERR_CUDA;
}

template <int ARCH, int ESZ, int SPARSE = 0>
static int run_fast(const DevModel &m, int kt, int M, int N, int K, const void *A, int64_t lda, const void *Bt,
                    int64_t ldb, const uint32_t *C, int64_t ldc, uint32_t *D, int64_t ldd, cudaStream_t s,
                    const uint8_t *meta = nullptr, int64_t ldm = 0) {
  const size_t shm = (size_t)6 * fast_chunk(kt) * kFS * 4 + 2 * kFB;
  auto kern = gemm_fast_kernel<ARCH, ESZ, SPARSE>;
  if (shm > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)shm) != cudaSuccess)
    return MCEMU_ERR_UNSUPPORTED;
  dim3 grid((N + kFB - 1) / kFB, (M + kFB - 1) / kFB);
  const int kblk = SPARSE ? 2 * m.k : m.k;
  kern<<<grid, kFThreads, shm, s>>>(m, kt, kblk, M, N, K, (const uint8_t *)A, lda, meta, ldm, (const uint8_t *)Bt,
                                    ldb, C, ldc, D, ldd);
  if (cudaGetLastError() != cudaSuccess) return MCEMU_ERR_CUDA;
  return run_fixup<ESZ, SPARSE>(m, kt, M, N, K, A, lda, meta, ldm, Bt, ldb, C, ldc, D, ldd, s);
}

}  // namespace mcemu

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
//  - between blocks the accumulator is an integer-valued float f and a scale g
//    (value f * 2^g): c is aligned by one exact multiply and a float->int conversion,
//    and the block's rounding is the int->fp32 conversion, so no fp32 encode or
//    decode runs per block.
// An output whose chain meets an Inf/NaN input or addend, a possible product overflow,
// a zero sum of zero terms, or a result outside the normal fp32 range is flagged, and
// its whole chain is evaluated again at the end with the general evaluator (rare; the
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
// that holds an Inf/NaN is flagged.
template <int ESZ>
__device__ __forceinline__ void stage_chunk(const DevModel &m, int bshift, int i0, int j0, int k0, int kc, int KC,
                                            int M, int N, const uint8_t *__restrict__ A, int64_t lda,
                                            const uint8_t *__restrict__ Bt, int64_t ldb, int32_t *aS, int32_t *aE,
                                            int32_t *aG, int32_t *bS, int32_t *bE, int32_t *bG, uint8_t *aSpec,
                                            uint8_t *bSpec) {
  for (int e = threadIdx.x; e < kFB * KC; e += blockDim.x) {
    const int r = e / KC, q = e % KC;
    int32_t S = 0, E = kZeroE, G = 1;
    if (i0 + r < M && q < kc && stage_elem(m.fa, fld<ESZ>(A, (int64_t)(i0 + r) * lda + k0 + q), S, E, G))
      aSpec[r] = 1;
    aS[q * kFS + r] = S; aE[q * kFS + r] = E; aG[q * kFS + r] = G;
    S = 0; E = kZeroE; G = 1;
    if (j0 + r < N && q < kc && stage_elem(m.fb, fld<ESZ>(Bt, (int64_t)(j0 + r) * ldb + k0 + q), S, E, G))
      bSpec[r] = 1;
    bS[q * kFS + r] = S << bshift; bE[q * kFS + r] = E; bG[q * kFS + r] = G;
  }
}

// The gather form of the 2:4-sparse GEMM (SPARSE = 1): a chunk holds KCA compressed
// terms of A (compressed k0c .. k0c + kcc) and the 2 KCA dense rows of B^T they draw on.
// Compressed term q of row r goes to [q][r] as (S, E, sign) plus, in aI, the offset of
// its B row in the panel, (4 (q / 2) + idx) * kFS with idx the metadata index of its
// group (k0c is even, so a chunk starts on a group).  A row with invalid metadata
// (idx0 >= idx1) or an Inf/NaN, and a column of B with an Inf/NaN, are flagged.
template <int ESZ>
__device__ __forceinline__ void stage_chunk_gather(const DevModel &m, int bshift, int i0, int j0, int k0c, int kcc,
                                                   int KCA, int M, int N, const uint8_t *__restrict__ Ac, int64_t ldac,
                                                   const uint8_t *__restrict__ meta, int64_t ldm,
                                                   const uint8_t *__restrict__ Bt, int64_t ldb, int32_t *aS,
                                                   int32_t *aE, int32_t *aG, int32_t *aI, int32_t *bS, int32_t *bE,
                                                   int32_t *bG, uint8_t *aSpec, uint8_t *bSpec) {
  for (int e = threadIdx.x; e < kFB * KCA; e += blockDim.x) {
    const int r = e / KCA, q = e % KCA;
    int32_t S = 0, E = kZeroE, G = 1, I = 0;
    if (i0 + r < M && q < kcc) {
      const int kq = k0c + q;
      const uint32_t mb = meta[(int64_t)(i0 + r) * ldm + (kq >> 1)];
      const uint32_t idx0 = mb & 3u, idx1 = (mb >> 2) & 3u;
      if (idx0 >= idx1) aSpec[r] = 1;                    // not a valid 2:4 pattern
      I = (4 * (q >> 1) + (int)((kq & 1) ? idx1 : idx0)) * kFS;
      if (stage_elem(m.fa, fld<ESZ>(Ac, (int64_t)(i0 + r) * ldac + kq), S, E, G)) aSpec[r] = 1;
    }
    aS[q * kFS + r] = S; aE[q * kFS + r] = E; aG[q * kFS + r] = G; aI[q * kFS + r] = I;
  }
  const int KB = 2 * KCA, kb = 2 * kcc, k0 = 2 * k0c;
  for (int e = threadIdx.x; e < kFB * KB; e += blockDim.x) {
    const int r = e / KB, q = e % KB;
    int32_t S = 0, E = kZeroE, G = 1;
    if (j0 + r < N && q < kb && stage_elem(m.fb, fld<ESZ>(Bt, (int64_t)(j0 + r) * ldb + k0 + q), S, E, G))
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

// A NaN pattern no model returns (their NaN results are always nan_bits): it marks
// an output the fast kernel left to the general evaluator.
__host__ __device__ __forceinline__ uint32_t redo_mark(const DevModel &m) {
  return m.nan_bits == 0x7FFFFFFFu ? 0xFFFFFFFFu : 0x7FFFFFFFu;
}

// Both kernels below: C == nullptr stands for C = 0.
//
// SPARSE = 1: A is given 2:4-compressed (Ac [M][K/2], meta [M][K/4]); kt and K are
// dense sizes.  The chain runs over the compressed terms (kt / 2 per instruction,
// blocks of N_FMA terms), and each term reads the B row its metadata index names
// (stage_chunk_gather).  Rows with invalid metadata (idx0 >= idx1) and rows or
// columns with an Inf/NaN go to the general evaluator of the compressed chain.
//
// Early-c global alignment (Table 3's early-c model) with the accumulator carried
// between blocks as f * 2^g: f is the block result's rounded significand as an
// integer-valued float (|f| < 2^31, or the addend's 24-bit significand before the
// first block) and g its scale.  Per block:
//  - e_c = max(floor(log2 |f|) + g, -126), read from f's exponent field (the -126
//    floor gives a subnormal addend the exponent e_min, as the decoder does);
//  - the aligned addend trunc(c * 2^(F_p - e_max)) = trunc(f * 2^(g + F_p - e_max)) is
//    one exact multiply by a power of two and one conversion with truncation toward
//    zero (RZ on the magnitude, the model's truncation); a scale below 2^-126 stands
//    for 0, which is the truncated value there since |f| < 2^31;
//  - the rounding of the sum S to 24 bits is the int->fp32 conversion (RNE or RZ,
//    RM), and the new scale is e_max - F_p.
// This equals rounding S * 2^(e_max - F_p) to fp32 while the result is normal.  A
// nonzero result lies in [2^(e_max - F_p), 2^(e_max + log2(4 kblk + 2))): each thread
// tracks the range of its e_max values, and one that could reach a subnormal or an
// overflowing result sends the thread's outputs to the fixup pass, as do Inf/NaN
// operands, a zero sum of zero terms (e_max = -inf) and a possible CDNA 3 product
// overflow.
template <int ESZ, int SPARSE, int RM>
__global__ void __launch_bounds__(kFThreads, 2) gemm_early_kernel(const __grid_constant__ DevModel m, int kt, int kblk,
                                                                int M, int N, int K, const uint8_t *__restrict__ A,
                                                                int64_t lda, const uint8_t *__restrict__ meta,
                                                                int64_t ldm, const uint8_t *__restrict__ Bt,
                                                                int64_t ldb, const uint32_t *C, int64_t ldc,
                                                                uint32_t *D, int64_t ldd) {
  extern __shared__ int32_t fsm[];
  constexpr bool GATHER = SPARSE != 0;
  const int KC = fast_chunk(kt);                                         // dense positions per chunk
  const int KCA = GATHER ? KC / 2 : KC;                                  // A panel rows
  int32_t *aS = fsm, *aE = aS + KCA * kFS, *aG = aE + KCA * kFS;        // [KCA][kFS]
  int32_t *aI = aG + KCA * kFS;                                          // gather: B row offsets
  int32_t *bS = aI + (GATHER ? KCA * kFS : 0), *bE = bS + KC * kFS, *bG = bE + KC * kFS;  // B significands << P0
  uint8_t *aSpec = reinterpret_cast<uint8_t *>(bG + KC * kFS);          // [kFB] per row
  uint8_t *bSpec = aSpec + kFB;
  const int i0 = blockIdx.y * kFB, j0 = blockIdx.x * kFB;
  const int tid = threadIdx.x;
  const int ti = (tid / (kFB / kFT)) * kFT, tj = (tid % (kFB / kFT)) * kFT;
  const int32_t F = m.F;
  // a zero sum is +0 when some term is nonzero.  Without a c = 0 exponent or an
  // exponent limit, all terms are zero exactly when e_max = -inf, which the range
  // check below already sends to the fixup pass; otherwise a zero sum goes there.
  const bool zero_check = m.c_zero_exp > -1024 || m.emin_lim > -1024;
  const int32_t hi_lim = 127 - (32 - __clz(4 * kblk + 1));   // 127 - ceil(log2(4 kblk + 2))

  float fv[kFT][kFT];                    // accumulator significand (integer-valued)
  int32_t gq[kFT][kFT];                  // its scale g, minus 127
  uint32_t redo = 0;                     // outputs to recompute with the general evaluator
  int32_t lo = 0, hi = -1024;            // range of this thread's e_max values
#pragma unroll
  for (int a = 0; a < kFT; a++)
#pragma unroll
    for (int b = 0; b < kFT; b++) {
      const int i = i0 + ti + a, j = j0 + tj + b;
      const uint32_t cb = (C && i < M && j < N) ? C[(int64_t)i * ldc + j] : 0u;
      uint32_t cS, cneg;
      int32_t cE;
      decode_c(m, cb, cS, cE, cneg);
      if ((cb & 0x7F800000u) == 0x7F800000u) {
        redo |= 1u << (a * kFT + b);
        cS = 0u;
      }
      fv[a][b] = cneg ? -(float)cS : (float)cS;
      gq[a][b] = cE - 23 - 127;
    }

  for (int k0 = 0; k0 < K; k0 += KC) {
    const int kc = min(KC, K - k0);
    __syncthreads();
    if (tid < kFB) { aSpec[tid] = 0; bSpec[tid] = 0; }
    __syncthreads();
    if constexpr (GATHER)
      stage_chunk_gather<ESZ>(m, m.P0, i0, j0, k0 / 2, kc / 2, KCA, M, N, A, lda, meta, ldm, Bt, ldb, aS, aE, aG, aI,
                              bS, bE, bG, aSpec, bSpec);
    else
      stage_chunk<ESZ>(m, m.P0, i0, j0, k0, kc, KC, M, N, A, lda, Bt, ldb, aS, aE, aG, bS, bE, bG, aSpec, bSpec);
    __syncthreads();
    // an Inf/NaN in a row of A or a column of B (or invalid metadata) sends the whole
    // row / column of this thread's tile to the fixup pass
#pragma unroll
    for (int a = 0; a < kFT; a++)
      if (aSpec[ti + a]) redo |= 0xFu << (a * kFT);
#pragma unroll
    for (int b = 0; b < kFT; b++)
      if (bSpec[tj + b]) redo |= 0x1111u << b;

    // the chain's units in this chunk: dense positions, or compressed terms (gather)
    const int ku = GATHER ? kc / 2 : kc, ktu = GATHER ? kt / 2 : kt;
    for (int s0 = 0; s0 < ku; s0 += ktu) {
      const int send = min(s0 + ktu, ku);
      for (int b0 = s0; b0 < send; b0 += kblk) {
        const int nt = min(kblk, send - b0);
        // ---- e_max: c's exponent and the limit first, then the products
        int32_t em[kFT][kFT];
#pragma unroll
        for (int a = 0; a < kFT; a++)
#pragma unroll
          for (int b = 0; b < kFT; b++) {
            // e_c = floor(log2 |c|) from f's exponent field, no lower than -126 (a
            // subnormal addend)
            const int32_t ec = fv[a][b] == 0.0f ? m.c_zero_exp
                               : max((int32_t)((__float_as_uint(fv[a][b]) >> 23) & 0xFFu) + gq[a][b], -126);
            em[a][b] = max(ec, m.emin_lim);
          }
        for (int q = b0; q < b0 + nt; q++) {
          const int4 ea = *reinterpret_cast<const int4 *>(aE + q * kFS + ti);
          const int32_t xa[4] = {ea.x, ea.y, ea.z, ea.w};
          if constexpr (GATHER) {
            const int4 ia = *reinterpret_cast<const int4 *>(aI + q * kFS + ti);
            const int32_t ra[4] = {ia.x, ia.y, ia.z, ia.w};
#pragma unroll
            for (int a = 0; a < kFT; a++) {
              const int4 eb = *reinterpret_cast<const int4 *>(bE + ra[a] + tj);
              const int32_t xb[4] = {eb.x, eb.y, eb.z, eb.w};
#pragma unroll
              for (int b = 0; b < kFT; b++) em[a][b] = __viaddmax_s32(xa[a], xb[b], em[a][b]);
            }
          } else {
            const int4 eb = *reinterpret_cast<const int4 *>(bE + q * kFS + tj);
            const int32_t xb[4] = {eb.x, eb.y, eb.z, eb.w};
#pragma unroll
            for (int a = 0; a < kFT; a++)
#pragma unroll
              for (int b = 0; b < kFT; b++) em[a][b] = __viaddmax_s32(xa[a], xb[b], em[a][b]);
          }
        }
        // ---- the aligned addend starts the sum
        int32_t Sp[kFT][kFT];
#pragma unroll
        for (int a = 0; a < kFT; a++)
#pragma unroll
          for (int b = 0; b < kFT; b++) {
            lo = min(lo, em[a][b]);
            hi = max(hi, em[a][b]);
            // 2^(g + F - e_max) as a float: exponent field g + F - e_max + 127, 0 below 2^-126
            const int32_t se = max(gq[a][b] + 254 + F - em[a][b], 0);
            const float sc = __fmul_rz(fv[a][b], __uint_as_float((uint32_t)se << 23));
            Sp[a][b] = fv[a][b] == 0.0f ? 0 : __float2int_rz(sc);
            em[a][b] += m.R0;                              // from here on: the shift base
          }
        // ---- aligned, truncated products
        for (int q = b0; q < b0 + nt; q++) {
          const int4 sa = *reinterpret_cast<const int4 *>(aS + q * kFS + ti);
          const int4 ea = *reinterpret_cast<const int4 *>(aE + q * kFS + ti);
          const int4 ga = *reinterpret_cast<const int4 *>(aG + q * kFS + ti);
          const int32_t SA[4] = {sa.x, sa.y, sa.z, sa.w}, EA[4] = {ea.x, ea.y, ea.z, ea.w}, GA[4] = {ga.x, ga.y, ga.z, ga.w};
          if constexpr (GATHER) {
            // each of the thread's A rows reads B at its own row of the panel
            const int4 ia = *reinterpret_cast<const int4 *>(aI + q * kFS + ti);
            const int32_t ra[4] = {ia.x, ia.y, ia.z, ia.w};
#pragma unroll
            for (int a = 0; a < kFT; a++) {
              const int4 sb = *reinterpret_cast<const int4 *>(bS + ra[a] + tj);
              const int4 eb = *reinterpret_cast<const int4 *>(bE + ra[a] + tj);
              const int4 gb = *reinterpret_cast<const int4 *>(bG + ra[a] + tj);
              const int32_t SB[4] = {sb.x, sb.y, sb.z, sb.w}, EB[4] = {eb.x, eb.y, eb.z, eb.w};
              const int32_t GB[4] = {gb.x, gb.y, gb.z, gb.w};
#pragma unroll
              for (int b = 0; b < kFT; b++) {
                const int32_t sh = em[a][b] - EA[a] - EB[b];
                const uint32_t U = (uint32_t)(SA[a] * SB[b]);
                const int32_t t = (int32_t)shr32(U, sh);
                Sp[a][b] += t * (GA[a] * GB[b]);
              }
            }
          } else {
            const int4 sb = *reinterpret_cast<const int4 *>(bS + q * kFS + tj);
            const int4 eb = *reinterpret_cast<const int4 *>(bE + q * kFS + tj);
            const int4 gb = *reinterpret_cast<const int4 *>(bG + q * kFS + tj);
            const int32_t SB[4] = {sb.x, sb.y, sb.z, sb.w}, EB[4] = {eb.x, eb.y, eb.z, eb.w}, GB[4] = {gb.x, gb.y, gb.z, gb.w};
#pragma unroll
            for (int a = 0; a < kFT; a++)
#pragma unroll
              for (int b = 0; b < kFT; b++) {
                const int32_t sh = em[a][b] - EA[a] - EB[b];
                const uint32_t U = (uint32_t)(SA[a] * SB[b]);
                const int32_t t = (int32_t)shr32(U, sh);
                Sp[a][b] += t * (GA[a] * GB[b]);
              }
          }
        }
        // ---- round: the new accumulator (the scale is e_max - F)
        const int32_t gk = m.R0 + F + 127;
#pragma unroll
        for (int a = 0; a < kFT; a++)
#pragma unroll
          for (int b = 0; b < kFT; b++) {
            fv[a][b] = RM ? __int2float_rn(Sp[a][b]) : __int2float_rz(Sp[a][b]);
            gq[a][b] = em[a][b] - gk;
          }
        if (zero_check) {
#pragma unroll
          for (int a = 0; a < kFT; a++)
#pragma unroll
            for (int b = 0; b < kFT; b++)
              if (Sp[a][b] == 0) redo |= 1u << (a * kFT + b);
        }
        if (m.prod_ovf) {
#pragma unroll
          for (int a = 0; a < kFT; a++)
#pragma unroll
            for (int b = 0; b < kFT; b++)
              if (em[a][b] - m.R0 >= 126) redo |= 1u << (a * kFT + b);
        }
      }
    }
  }
  // an e_max that allows a result outside the normal range anywhere in this thread's
  // chains: all its outputs take the fixup pass (gemm_fixup_kernel; C does not alias D)
  if (lo - F < -126 || hi > hi_lim) redo = 0xFFFFu;
#pragma unroll
  for (int a = 0; a < kFT; a++)
#pragma unroll
    for (int b = 0; b < kFT; b++) {
      const int i = i0 + ti + a, j = j0 + tj + b;
      if (i >= M || j >= N) continue;
      uint32_t r;
      if (K == 0) {
        r = C ? C[(int64_t)i * ldc + j] : 0u;
      } else if ((redo >> (a * kFT + b)) & 1u) {
        r = redo_mark(m);
      } else {
        // f * 2^g is a normal float (or f = 0): the two scalings are exact
        const int32_t g = gq[a][b] + 127;
        const int32_t k1 = min(max(g, -96), 96), k2 = g - k1;
        const float y = __fmul_rn(__fmul_rn(fv[a][b], __uint_as_float((uint32_t)(k1 + 127) << 23)),
                                  __uint_as_float((uint32_t)(k2 + 127) << 23));
        r = fv[a][b] == 0.0f ? 0u : __float_as_uint(y);
      }
      D[(int64_t)i * ldd + j] = r;
    }
}

// Algorithm 1 (late c) with the accumulator carried as f * 2^g (as in
// gemm_early_kernel) and both branches of the merge (lines 6-14) in one branch-free
// sequence.  With d = e_c - e_max and s = max(d - (psum_frac - F_p), 0), the sum is
// formed in units of 2^(e_max - F_p + s): the units of the product sum S_p while c's
// grid of psum_frac fraction bits (line 10) is no coarser than S_p's, else c's grid.
//  - X = floor(c * 2^-(e_max - F_p + s)) is c aligned to c_frac = F_p fraction bits and
//    rounded down (line 7) when d <= 0, and c exactly when d > 0 (line 11: c's grid
//    2^(e_c - 23) is then no finer than the units); |X| < 2^(psum_frac + 1).  One exact
//    multiply by a power of two and one conversion rounding down;
//  - floor(S_p / 2^s) is line 10's round-down of S_p onto c's grid (s = 0: exact);
//  - T = floor(S_p / 2^s) + X is then the sum of line 8 (d <= 0) or that of line 11
//    (d > 0) up to a power of two; for d > 0 lines 12-13 floor T to post_norm_frac + 1
//    significant bits, which in two's complement clears the low bits;
//  - line 15 is the int64 -> fp32 conversion, and g becomes e_max - F_p + s.
// The normalisation's exponent floor at -126 and the fp32 range are handled as in
// gemm_early_kernel: a nonzero result lies in [2^(e_max - F_p),
// 2^(max(e_max, e_c) + log2(4 kblk + 2))), and a thread whose exponents allow a result
// outside the normal range sends its outputs to the fixup pass.  So does a block
// without products (e_max = -inf).
// TJ consecutive words of a panel row (TJ = 4: one 16-byte load; 2: one 8-byte load)
template <int TJ>
__device__ __forceinline__ void ld_cols(const int32_t *p, int32_t (&x)[TJ]) {
  if constexpr (TJ == 4) {
    const int4 v = *reinterpret_cast<const int4 *>(p);
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  } else {
    static_assert(TJ == 2, "2 or 4 columns per thread");
    const int2 v = *reinterpret_cast<const int2 *>(p);
    x[0] = v.x; x[1] = v.y;
  }
}

template <int ESZ, int SPARSE, int RM, int TJ = kFT>
__global__ void __launch_bounds__((kFB / kFT) * (kFB / TJ), 2) gemm_late_kernel(const __grid_constant__ DevModel m, int kt, int kblk,
                                                               int M, int N, int K, const uint8_t *__restrict__ A,
                                                               int64_t lda, const uint8_t *__restrict__ meta,
                                                               int64_t ldm, const uint8_t *__restrict__ Bt,
                                                               int64_t ldb, const uint32_t *C, int64_t ldc,
                                                               uint32_t *D, int64_t ldd) {
  extern __shared__ int32_t fsm[];
  constexpr bool GATHER = SPARSE != 0;
  const int KC = fast_chunk(kt);                                         // dense positions per chunk
  const int KCA = GATHER ? KC / 2 : KC;                                  // A panel rows
  int32_t *aS = fsm, *aE = aS + KCA * kFS, *aG = aE + KCA * kFS;        // [KCA][kFS]
  int32_t *aI = aG + KCA * kFS;                                          // gather: B row offsets
  int32_t *bS = aI + (GATHER ? KCA * kFS : 0), *bE = bS + KC * kFS, *bG = bE + KC * kFS;  // B significands << P0
  uint8_t *aSpec = reinterpret_cast<uint8_t *>(bG + KC * kFS);          // [kFB] per row
  uint8_t *bSpec = aSpec + kFB;
  const int i0 = blockIdx.y * kFB, j0 = blockIdx.x * kFB;
  const int tid = threadIdx.x;
  const int ti = (tid / (kFB / TJ)) * kFT, tj = (tid % (kFB / TJ)) * TJ;
  const int32_t F = m.F;
  const int32_t dpsum = m.psum_frac - F;              // line 10 floors S_p only beyond this gap
  const int32_t hi_lim = 127 - (32 - __clz(4 * kblk + 1));   // 127 - ceil(log2(4 kblk + 2))

  float fv[kFT][TJ];                    // accumulator significand (integer-valued)
  int32_t gs[kFT][TJ];                  // its scale g
  uint32_t redo = 0;
  int32_t lo = 0, hi = -1024;            // range of this thread's e_max and e_c values
#pragma unroll
  for (int a = 0; a < kFT; a++)
#pragma unroll
    for (int b = 0; b < TJ; b++) {
      const int i = i0 + ti + a, j = j0 + tj + b;
      const uint32_t cb = (C && i < M && j < N) ? C[(int64_t)i * ldc + j] : 0u;
      uint32_t cS, cneg;
      int32_t cE;
      decode_c(m, cb, cS, cE, cneg);
      if ((cb & 0x7F800000u) == 0x7F800000u) {
        redo |= 1u << (a * TJ + b);
        cS = 0u;
      }
      fv[a][b] = cneg ? -(float)cS : (float)cS;
      gs[a][b] = cE - 23;
    }

  for (int k0 = 0; k0 < K; k0 += KC) {
    const int kc = min(KC, K - k0);
    __syncthreads();
    if (tid < kFB) { aSpec[tid] = 0; bSpec[tid] = 0; }
    __syncthreads();
    if constexpr (GATHER)
      stage_chunk_gather<ESZ>(m, m.P0, i0, j0, k0 / 2, kc / 2, KCA, M, N, A, lda, meta, ldm, Bt, ldb, aS, aE, aG, aI,
                              bS, bE, bG, aSpec, bSpec);
    else
      stage_chunk<ESZ>(m, m.P0, i0, j0, k0, kc, KC, M, N, A, lda, Bt, ldb, aS, aE, aG, bS, bE, bG, aSpec, bSpec);
    __syncthreads();
#pragma unroll
    for (int a = 0; a < kFT; a++)
      if (aSpec[ti + a]) redo |= ((1u << TJ) - 1u) << (a * TJ);
#pragma unroll
    for (int b = 0; b < TJ; b++)
      if (bSpec[tj + b]) redo |= (TJ == 4 ? 0x1111u : 0x55u) << b;

    // the chain's units in this chunk: dense positions, or compressed terms (gather)
    const int ku = GATHER ? kc / 2 : kc, ktu = GATHER ? kt / 2 : kt;
    for (int s0 = 0; s0 < ku; s0 += ktu) {
      const int send = min(s0 + ktu, ku);
      for (int b0 = s0; b0 < send; b0 += kblk) {
        const int nt = min(kblk, send - b0);
        // ---- e_max of the products (line 3)
        int32_t em[kFT][TJ];
#pragma unroll
        for (int a = 0; a < kFT; a++)
#pragma unroll
          for (int b = 0; b < TJ; b++) em[a][b] = kNegE;
        for (int q = b0; q < b0 + nt; q++) {
          const int4 ea = *reinterpret_cast<const int4 *>(aE + q * kFS + ti);
          const int32_t xa[4] = {ea.x, ea.y, ea.z, ea.w};
          if constexpr (GATHER) {
            const int4 ia = *reinterpret_cast<const int4 *>(aI + q * kFS + ti);
            const int32_t ra[4] = {ia.x, ia.y, ia.z, ia.w};
#pragma unroll
            for (int a = 0; a < kFT; a++) {
              int32_t xb[TJ];
              ld_cols<TJ>(bE + ra[a] + tj, xb);
#pragma unroll
              for (int b = 0; b < TJ; b++) em[a][b] = __viaddmax_s32(xa[a], xb[b], em[a][b]);
            }
          } else {
            int32_t xb[TJ];
            ld_cols<TJ>(bE + q * kFS + tj, xb);
#pragma unroll
            for (int a = 0; a < kFT; a++)
#pragma unroll
              for (int b = 0; b < TJ; b++) em[a][b] = __viaddmax_s32(xa[a], xb[b], em[a][b]);
          }
        }
        // ---- aligned, truncated products (line 4)
        int32_t Sp[kFT][TJ];
#pragma unroll
        for (int a = 0; a < kFT; a++)
#pragma unroll
          for (int b = 0; b < TJ; b++) {
            Sp[a][b] = 0;
            em[a][b] += m.R0;                              // the shift base until the merge
          }
        for (int q = b0; q < b0 + nt; q++) {
          const int4 sa = *reinterpret_cast<const int4 *>(aS + q * kFS + ti);
          const int4 ea = *reinterpret_cast<const int4 *>(aE + q * kFS + ti);
          const int4 ga = *reinterpret_cast<const int4 *>(aG + q * kFS + ti);
          const int32_t SA[4] = {sa.x, sa.y, sa.z, sa.w}, EA[4] = {ea.x, ea.y, ea.z, ea.w}, GA[4] = {ga.x, ga.y, ga.z, ga.w};
          if constexpr (GATHER) {
            // each of the thread's A rows reads B at its own row of the panel
            const int4 ia = *reinterpret_cast<const int4 *>(aI + q * kFS + ti);
            const int32_t ra[4] = {ia.x, ia.y, ia.z, ia.w};
#pragma unroll
            for (int a = 0; a < kFT; a++) {
              int32_t SB[TJ], EB[TJ], GB[TJ];
              ld_cols<TJ>(bS + ra[a] + tj, SB);
              ld_cols<TJ>(bE + ra[a] + tj, EB);
              ld_cols<TJ>(bG + ra[a] + tj, GB);
#pragma unroll
              for (int b = 0; b < TJ; b++) {
                const int32_t sh = em[a][b] - EA[a] - EB[b];
                const uint32_t U = (uint32_t)(SA[a] * SB[b]);
                const int32_t t = (int32_t)shr32(U, sh);
                Sp[a][b] += t * (GA[a] * GB[b]);
              }
            }
          } else {
            int32_t SB[TJ], EB[TJ], GB[TJ];
            ld_cols<TJ>(bS + q * kFS + tj, SB);
            ld_cols<TJ>(bE + q * kFS + tj, EB);
            ld_cols<TJ>(bG + q * kFS + tj, GB);
#pragma unroll
            for (int a = 0; a < kFT; a++)
#pragma unroll
              for (int b = 0; b < TJ; b++) {
                const int32_t sh = em[a][b] - EA[a] - EB[b];
                const uint32_t U = (uint32_t)(SA[a] * SB[b]);
                const int32_t t = (int32_t)shr32(U, sh);
                Sp[a][b] += t * (GA[a] * GB[b]);
              }
          }
        }
        // ---- the merge with c (lines 5-15)
#pragma unroll
        for (int a = 0; a < kFT; a++)
#pragma unroll
          for (int b = 0; b < TJ; b++) {
            const int32_t e = em[a][b] - m.R0;
            // e_c = floor(log2 |c|), no lower than -126 (a subnormal addend), from f's
            // exponent field; c_zero_exp for c = 0
            const int32_t ecv = fv[a][b] == 0.0f ? m.c_zero_exp
                                : max((int32_t)((__float_as_uint(fv[a][b]) >> 23) & 0xFFu) + gs[a][b] - 127, -126);
            const int32_t d = ecv - e;
            lo = min(lo, e);
            hi = max(hi, max(e, ecv));
            const int32_t sg = max(d - dpsum, 0);
            const int32_t u = e - F + sg;                  // the units' exponent
            // X: 2^(g - u) as a float, no lower than 2^-126 (|f| * 2^-126 < 1 floors
            // like any smaller positive or negative value)
            const int32_t se = max(gs[a][b] + 127 - u, 1);
            const int64_t X = fv[a][b] == 0.0f ? 0ll
                              : __float2ll_rd(__fmul_rn(fv[a][b], __uint_as_float((uint32_t)se << 23)));
            int64_t T = (int64_t)(Sp[a][b] >> min(sg, 31)) + X;
            // the leading bit of |T| (one place low when |T| is a power of two, where
            // every lower bit is zero and the round-down is exact anyway)
            const int32_t p = 63 - __clzll((long long)(T ^ (T >> 63)));
            const int32_t rsh = d > 0 ? max(p - m.post_norm_frac, 0) : 0;
            T = (T >> rsh) << rsh;
            fv[a][b] = RM ? __ll2float_rn(T) : __ll2float_rz(T);
            gs[a][b] = u;
          }
        if (m.prod_ovf) {
#pragma unroll
          for (int a = 0; a < kFT; a++)
#pragma unroll
            for (int b = 0; b < TJ; b++)
              if (em[a][b] - m.R0 >= 126) redo |= 1u << (a * TJ + b);
        }
      }
    }
  }
  if (lo - F < -126 || hi > hi_lim) redo = (1u << (kFT * TJ)) - 1u;
#pragma unroll
  for (int a = 0; a < kFT; a++)
#pragma unroll
    for (int b = 0; b < TJ; b++) {
      const int i = i0 + ti + a, j = j0 + tj + b;
      if (i >= M || j >= N) continue;
      uint32_t r;
      if (K == 0) {
        r = C ? C[(int64_t)i * ldc + j] : 0u;
      } else if ((redo >> (a * TJ + b)) & 1u) {
        r = redo_mark(m);
      } else {
        const int32_t g = gs[a][b];
        const int32_t k1 = min(max(g, -96), 96), k2 = g - k1;
        const float y = __fmul_rn(__fmul_rn(fv[a][b], __uint_as_float((uint32_t)(k1 + 127) << 23)),
                                  __uint_as_float((uint32_t)(k2 + 127) << 23));
        r = fv[a][b] == 0.0f ? 0u : __float_as_uint(y);
      }
      D[(int64_t)i * ldd + j] = r;
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
  const int KC = fast_chunk(kt);
  const size_t shm = (size_t)(SPARSE ? 5 * KC : 6 * KC) * kFS * 4 + 2 * kFB;   // gather: 4 (KC / 2) + 3 KC rows
  // the late-c kernel runs 4 x 2 thread tiles in 512-thread CTAs: twice the warps per SM
  // to hide the latency of its per-block merge
  constexpr int TJL = 2;
  auto kern = ARCH == MCEMU_ARCH_GA_EARLY ? (m.rne ? gemm_early_kernel<ESZ, SPARSE, 1> : gemm_early_kernel<ESZ, SPARSE, 0>)
                                          : (m.rne ? gemm_late_kernel<ESZ, SPARSE, 1, TJL> : gemm_late_kernel<ESZ, SPARSE, 0, TJL>);
  const int threads = ARCH == MCEMU_ARCH_GA_EARLY ? kFThreads : (kFB / kFT) * (kFB / TJL);
  if (shm > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)shm) != cudaSuccess)
    return MCEMU_ERR_UNSUPPORTED;
  dim3 grid((N + kFB - 1) / kFB, (M + kFB - 1) / kFB);
  const int kblk = m.k;                             // a block of N_FMA (compressed) terms
  kern<<<grid, threads, shm, s>>>(m, kt, kblk, M, N, K, (const uint8_t *)A, lda, meta, ldm, (const uint8_t *)Bt,
                                    ldb, C, ldc, D, ldd);
  if (cudaGetLastError() != cudaSuccess) return MCEMU_ERR_CUDA;
  return run_fixup<ESZ, SPARSE>(m, kt, M, N, K, A, lda, meta, ldm, Bt, ldb, C, ldc, D, ldd, s);
}

}  // namespace mcemu

// stream_fp8.cu -- block-FMA stream for FP8 operands (E4M3, E5M2; OCP and FNUZ)
// through a product table: early-c global alignment and exact-then-round.
//
// One table read per product replaces two element decodes and a multiplication:
// the table, indexed by the magnitudes of an operand pair, holds the integer
// product S_a * S_b, the denormalised product exponent E_a + E_b ("Accurate Models
// of AMD Matrix Cores", Sec. 4.3.1) and the special-value class of the pair.  The
// table follows from the format definitions of Table 1 at compile time, lives in
// global memory, and every CTA copies it into shared memory once (64 KB).  The
// product sign is the xor of the operand sign bits, taken four products at a time.
#include <cuda_runtime.h>

#include "core.cuh"
#include "stream_pair.cuh"

namespace mcemu {

// ---------------------------------------------------------------------------
// the product table
// ---------------------------------------------------------------------------
// Entry (16 bits):
//   bits 0-7   P = S_a * S_b, 0 when a or b is zero
//   bit  8     the pair is special and its product is an infinity
//   bit  9     the pair is special and its product is NaN (a NaN operand, or Inf * 0)
//   bits 10-15 X = E_a + E_b - XMIN + 1 for a nonzero product, 0 for a zero
//              product, 63 for a special pair
// X sits on top, so the largest entry of a block carries e_max, and the special
// entries lie above every finite one with NaN highest: the block's largest entry
// alone says whether it holds a NaN product (kF8NaN), an infinite one and no NaN
// (kF8Inf), or neither.  Index: (a & 0x7F) | (b & 0x7F) << 8; bit 7 of the index is
// unused.
constexpr int kF8Entries = 32768;
constexpr uint32_t kF8Special = 63u;
constexpr uint32_t kF8Inf = (kF8Special << 10) | 0x100u, kF8NaN = (kF8Special << 10) | 0x200u;
constexpr int kF8Threads = 512;

template <int ID>
struct F8 {
  static constexpr int XMIN = 2 * (1 - Fmt<ID>::BIAS);    // smallest E_a + E_b
  static constexpr int MAB = 2 * Fmt<ID>::MEFF;           // fraction bits of S_a * S_b
};

struct F8Table {
  uint16_t v[kF8Entries];
};

// class of a 7-bit magnitude: 0 finite, 1 Inf, 2 NaN (FNUZ marks NaN with the sign
// bit, which the magnitude does not hold; that case is tested on the raw words)
template <int ID>
constexpr uint32_t f8_class(uint32_t x) {
  using F = Fmt<ID>;
  if (F::FNUZ) return 0u;
  if (F::E4OCP) return x == 0x7Fu ? 2u : 0u;
  if (((x >> F::MB) & F::EMASK) != F::EMASK) return 0u;
  return (x & F::MMASK) ? 2u : 1u;
}

template <int ID>
constexpr uint16_t f8_entry(uint32_t a, uint32_t b) {
  using F = Fmt<ID>;
  const uint32_t ea = (a >> F::MB) & F::EMASK, eb = (b >> F::MB) & F::EMASK;
  const uint32_t sa = ea ? ((a & F::MMASK) | (1u << F::MB)) : (a & F::MMASK);
  const uint32_t sb = eb ? ((b & F::MMASK) | (1u << F::MB)) : (b & F::MMASK);
  const uint32_t ca = f8_class<ID>(a), cb = f8_class<ID>(b);
  if (ca || cb) {
    const bool nan = ca == 2u || cb == 2u || (ca == 1u && sb == 0u) || (cb == 1u && sa == 0u);
    return (uint16_t)(nan ? kF8NaN : kF8Inf);
  }
  const int Ea = (int)(ea ? ea : 1u) - F::BIAS, Eb = (int)(eb ? eb : 1u) - F::BIAS;
  const uint32_t P = sa * sb;
  const uint32_t X = P ? (uint32_t)(Ea + Eb - F8<ID>::XMIN + 1) : 0u;
  return (uint16_t)(P | (X << 10));
}

template <int ID>
constexpr F8Table f8_make_table() {
  F8Table t{};
  for (uint32_t b = 0; b < 128u; b++)
    for (uint32_t a = 0; a < 128u; a++) t.v[a | (b << 8)] = f8_entry<ID>(a, b);
  return t;
}

__device__ constexpr F8Table kF8TabE4M3 = f8_make_table<F_E4M3>();
__device__ constexpr F8Table kF8TabE4M3Z = f8_make_table<F_E4M3Z>();
__device__ constexpr F8Table kF8TabE5M2 = f8_make_table<F_E5M2>();
__device__ constexpr F8Table kF8TabE5M2Z = f8_make_table<F_E5M2Z>();

template <int ID>
__device__ __forceinline__ const F8Table &f8_table() {
  if constexpr (ID == F_E4M3) return kF8TabE4M3;
  else if constexpr (ID == F_E4M3Z) return kF8TabE4M3Z;
  else if constexpr (ID == F_E5M2) return kF8TabE5M2;
  else return kF8TabE5M2Z;
}

// byte permute (PTX prmt, generic mode): a selector nibble 8 + j copies the sign
// bit of source byte j into all eight bits of the result byte
template <uint32_t SEL>
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "n"(SEL));
  return r;
}

// entries and sign masks (0 or all ones) of the K products of one vector set
template <int K>
__device__ __forceinline__ void f8_lookup(const uint16_t *tab, const uint32_t (&wa)[K / 4],
                                          const uint32_t (&wb)[K / 4], uint32_t (&e)[K], uint32_t (&sg)[K]) {
#pragma unroll
  for (int w = 0; w < K / 4; w++) {
    const uint32_t ma = wa[w] & 0x7F7F7F7Fu, mb = wb[w] & 0x7F7F7F7Fu, xs = wa[w] ^ wb[w];
    // index of product i: byte i of ma, byte i of mb, then two zero bytes (the
    // replicated sign bit of byte 0 of ma, which the mask cleared)
    e[4 * w + 0] = tab[prmt<0x8840u>(ma, mb)];
    e[4 * w + 1] = tab[prmt<0x8851u>(ma, mb)];
    e[4 * w + 2] = tab[prmt<0x8862u>(ma, mb)];
    e[4 * w + 3] = tab[prmt<0x8873u>(ma, mb)];
    sg[4 * w + 0] = prmt<0x8888u>(xs, xs);
    sg[4 * w + 1] = prmt<0x9999u>(xs, xs);
    sg[4 * w + 2] = prmt<0xAAAAu>(xs, xs);
    sg[4 * w + 3] = prmt<0xBBBBu>(xs, xs);
  }
}

// Result of a block with a special operand (1 NaN, 2 +Inf, 4 -Inf as in core.cuh).
// `mx` is the largest entry: kF8NaN when some product is NaN.
template <int ID, int K>
__device__ __forceinline__ uint32_t f8_special(const DevModel &m, const uint32_t (&e)[K], const uint32_t (&sg)[K],
                                               uint32_t mx, uint32_t cb, uint32_t fnuz_nan) {
  uint32_t s = c_special(cb) | (fnuz_nan || mx == kF8NaN ? 1u : 0u);
  if constexpr (Fmt<ID>::IEEE) {
    // E5M2 (OCP) has infinities: the entries' Inf bit (8) under the positive and the
    // negative sign masks, branch-free (E4M3 and the FNUZ encodings have none); a NaN
    // product makes the result NaN whatever these say
    uint32_t pinf = 0u, ninf = 0u;
#pragma unroll
    for (int l = 0; l < K; l++) {
      pinf |= e[l] & ~sg[l];
      ninf |= e[l] & sg[l];
    }
    s |= ((pinf & 0x100u) ? 2u : 0u) | ((ninf & 0x100u) ? 4u : 0u);
  }
  return resolve_special(m, s);
}

// fp32 bits of S * 2^k, S != 0 an integer, rounded (RNE or RZ) in hardware; false
// when k is out of the single-multiply range or the result is 2^-126 or below in
// magnitude (where the two roundings could differ from one, see hw_scale)
template <bool RNE>
__device__ __forceinline__ bool f8_round(int32_t S, int32_t k, uint32_t &bits) {
  if ((uint32_t)(k + 126) > 253u) return false;
  const float x = RNE ? __int2float_rn(S) : __int2float_rz(S);
  const float sc = __uint_as_float((uint32_t)(k + 127) << 23);
  bits = __float_as_uint(RNE ? __fmul_rn(x, sc) : __fmul_rz(x, sc));
  return hw_normal(bits);
}

// Early-c global alignment (Table 3): e_max over the products, c and e_min^lim;
// each term truncated to F_p fraction bits at e_max, summed exactly, rounded once.
struct PipeConsts {
  uint32_t m1, p24, p22;
};

template <int ID, int K, bool RNE>
__device__ __forceinline__ uint32_t f8_ga_early(const DevModel &m, const PipeConsts &pc, const uint32_t (&e)[K],
                                                const uint32_t (&sg)[K], uint32_t cb, uint32_t mx) {
  uint32_t cS, cneg;
  int32_t cE;
  decode_c(m, cb, cS, cE, cneg);
  int32_t emax = mx ? (int32_t)(mx >> 10) + F8<ID>::XMIN - 1 : kNegE;
  const int32_t ec = cS ? cE : m.c_zero_exp;
  emax = max(max(emax, ec), m.emin_lim);
  // term l = (P << P0) >> (e_max + R0 - e_l) = (entry << 24) >> (C0 - X_l), and
  // C0 - X_l = ((C0 << 10 | 0x3FF) - entry) >> 10 since the low ten bits hold P
  const uint32_t C0s = ((uint32_t)(24 - m.P0 + m.R0 + emax - F8<ID>::XMIN + 1) << 10) | 0x3FFu;
  int32_t S = 0;
  // pc.m1 = -1, pc.p24 = 2^24, pc.p22 = 2^22 are kernel arguments, so the shift-count
  // arithmetic, the pre-shift and the sign stay multiplies on the FMA pipe while the
  // ALU pipe does the byte permutes, the maximum and the one funnel shift per term
#pragma unroll
  for (int l = 0; l < K; l++) {
    const uint32_t sh = __umulhi(C0s + e[l] * pc.m1, pc.p22);             // (C0s - e) >> 10
    const uint32_t t = shr32(e[l] * pc.p24, (int32_t)sh);                  // P << 24 >> sh
    S += (int32_t)t * (int32_t)(sg[l] * 2u + 1u);                          // +-1
  }
  if (cS) S += align_term<uint32_t, int32_t>(cS << m.P0c, cneg, emax + m.R0c - cE, 0);
  if (S == 0) {
    // a negative zero needs every product to be a negative zero and c = -0
    uint32_t all = cS == 0u && cneg && mx == 0u ? 0xFFFFFFFFu : 0u;
#pragma unroll
    for (int l = 0; l < K; l++) all &= sg[l];
    return all ? 0x80000000u : 0u;
  }
  uint32_t bits;
  if (f8_round<RNE>(S, emax - m.F, bits)) return bits;
  return pack_sum<int32_t>(S, emax - m.F, m);
}

// Exact-then-round (CDNA 1): every product is +-P * 2^X on the grid 2^G with
// G = XMIN - MAB - 1.  E4M3 sums fit one 64-bit accumulator; E5M2 products span
// 2^0 .. 2^66 on that grid and are split at 2^31 into two.  The addend and the single
// rounding follow arch_exact_fixed, on the same 2^(G - 39) window.
__device__ __forceinline__ int64_t mad_wide(int32_t a, int32_t b, int64_t c) {
  int64_t r;
  asm("mad.wide.s32 %0, %1, %2, %3;" : "=l"(r) : "r"(a), "r"(b), "l"(c));
  return r;
}

template <int ID, int K>
__device__ __forceinline__ uint32_t f8_exact(const DevModel &m, const uint32_t (&e)[K], const uint32_t (&sg)[K],
                                             uint32_t cb, uint32_t mx) {
  // the exact sum W = lo + hi * 2^31 (hi = 0 for E4M3), |lo|, |hi| < 2^42
  int64_t lo = 0, hi = 0;
  if constexpr (Fmt<ID>::EB == 4) {
#pragma unroll
    for (int l = 0; l < K; l++) {
      const int32_t sP = (int32_t)(((e[l] & 0xFFu) ^ sg[l]) - sg[l]);
      lo = mad_wide(sP, (int32_t)shl_clamp(1u, e[l] >> 10), lo);     // X <= 29
    }
  } else {
#pragma unroll
    for (int l = 0; l < K; l++) {
      const uint32_t X = e[l] >> 10;
      const int32_t sP = (int32_t)(((e[l] & 0xFFu) ^ sg[l]) - sg[l]);
      lo = mad_wide(sP, (int32_t)(shl_clamp(2u, X) >> 1), lo);      // 2^X for X <= 30, else 0
      hi = mad_wide(sP, (int32_t)shl_clamp(1u, X - 31u), hi);       // 2^(X-31) for X >= 31, else 0
    }
  }
  // W in a 64-bit window: Wt * 2^Gw plus an unknown amount below it when stW.  hi * 2^31
  // has no bits below 2^31, so W >> sh (sh <= 31) is hi * 2^(31 - sh) + (lo >> sh) exactly
  // and only lo's low sh bits drop out; sh keeps |Wt| < 2^61.
  constexpr int32_t G = F8<ID>::XMIN - F8<ID>::MAB - 1;
  int64_t Wt = lo;
  int32_t Gw = G, stW = 0, sh = 0;
  if constexpr (Fmt<ID>::EB != 4) {
    const uint64_t ah = hi < 0 ? 0ull - (uint64_t)hi : (uint64_t)hi;
    sh = max(0, 64 - __clzll((long long)ah) - 29);
    Wt = (int64_t)((uint64_t)hi << (31 - sh)) + (lo >> sh);
    stW = (sh > 0 && (lo & ((1ll << sh) - 1)) != 0) ? 1 : 0;
    Gw = G + sh;
  }
  uint32_t cS, cneg;
  int32_t cE;
  decode_c(m, cb, cS, cE, cneg);
  if (Wt == 0 && sh == 0) {                              // the products cancel exactly
    if (cS) return cb;                                  // c alone: already an fp32 value
    uint32_t all = cneg && mx == 0u ? 0xFFFFFFFFu : 0u;
#pragma unroll
    for (int l = 0; l < K; l++) all &= sg[l];
    return all ? 0x80000000u : 0u;
  }
  uint32_t r;
  if (merge_c64(m, Wt, Gw, stW, cS, cE, cneg, r)) return r;
  const i128 W = (i128)lo + ((i128)hi << 31);
  return exact_fixed_merge<ID>(m, W << 39, cS, cE, cneg, cb);
}

// One vector set through the product table: specials, then the model.
template <int ARCH, int ID, int K, bool RNE>
__device__ __forceinline__ uint32_t f8_eval(const DevModel &m, const PipeConsts &pc, const uint16_t *tab,
                                            const uint32_t (&wa)[K / 4], const uint32_t (&wb)[K / 4], uint32_t cb) {
  constexpr int NW = K / 4;
  uint32_t e[K], sg[K];
  f8_lookup<K>(tab, wa, wb, e, sg);
  uint32_t mx = 0;
#pragma unroll
  for (int l = 0; l < K; l++) mx = max(mx, e[l]);
  uint32_t fnuz_nan = 0;
  if constexpr (Fmt<ID>::FNUZ) {
#pragma unroll
    for (int w = 0; w < NW; w++) fnuz_nan |= fspecial_word<ID>(wa[w]) | fspecial_word<ID>(wb[w]);
  }
  if (mx >= kF8Inf || (cb & 0x7F800000u) == 0x7F800000u || fnuz_nan)
    return f8_special<ID, K>(m, e, sg, mx, cb, fnuz_nan);
  if constexpr (ARCH == MCEMU_ARCH_GA_EARLY) return f8_ga_early<ID, K, RNE>(m, pc, e, sg, cb, mx);
  else return f8_exact<ID, K>(m, e, sg, cb, mx);
}

template <int K>
__device__ __forceinline__ void f8_load(const uint8_t *__restrict__ a, const uint8_t *__restrict__ b,
                                        const uint32_t *__restrict__ c, size_t u, uint32_t (&wa)[K / 4],
                                        uint32_t (&wb)[K / 4], uint32_t &cb) {
#pragma unroll
  for (int w = 0; w < K / 4; w += 2) {
    const uint2 x = __ldcs(reinterpret_cast<const uint2 *>(a + u * K) + w / 2);
    const uint2 y = __ldcs(reinterpret_cast<const uint2 *>(b + u * K) + w / 2);
    wa[w] = x.x; wa[w + 1] = x.y;
    wb[w] = y.x; wb[w + 1] = y.y;
  }
  cb = __ldcs(c + u);
}

// Exact-then-round of one OCP FP8 set on the FP32 pipe (exact_fp32_sum): FP8 -> f16
// -> f32 is exact, and so are the products.  False when the rounding is not decided
// there.
template <int ID, int K>
__device__ __forceinline__ bool f8_exact_fp32(const DevModel &m, const uint32_t (&wa)[K / 4],
                                              const uint32_t (&wb)[K / 4], uint32_t cb, uint32_t &r) {
  float p[K];
  constexpr __nv_fp8_interpretation_t kind = ID == F_E4M3 ? __NV_E4M3 : __NV_E5M2;
#pragma unroll
  for (int w = 0; w < K / 4; w++)
#pragma unroll
    for (int h = 0; h < 2; h++) {
      const float2 fa = __half22float2(__half2(
          __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(wa[w] >> (16 * h)), kind)));
      const float2 fb = __half22float2(__half2(
          __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(wb[w] >> (16 * h)), kind)));
      p[4 * w + 2 * h] = __fmul_rn(fa.x, fb.x);
      p[4 * w + 2 * h + 1] = __fmul_rn(fa.y, fb.y);
    }
  return exact_fp32_sum<K>(p, cb, m.rne, m.nan_bits, r) == 0;
}

// FP8 K=8 sets (8 bytes per operand set) through the paired kernel of stream_pair.cuh:
// early-c global alignment through the product table with special values in line, and
// OCP exact-then-round on the FP32 pipe with the undecided sets (ties that the error
// bound leaves open) batched per warp for the integer path.
template <int ID, int RM> struct F8GaPairEv {
  static constexpr bool kSpecialQueue = false, kSlowQueue = false, kTable = true;
  static constexpr size_t kTableBytes = sizeof(F8Table);
  // the table lookups want two 512-thread CTAs per SM; sized for two, the registers
  // (54 a thread) schedule the lookups 3 % faster than the compiler's own choice (48)
  static constexpr int kThreads = 512, kMinBlocks = 2;
  static __device__ __forceinline__ const void *table() { return f8_table<ID>().v; }
  static __device__ __forceinline__ uint32_t eval(const DevModel &m, const GaPairK &k, const uint16_t *tab,
                                                  const uint32_t (&wa)[2], const uint32_t (&wb)[2], uint32_t cb,
                                                  uint32_t &flag) {
    flag = 0u;
    return f8_eval<MCEMU_ARCH_GA_EARLY, ID, 8, RM != 0>(m, PipeConsts{(uint32_t)k.m1, k.p24, k.p22}, tab, wa, wb, cb);
  }
  static __device__ __forceinline__ uint32_t special(const DevModel &m, const uint32_t (&wa)[2],
                                                     const uint32_t (&wb)[2], uint32_t cb) {
    return pair_general<MCEMU_ARCH_GA_EARLY, ID, RM>(m, wa, wb, cb);
  }
  static __device__ __forceinline__ uint32_t general(const DevModel &m, const uint32_t (&wa)[2],
                                                     const uint32_t (&wb)[2], uint32_t cb) {
    return pair_general<MCEMU_ARCH_GA_EARLY, ID, RM>(m, wa, wb, cb);
  }
};

template <int ID, int RM> struct F8ExactPairEv {
  static constexpr bool kSpecialQueue = false, kSlowQueue = true, kTable = false;
  static constexpr size_t kTableBytes = 0;
  static constexpr int kThreads = kPairThreads, kMinBlocks = 0;
  static __device__ __forceinline__ const void *table() { return nullptr; }
  static __device__ __forceinline__ uint32_t eval(const DevModel &m, const GaPairK &, const uint16_t *,
                                                  const uint32_t (&wa)[2], const uint32_t (&wb)[2], uint32_t cb,
                                                  uint32_t &flag) {
    uint32_t r = 0u;
    flag = f8_exact_fp32<ID, 8>(m, wa, wb, cb, r) ? 0u : 2u;
    return r;
  }
  static __device__ __forceinline__ uint32_t special(const DevModel &m, const uint32_t (&wa)[2],
                                                     const uint32_t (&wb)[2], uint32_t cb) {
    return pair_general<MCEMU_ARCH_EXACT, ID, RM>(m, wa, wb, cb);
  }
  static __device__ __forceinline__ uint32_t general(const DevModel &m, const uint32_t (&wa)[2],
                                                     const uint32_t (&wb)[2], uint32_t cb) {
    return pair_general<MCEMU_ARCH_EXACT, ID, RM>(m, wa, wb, cb);
  }
};

template <class Ev>
static int f8_run_pair(const DevModel &m, size_t n, const void *a, const void *b, const uint32_t *c, uint32_t *d,
                       cudaStream_t s) {
  auto kern = pair_kernel<Ev>;
  const int shm = Ev::kTable ? (int)Ev::kTableBytes : 0;
  if (shm && cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, shm) != cudaSuccess)
    return MCEMU_ERR_CUDA;
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, Ev::kThreads, shm);
  if (per_sm < 1) per_sm = 1;
  const size_t np = n / 2, want = (np + Ev::kThreads - 1) / Ev::kThreads, full = (size_t)sms * per_sm;
  const int grid = (int)(want < full ? want : full);
  const GaPairK k{m.p0mul, m.p0cmul, 0, 1u, 2u, 1u << 16, 0u, 1u << 9, 1u << 23, -1, -2, 1u << 24, 1u << 22};
  kern<<<grid, Ev::kThreads, shm, s>>>(m, (uint32_t)np, (const uint4 *)a, (const uint4 *)b, (const uint2 *)c,
                                       (uint2 *)d, k);
  return cudaGetLastError() == cudaSuccess ? MCEMU_OK : MCEMU_ERR_CUDA;
}

// The paired kernel takes K = 8 sets with 16-byte-aligned operands and 8-byte-aligned
// c, d: global alignment through the product table (512-thread CTAs), and OCP
// exact-then-round on the FP32 pipe.  FNUZ exact-then-round, other block sizes and
// unaligned buffers keep f8_kernel, one set per thread.
template <int ID>
static bool f8_pair_ok(const DevModel &m, size_t n, const void *a, const void *b, const uint32_t *c, const uint32_t *d) {
  if (m.k != 8 || n < 2 || n / 2 >= (1u << 31)) return false;
  if (m.arch == MCEMU_ARCH_EXACT && Fmt<ID>::FNUZ) return false;
  return ((uintptr_t)a % 16) == 0 && ((uintptr_t)b % 16) == 0 && ((uintptr_t)c % 8) == 0 && ((uintptr_t)d % 8) == 0;
}

template <int ARCH, int ID, int K, bool RNE>
__global__ void __launch_bounds__(kF8Threads, 2) f8_kernel(const __grid_constant__ DevModel m, size_t n,
                                                           const uint8_t *__restrict__ a,
                                                           const uint8_t *__restrict__ b,
                                                           const uint32_t *__restrict__ c,
                                                           uint32_t *__restrict__ d, PipeConsts pc) {
  extern __shared__ uint4 f8_smem[];
  {
    const uint4 *src = reinterpret_cast<const uint4 *>(f8_table<ID>().v);
    for (int i = threadIdx.x; i < (int)(sizeof(F8Table) / sizeof(uint4)); i += blockDim.x) f8_smem[i] = src[i];
  }
  __syncthreads();
  const uint16_t *tab = reinterpret_cast<const uint16_t *>(f8_smem);
  constexpr int NW = K / 4;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  // software pipeline: the next vector set's words are loaded while this one is evaluated
  uint32_t na[NW], nb[NW], nc = 0;
  if constexpr (!(ARCH == MCEMU_ARCH_EXACT && !Fmt<ID>::FNUZ)) {
    // the table path with special values resolved in line (cheap next to the queue
    // below for these models)
    size_t v = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (v < n) f8_load<K>(a, b, c, v, na, nb, nc);
    for (; v < n; v += stride) {
      uint32_t wa[NW], wb[NW];
#pragma unroll
      for (int w = 0; w < NW; w++) { wa[w] = na[w]; wb[w] = nb[w]; }
      const uint32_t cb = nc;
      if (v + stride < n) f8_load<K>(a, b, c, v + stride, na, nb, nc);
      __stcs(d + v, f8_eval<ARCH, ID, K, RNE>(m, pc, tab, wa, wb, cb));
    }
  } else {
    // OCP exact-then-round: the FP32-pipe evaluation, special values included.  A
    // set whose rounding it leaves undecided joins a per-warp queue, and each time 32
    // have gathered the warp evaluates them through the table with every lane busy.
    __shared__ size_t queue[kF8Threads / 32][64];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t below = (1u << lane) - 1u;
    size_t *q = queue[warp];
    int qn = 0;                                          // warp-uniform queue length
    size_t base = (size_t)blockIdx.x * blockDim.x + (size_t)warp * 32;
    if (base + lane < n) f8_load<K>(a, b, c, base + lane, na, nb, nc);
    for (; base < n; base += stride) {
      const size_t v = base + lane;
      uint32_t wa[NW], wb[NW];
  #pragma unroll
      for (int w = 0; w < NW; w++) { wa[w] = na[w]; wb[w] = nb[w]; }
      const uint32_t cb = nc;
      if (v + stride < n) f8_load<K>(a, b, c, v + stride, na, nb, nc);
      bool defer = false;
      if (v < n) {
        uint32_t r;
        defer = !f8_exact_fp32<ID, K>(m, wa, wb, cb, r);
        if (!defer) __stcs(d + v, r);
      }
      const uint32_t mask = __ballot_sync(0xFFFFFFFFu, defer);
      if (mask) {
        if (defer) q[qn + __popc(mask & below)] = v;
        qn += __popc(mask);
        if (qn >= 32) {
          __syncwarp();
          const size_t u = q[qn - 32 + lane];
          uint32_t ua[NW], ub[NW], uc;
          f8_load<K>(a, b, c, u, ua, ub, uc);
          __stcs(d + u, f8_eval<ARCH, ID, K, RNE>(m, pc, tab, ua, ub, uc));
          qn -= 32;
          __syncwarp();
        }
      }
    }
    __syncwarp();
    if (lane < qn) {
      const size_t u = q[lane];
      uint32_t ua[NW], ub[NW], uc;
      f8_load<K>(a, b, c, u, ua, ub, uc);
      __stcs(d + u, f8_eval<ARCH, ID, K, RNE>(m, pc, tab, ua, ub, uc));
    }
  }
}

// ---------------------------------------------------------------------------
// launcher
// ---------------------------------------------------------------------------
// true when the table kernel implements the model: FP8 operands of one format,
// early-c global alignment with truncation and 32-bit sums, or exact-then-round;
// subnormals kept
bool f8_stream_ok(const DevModel &m, int id) {
  if (id != F_E4M3 && id != F_E4M3Z && id != F_E5M2 && id != F_E5M2Z) return false;
  if (m.acc16) return false;
  if (m.fa.sub_keep == 0u || m.c_sub_keep == 0u || m.sub_out_flush) return false;
  if (m.k != 8 && m.k != 16 && m.k != 32) return false;
  if (m.arch == MCEMU_ARCH_EXACT) return true;
  return m.arch == MCEMU_ARCH_GA_EARLY && !m.align_rd && !m.wide && m.P0 <= 24;
}

template <int ARCH, int ID, int K, bool RNE>
static int f8_run(const DevModel &m, size_t n, const void *a, const void *b, const uint32_t *c, uint32_t *d,
                  cudaStream_t s) {
  auto kern = f8_kernel<ARCH, ID, K, RNE>;
  const int shm = (int)sizeof(F8Table);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, shm) != cudaSuccess)
    return MCEMU_ERR_CUDA;
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kF8Threads, shm);
  if (per_sm < 1) per_sm = 1;
  size_t want = (n + kF8Threads - 1) / kF8Threads, full = (size_t)sms * per_sm;
  const int grid = (int)(want < full ? want : full);
  kern<<<grid, kF8Threads, shm, s>>>(m, n, (const uint8_t *)a, (const uint8_t *)b, c, d,
                                     PipeConsts{0xFFFFFFFFu, 1u << 24, 1u << 22});
  return cudaGetLastError() == cudaSuccess ? MCEMU_OK : MCEMU_ERR_CUDA;
}

template <int ARCH, int ID, bool RNE>
static int f8_run_k(const DevModel &m, size_t n, const void *a, const void *b, const uint32_t *c, uint32_t *d,
                    cudaStream_t s) {
  if (m.k == 8) return f8_run<ARCH, ID, 8, RNE>(m, n, a, b, c, d, s);
  if (m.k == 16) return f8_run<ARCH, ID, 16, RNE>(m, n, a, b, c, d, s);
  return f8_run<ARCH, ID, 32, RNE>(m, n, a, b, c, d, s);
}

template <int ID>
static int f8_run_id(const DevModel &m, size_t n, const void *a, const void *b, const uint32_t *c, uint32_t *d,
                     cudaStream_t s) {
  if (f8_pair_ok<ID>(m, n, a, b, c, d)) {
    int st;
    if (m.arch == MCEMU_ARCH_EXACT) st = m.rne ? f8_run_pair<F8ExactPairEv<ID, 1>>(m, n, a, b, c, d, s)
                                               : f8_run_pair<F8ExactPairEv<ID, 0>>(m, n, a, b, c, d, s);
    else st = m.rne ? f8_run_pair<F8GaPairEv<ID, 1>>(m, n, a, b, c, d, s)
                    : f8_run_pair<F8GaPairEv<ID, 0>>(m, n, a, b, c, d, s);
    if (st != MCEMU_OK || n % 2 == 0) return st;
    const size_t t = n - 1;                           // the odd last set: the one-set kernel
    return f8_run_id<ID>(m, 1, (const uint8_t *)a + 8 * t, (const uint8_t *)b + 8 * t, c + t, d + t, s);
  }
  if (m.arch == MCEMU_ARCH_EXACT) return f8_run_k<MCEMU_ARCH_EXACT, ID, true>(m, n, a, b, c, d, s);
  if (m.rne) return f8_run_k<MCEMU_ARCH_GA_EARLY, ID, true>(m, n, a, b, c, d, s);
  return f8_run_k<MCEMU_ARCH_GA_EARLY, ID, false>(m, n, a, b, c, d, s);
}

int launch_block_fma_f8(const DevModel &m, int id, size_t n, const void *a, const void *b, const uint32_t *c,
                        uint32_t *d, void *stream) {
  cudaStream_t s = (cudaStream_t)stream;
  switch (id) {
    case F_E4M3: return f8_run_id<F_E4M3>(m, n, a, b, c, d, s);
    case F_E4M3Z: return f8_run_id<F_E4M3Z>(m, n, a, b, c, d, s);
    case F_E5M2: return f8_run_id<F_E5M2>(m, n, a, b, c, d, s);
    default: return f8_run_id<F_E5M2Z>(m, n, a, b, c, d, s);
  }
}

}  // namespace mcemu

// stream_pair.cuh -- the paired block-FMA stream kernel for 8-byte operand sets
// (FP16/BF16 K=4, XF32 K=2, FP8 K=8): two vector sets per thread and iteration, and
// the evaluators of the model families it serves.  Included by stream.cu and
// stream_fp8.cu.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "core.cuh"

namespace mcemu {

constexpr int kPairThreads = 256;   // CTA size unless the evaluator names another (kThreads)

// ---------------------------------------------------------------------------
// Early-c global alignment with truncation on 8-byte operand sets (FP16/BF16 K=4),
// two vector sets per thread and iteration: one 16-byte load of a and of b, one
// 8-byte load of c, one 8-byte store of d.
//
// Two 16-bit elements are decoded at once: exponent fields by a mask, hidden bits
// and max(field, 1) by 16-bit-lane min/max, the products' field sums by one add.  A
// product with a zero significand takes no part in e_max (its exponent is replaced
// by -1024).  Each term is (U << P0) >> (e_max - e_l) with its sign applied by a
// multiply, and the integer sum S is rounded by the int -> fp32 conversion (RN or
// RZ) with e_max - F_p added to the exponent field.  Results that are zero, at or
// below 2^-126 in magnitude (subnormal, or the double-rounding boundary) take the
// general path in place; an overflow gives +-Inf (RNE) or +-max-finite (RTZ).  Sets
// with an Inf or NaN operand or addend are queued per warp with their words in
// shared memory and resolved 32 at a time from their special-value classes.
// Multiplies by run-time constants (GaPairK) keep shifts and signs on the FMA pipe.
// ---------------------------------------------------------------------------
struct GaPairK {
  uint32_t p0mul, p0cmul;   // 2^P0, 2^P0c
  int32_t lsb0;             // -(2 bias_a) - F_p: the result LSB exponent is e_max + lsb0
  uint32_t one, two, k16, kE, k9, k23;
  int32_t m1, m2;
  uint32_t p24, p22;        // 2^24, 2^22 (the FP8 table evaluator)
};

__device__ __forceinline__ uint32_t vmin2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("min.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t vmax2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

template <int ID> struct Pack16 {
  using F = Fmt<ID>;
  static constexpr uint32_t EM2 = (F::EMASK << F::MB) * 0x10001u;   // exponent fields
  static constexpr uint32_t MM2 = F::MMASK * 0x10001u;                // mantissa fields
  static constexpr uint32_t LSB2 = (1u << F::MB) * 0x10001u;          // field LSBs
};

// One FP16/BF16 K=4 set; flag bit 0: an Inf/NaN operand or addend, bit 1: the result is
// left to the general path.
template <int ID, int RM>
__device__ __forceinline__ uint32_t ga16_pair_eval(const GaPairK &k, const uint32_t (&wa)[2], const uint32_t (&wb)[2],
                                                   uint32_t cb, uint32_t &flag) {
  using P = Pack16<ID>;
  constexpr int BIAS = Fmt<ID>::BIAS;
  uint32_t U[4], E[4], X[2], top = 0;
#pragma unroll
  for (int i = 0; i < 2; i++) {
    const uint32_t ea = wa[i] & P::EM2, eb = wb[i] & P::EM2;
    top = vmax2(top, vmax2(ea, eb));
    const uint32_t Sa = (wa[i] & P::MM2) | vmin2(ea, P::LSB2);
    const uint32_t Sb = (wb[i] & P::MM2) | vmin2(eb, P::LSB2);
    const uint32_t Es = vmax2(ea, P::LSB2) * k.one + vmax2(eb, P::LSB2);   // (E_a' + E_b') << MB per half
    // hi products: the low half of Sa times the high half of Sb stays below 2^16 for
    // BF16, so it cannot reach the high word; FP16 masks both operands
    if constexpr (ID == F_BF16) U[2 * i + 1] = __umulhi(Sa, Sb & 0xFFFF0000u);
    else U[2 * i + 1] = __umulhi(Sa & 0xFFFF0000u, Sb & 0xFFFF0000u);
    U[2 * i] = __umulhi(Sa * k.k16, Sb * k.k16);
    E[2 * i + 1] = __umulhi(Es, k.kE);
    E[2 * i] = __umulhi(Es * k.k16, k.kE);
    X[i] = wa[i] ^ wb[i];
  }
  // the addend, its exponent on the products' biased scale (-1024 for c = 0)
  const uint32_t cef = cb & 0x7F800000u;
  const uint32_t cS = (cb & 0x7FFFFFu) | min(cef, 0x00800000u);
  const int32_t ce = cS ? (int32_t)(max(cef, 0x00800000u) >> 23) + (2 * BIAS - 127) : -1024;
  int32_t emax = ce;
#pragma unroll
  for (int l = 0; l < 4; l++) {
    const uint32_t nz = ID == F_BF16 ? U[l] : min(U[l], 1u);   // keeps nz * 2048 below 2^32
    emax = max(emax, min((int32_t)E[l], (int32_t)(nz * 2048u) - 1024));
  }
  int32_t S = 0;
#pragma unroll
  for (int l = 0; l < 4; l++) {
    const uint32_t t = shr32(U[l] * k.p0mul, (int32_t)E[l] * k.m1 + emax);
    const uint32_t xs = (l & 1) ? X[l / 2] : X[l / 2] * k.k16;
    S += (int32_t)t * ((int32_t)__umulhi(xs, k.two) * k.m2 + 1);
  }
  S += (int32_t)shr32(cS * k.p0cmul, ce * k.m1 + emax) * ((int32_t)__umulhi(cb, k.two) * k.m2 + 1);
  flag = (((top + P::LSB2) & 0x80008000u) || cef == 0x7F800000u) ? 1u : 0u;
  // |S| in [1, 2^31): the conversion rounds it to 24 bits as the model does; adding
  // e_max - F_p to the exponent field is exact while the result stays normal
  const uint32_t aS = (uint32_t)abs(S);
  const float f = RM ? __uint2float_rn(aS) : __uint2float_rz(aS);
  const int32_t lsb = emax + k.lsb0;
  const int32_t fb = (int32_t)__float_as_uint(f);
  const int32_t rb = fb + lsb * (int32_t)k.k23;
  const int32_t ex = (int32_t)__umulhi((uint32_t)fb, k.k9) + lsb;   // exponent field of the result
  uint32_t r = (uint32_t)rb;
  if (ex >= 255) r = overflow_bits(RM);
  if ((rb <= 0x00800000 && ex < 255) || S == 0) flag |= 2u;
  return r | ((uint32_t)S & 0x80000000u);
}

// Special result of a BF16 set with an Inf or NaN operand or addend, from the classes
// of its elements (two per word, flags at bits 15 and 31): NaN for a NaN, Inf * 0 or
// +Inf and -Inf together, else the signed Inf.
template <int ID>
__device__ __forceinline__ uint32_t special16_classes(const DevModel &m, const uint32_t (&wa)[2],
                                                      const uint32_t (&wb)[2], uint32_t cb) {
  using P = Pack16<ID>;
  constexpr uint32_t SB2 = 0x80008000u;
  uint32_t nan = 0, pinf = 0, ninf = 0;
#pragma unroll
  for (int i = 0; i < 2; i++) {
    uint32_t in[2], nn[2], z[2];
#pragma unroll
    for (int o = 0; o < 2; o++) {
      const uint32_t w = o ? wb[i] : wa[i];
      const uint32_t top = ((w & P::EM2) + P::LSB2) & SB2;          // field all ones
      const uint32_t mz = ((w & P::MM2) + 0x7FFF7FFFu) & SB2;       // mantissa nonzero
      z[o] = ~((w & 0x7FFF7FFFu) + 0x7FFF7FFFu) & SB2;              // +-0
      nn[o] = top & mz;
      in[o] = top & ~mz;
    }
    nan |= nn[0] | nn[1] | (in[0] & z[1]) | (z[0] & in[1]);
    const uint32_t ip = in[0] | in[1], sg = (wa[i] ^ wb[i]) & SB2;
    pinf |= ip & ~sg;
    ninf |= ip & sg;
  }
  if ((cb & 0x7F800000u) == 0x7F800000u) {
    if (cb & 0x7FFFFFu) nan = 1u;
    else if (cb >> 31) ninf = 1u;
    else pinf = 1u;
  }
  if (nan || (pinf && ninf)) return m.nan_bits;
  return pinf ? 0x7F800000u : 0xFF800000u;
}

template <int ID>
__device__ __forceinline__ uint32_t ga16_pair_special(const DevModel &m, const uint32_t (&wa)[2], const uint32_t (&wb)[2],
                                                      uint32_t cb) {
  if constexpr (ID == F_FP16) {
    // FP16 products and sums with an fp32 c stay finite in fp32: the IEEE sum's class
    // is the model's special result
    uint32_t ea[4], eb[4];
#pragma unroll
    for (int l = 0; l < 4; l++) {
      ea[l] = felem<ID>(wa, l);
      eb[l] = felem<ID>(wb, l);
    }
    return resolve_special(m, fspecial_bits<ID, 4>(m, ea, eb, cb));
  } else {
    return special16_classes<ID>(m, wa, wb, cb);
  }
}

// XF32 (truncated to 10 mantissa bits) K=2 sets in the same way: one element per word.
template <int RM>
__device__ __forceinline__ uint32_t gaxf_pair_eval(const GaPairK &k, const uint32_t (&wa)[2], const uint32_t (&wb)[2],
                                                   uint32_t cb, uint32_t &flag) {
  uint32_t U[2], E[2], top = 0;
#pragma unroll
  for (int l = 0; l < 2; l++) {
    const uint32_t ea = wa[l] & 0x7F800000u, eb = wb[l] & 0x7F800000u;
    top = max(top, max(ea, eb));
    // significand with its hidden bit, shifted down by the 13 truncated bits
    const uint32_t Sa = __umulhi((wa[l] & 0x007FE000u) | min(ea, 0x00800000u), k.k9 << 10);
    const uint32_t Sb = __umulhi((wb[l] & 0x007FE000u) | min(eb, 0x00800000u), k.k9 << 10);
    U[l] = Sa * Sb;
    E[l] = __umulhi(max(ea, 0x00800000u) * k.one + max(eb, 0x00800000u), k.k9);
  }
  const uint32_t cef = cb & 0x7F800000u;
  const uint32_t cS = (cb & 0x7FFFFFu) | min(cef, 0x00800000u);
  const int32_t ce = cS ? (int32_t)(max(cef, 0x00800000u) >> 23) + 127 : -1024;
  int32_t emax = ce;
#pragma unroll
  for (int l = 0; l < 2; l++) emax = max(emax, min((int32_t)E[l], (int32_t)(min(U[l], 1u) * 2048u) - 1024));
  int32_t S = 0;
#pragma unroll
  for (int l = 0; l < 2; l++) {
    const uint32_t t = shr32(U[l] * k.p0mul, (int32_t)E[l] * k.m1 + emax);
    S += (int32_t)t * ((int32_t)__umulhi(wa[l] ^ wb[l], k.two) * k.m2 + 1);
  }
  S += (int32_t)shr32(cS * k.p0cmul, ce * k.m1 + emax) * ((int32_t)__umulhi(cb, k.two) * k.m2 + 1);
  flag = (top == 0x7F800000u || cef == 0x7F800000u) ? 1u : 0u;
  const uint32_t aS = (uint32_t)abs(S);
  const float f = RM ? __uint2float_rn(aS) : __uint2float_rz(aS);
  const int32_t lsb = emax + k.lsb0;
  const int32_t fb = (int32_t)__float_as_uint(f);
  const int32_t rb = fb + lsb * (int32_t)k.k23;
  const int32_t ex = (int32_t)__umulhi((uint32_t)fb, k.k9) + lsb;
  uint32_t r = (uint32_t)rb;
  if (ex >= 255) r = overflow_bits(RM);
  if ((rb <= 0x00800000 && ex < 255) || S == 0) flag |= 2u;
  return r | ((uint32_t)S & 0x80000000u);
}

// Special result of an XF32 set with an Inf or NaN operand or addend (classes of the
// fp32 containers; zero means no mantissa bit above the 13 truncated ones).
__device__ __forceinline__ uint32_t specialxf_classes(const DevModel &m, const uint32_t (&wa)[2],
                                                      const uint32_t (&wb)[2], uint32_t cb) {
  bool nan = false, pinf = false, ninf = false;
#pragma unroll
  for (int l = 0; l < 2; l++) {
    const uint32_t x = wa[l], y = wb[l];
    const bool tx = (x & 0x7F800000u) == 0x7F800000u, ty = (y & 0x7F800000u) == 0x7F800000u;
    const bool nx = tx && (x & 0x7FFFFFu), ny = ty && (y & 0x7FFFFFu);
    const bool ix = tx && !nx, iy = ty && !ny;
    const bool zx = (x & 0x7FFFE000u) == 0u, zy = (y & 0x7FFFE000u) == 0u;
    nan = nan || nx || ny || (ix && zy) || (zx && iy);
    if (ix || iy) {
      if ((x ^ y) >> 31) ninf = true;
      else pinf = true;
    }
  }
  if ((cb & 0x7F800000u) == 0x7F800000u) {
    if (cb & 0x7FFFFFu) nan = true;
    else if (cb >> 31) ninf = true;
    else pinf = true;
  }
  if (nan || (pinf && ninf)) return m.nan_bits;
  return pinf ? 0x7F800000u : 0xFF800000u;
}

// Evaluators of the pair kernel.  eval() returns the result of one set and a flag
// (bit 0: an Inf/NaN operand or addend, bit 1: the general path decides); special()
// resolves a flagged set from its words; general() evaluates one set on the integer
// path.  kSpecialQueue: eval() may set flag bit 0 (else it never does, and the kernel
// keeps no queue for it); kSlowQueue: sets with flag 2 are common enough to be batched
// per warp (else they are evaluated in place).
template <int ID> struct PairFmt {
  static constexpr int K = ID == F_XF32T ? 2 : (Fmt<ID>::BYTES == 2 ? 4 : 8);
};

template <int ARCH, int ID, int RM>
__device__ __forceinline__ uint32_t pair_general(const DevModel &m, const uint32_t (&wa)[2], const uint32_t (&wb)[2],
                                                 uint32_t cb) {
  constexpr int K = PairFmt<ID>::K;
  uint32_t ea[K], eb[K];
#pragma unroll
  for (int l = 0; l < K; l++) {
    ea[l] = felem<ID>(wa, l);
    eb[l] = felem<ID>(wb, l);
  }
  return block_fma_fast<ARCH, ID, K, uint32_t, int32_t, RM>(m, ea, eb, cb, true);
}

template <int ID, int RM> struct GaPairEv {
  static constexpr bool kSpecialQueue = true, kSlowQueue = false, kTable = false;
  static constexpr size_t kTableBytes = 0;
  static constexpr int kThreads = kPairThreads, kMinBlocks = 0;
  static __device__ __forceinline__ const void *table() { return nullptr; }
  static __device__ __forceinline__ uint32_t eval(const DevModel &, const GaPairK &k, const uint16_t *, const uint32_t (&wa)[2],
                                                  const uint32_t (&wb)[2], uint32_t cb, uint32_t &flag) {
    if constexpr (ID == F_XF32T) return gaxf_pair_eval<RM>(k, wa, wb, cb, flag);
    else return ga16_pair_eval<ID, RM>(k, wa, wb, cb, flag);
  }
  static __device__ __forceinline__ uint32_t special(const DevModel &m, const uint32_t (&wa)[2],
                                                     const uint32_t (&wb)[2], uint32_t cb) {
    if constexpr (ID == F_XF32T) return specialxf_classes(m, wa, wb, cb);
    else return ga16_pair_special<ID>(m, wa, wb, cb);
  }
  static __device__ __forceinline__ uint32_t general(const DevModel &m, const uint32_t (&wa)[2],
                                                     const uint32_t (&wb)[2], uint32_t cb) {
    return pair_general<MCEMU_ARCH_GA_EARLY, ID, RM>(m, wa, wb, cb);
  }
};

// Exact-then-round with RNE of one BF16 (K = 4, two elements per word) or truncated
// XF32 (K = 2) set on the FP32 pipe, every term split against one constant
// (ExtractScalar of Rump, Ogita and Oishi, "Accurate floating-point summation part I:
// faithful rounding", SIAM J. Sci. Comput. 31, 2008, Lemma 3.3):
//  - an element a with exponent field f_a (taken as min(max(f_a, 1), 254)) becomes
//    a1 = a 2^(128 - f_a), in [2, 4) when normal and (0, 2) when subnormal, so p = a1 b1
//    is exact (8 x 8 or 11 x 11 significand bits) and a b = p 2^(F - 256), F = f_a + f_b;
//  - with M = max(F over the products, max(f_c, 1) + 127) every term is scaled by
//    2^(256 - M): a product to x = p 2^(F - M), |x| < 16, and c to x_c = c 2^(256 - M),
//    |x_c| < 8, by two exact power-of-two multiplies (exponents in [-126, 64]; only a
//    subnormal x_c, below 2^-126, is rounded).  A product with F - M < -126 keeps the
//    scale 2^-126 instead: the term it adds and the one it stands for are both below
//    2^-122;
//  - with sigma = 2^7 (K = 4) or 2^6 (K = 2), q = fl(sigma + x) - sigma and r = x - q are
//    exact (x enters through one fused multiply-add each); every q is a multiple of
//    ulp(sigma) / 2 and |sum q| < sigma, so tau = sum q is exact, and |r| <= ulp(sigma) / 2;
//  - P = fl(sum r) (K additions) is off from sum r by at most gamma_K (K + 1) ulp(sigma)
//    / 2 < 2^-36.6 (K = 4) or 2^-39.4 (K = 2) (Higham, Accuracy and Stability of Numerical
//    Algorithms, Sec. 4.2); with the rescaled small terms that stays below kBound;
//  - when |tau| >= |P|, Dekker's Fast2Sum gives t + r = tau + P exactly, so the exact sum
//    is t + r + d with |d| < kBound, and t is its RNE rounding when |r| + kBound is below
//    half the spacing of the floats next to t (the smaller one, below |t|).
// The rounded t goes back by 2^(M - 256) on its exponent field; one at or beyond 2^128
// is +-Inf.  A zero, tiny (< 2^-124 after scaling), subnormal or undecided result
// returns 2 (the integer path).  Special values:
//  - BF16: an Inf or NaN operand or c keeps its class through the positive scales, so
//    tau is the IEEE sum's special value: NaN (nan_bits) for a NaN, Inf * 0 or Inf - Inf,
//    else the signed Inf (the model's special results); sw stays 0;
//  - XF32: a NaN whose mantissa lies in the 13 truncated bits would read as an Inf
//    here, so sw flags any operand or c with an exponent field of all ones and the
//    caller resolves the set from its raw words.
template <int ID>
__device__ __forceinline__ int sigma_exact_rn(const uint32_t (&wa)[2], const uint32_t (&wb)[2], uint32_t cb,
                                              uint32_t nan_bits, uint32_t &out, uint32_t &sw) {
  static_assert(ID == F_BF16 || ID == F_XF32T, "BF16 or truncated XF32 elements");
  constexpr int K = ID == F_BF16 ? 4 : 2;
  constexpr float kSigma = K == 4 ? 0x1p7f : 0x1p6f;
  constexpr float kBound = K == 4 ? 0x1p-36f : 0x1p-39f;
  constexpr uint32_t kE255 = 255u << 23, kE127 = 127u << 23;
  float p[K];
  uint32_t F23[K];                                     // F << 23 (F <= 508: fits unsigned)
  if constexpr (ID == F_BF16) {
#pragma unroll
    for (int i = 0; i < 2; i++) {
      // min(max(field, 1), 254) << 7 in each 16-bit half; << 16 and the high half's mask
      // put it at bit 23
      const uint32_t Ea = vmin2(vmax2(wa[i] & 0x7F807F80u, 0x00800080u), 0x7F007F00u);
      const uint32_t Eb = vmin2(vmax2(wb[i] & 0x7F807F80u, 0x00800080u), 0x7F007F00u);
      const float a_lo = __fmul_rn(__uint_as_float(wa[i] << 16), __uint_as_float(kE255 - (Ea << 16)));
      const float b_lo = __fmul_rn(__uint_as_float(wb[i] << 16), __uint_as_float(kE255 - (Eb << 16)));
      const float a_hi = __fmul_rn(__uint_as_float(wa[i] & 0xFFFF0000u), __uint_as_float(kE255 - (Ea & 0xFFFF0000u)));
      const float b_hi = __fmul_rn(__uint_as_float(wb[i] & 0xFFFF0000u), __uint_as_float(kE255 - (Eb & 0xFFFF0000u)));
      p[2 * i] = __fmul_rn(a_lo, b_lo);
      p[2 * i + 1] = __fmul_rn(a_hi, b_hi);
      const uint32_t Es = Ea + Eb;                     // per half (F << 7) <= 508 << 7: no carry
      F23[2 * i] = Es << 16;
      F23[2 * i + 1] = Es & 0xFFFF0000u;
    }
    sw = 0u;
  } else {
    // the fields are not clamped: a set with an Inf or NaN is resolved by the caller
    uint32_t top = cb & 0x7F800000u;
#pragma unroll
    for (int l = 0; l < 2; l++) {
      const uint32_t xa = wa[l] & 0xFFFFE000u, xb = wb[l] & 0xFFFFE000u;   // 10 mantissa bits
      const uint32_t Ea = max(xa & 0x7F800000u, 1u << 23), Eb = max(xb & 0x7F800000u, 1u << 23);
      top = max(top, max(Ea, Eb));
      p[l] = __fmul_rn(__fmul_rn(__uint_as_float(xa), __uint_as_float(kE255 - Ea)),
                       __fmul_rn(__uint_as_float(xb), __uint_as_float(kE255 - Eb)));
      F23[l] = Ea + Eb;
    }
    sw = top == kE255 ? 1u : 0u;
  }
  const uint32_t cf = cb & 0x7F800000u;
  uint32_t M23 = (ID == F_BF16 ? min(max(cf, 1u << 23), 254u << 23) : max(cf, 1u << 23)) + kE127;
#pragma unroll
  for (int l = 0; l < K; l++) M23 = max(M23, F23[l]);
  // c * 2^k, k = 256 - M in [-252, 128], as 2^k1 2^k2 with k1 = floor(k / 2)
  const int32_t k23 = (int32_t)(0x80000000u - M23);
  const int32_t k1 = (k23 >> 1) & (int32_t)0xFF800000;
  const float xc = __fmul_rn(__fmul_rn(__uint_as_float(cb), __uint_as_float((uint32_t)k1 + kE127)),
                             __uint_as_float((uint32_t)(k23 - k1) + kE127));
  float tq = __fadd_rn(__fadd_rn(xc, kSigma), -kSigma);
  float P = __fadd_rn(xc, -tq);
#pragma unroll
  for (int l = 0; l < K; l++) {
    const float sc = __uint_as_float(kE127 - min(M23 - F23[l], 126u << 23));   // 2^(F - M), >= 2^-126
    const float q = __fadd_rn(__fmaf_rn(p[l], sc, kSigma), -kSigma);
    tq = __fadd_rn(tq, q);
    P = __fadd_rn(P, __fmaf_rn(p[l], sc, -q));
  }
  if (!(fabsf(tq) <= 0x1p7f)) {                        // an Inf or NaN operand or c
    out = tq != tq ? nan_bits : __float_as_uint(tq);
    return 0;
  }
  const float t = __fadd_rn(tq, P);
  const float r = __fadd_rn(P, -__fadd_rn(t, -tq));
  const uint32_t tb = __float_as_uint(t), ta = tb & 0x7FFFFFFFu;
  const int32_t fr = (int32_t)(ta >> 23) - (k23 >> 23);   // the result's exponent field
  // 2^e of the float just below |t|: half its spacing is 2^(e - 24)
  const float h = __uint_as_float((ta - 1u) & 0x7F800000u);
  out = fr > 254 ? (tb & 0x80000000u) | 0x7F800000u : tb - (uint32_t)k23;
  const bool ok = fabsf(tq) >= fabsf(P) && ta >= (3u << 23) && fr >= 1 &&
                  fabsf(r) < __fmaf_rd(h, 0x1p-24f, -kBound);
  return ok ? 0 : 2;
}

// Exact-then-round on the FP32 pipe: FP16 with exact fp32 products and BF16 with RNE
// through sigma_exact_rn, both with special values from the IEEE sums in line;
// truncated XF32 with RNE through sigma_exact_rn, and BF16 and XF32 with RZ through
// exact_scaled, whose error bound follows the terms (an RZ decision needs the sign of a
// remainder that can lie far below any fixed bound), with special values queued and
// resolved from their classes.  A rounding the error bound leaves
// undecided, a subnormal addend or result goes to the integer path, 32 at a time.
template <int ID, int RM> struct ExactPairEv {
  static constexpr bool kSpecialQueue = ID == F_XF32T || (ID == F_BF16 && RM == 0), kSlowQueue = true, kTable = false;
  static constexpr size_t kTableBytes = 0;
  // truncated XF32 with RNE: registers sized for three CTAs per SM (80 a thread)
  // run 7 % faster than the compiler's own choice (64, four CTAs)
  static constexpr int kThreads = kPairThreads, kMinBlocks = ID == F_XF32T && RM == 1 ? 3 : 0;
  static __device__ __forceinline__ const void *table() { return nullptr; }
  static __device__ __forceinline__ uint32_t eval(const DevModel &m, const GaPairK &, const uint16_t *, const uint32_t (&wa)[2],
                                                  const uint32_t (&wb)[2], uint32_t cb, uint32_t &flag) {
    uint32_t r = 0u;
    if constexpr (ID == F_FP16) {
      float p[4];
#pragma unroll
      for (int i = 0; i < 2; i++) {
        const float2 fa = __half22float2(*reinterpret_cast<const __half2 *>(&wa[i]));
        const float2 fb = __half22float2(*reinterpret_cast<const __half2 *>(&wb[i]));
        p[2 * i] = __fmul_rn(fa.x, fb.x);
        p[2 * i + 1] = __fmul_rn(fa.y, fb.y);
      }
      flag = exact_fp32_sum<4>(p, cb, RM, m.nan_bits, r) ? 2u : 0u;
    } else if constexpr (RM == 1) {
      uint32_t sw;
      const int st = sigma_exact_rn<ID>(wa, wb, cb, m.nan_bits, r, sw);
      flag = sw ? 1u : (st ? 2u : 0u);
    } else {
      uint32_t sw = (cb & 0x7F800000u) == 0x7F800000u;
#pragma unroll
      for (int i = 0; i < 2; i++) sw |= fspecial_word<ID>(wa[i]) | fspecial_word<ID>(wb[i]);
      const int st = exact_scaled<ID, PairFmt<ID>::K, 2>(wa, wb, cb, RM, r);
      flag = sw ? 1u : (st ? 2u : 0u);
    }
    return r;
  }
  static __device__ __forceinline__ uint32_t special(const DevModel &m, const uint32_t (&wa)[2],
                                                     const uint32_t (&wb)[2], uint32_t cb) {
    if constexpr (ID == F_XF32T) return specialxf_classes(m, wa, wb, cb);
    else return special16_classes<ID>(m, wa, wb, cb);
  }
  static __device__ __forceinline__ uint32_t general(const DevModel &m, const uint32_t (&wa)[2],
                                                     const uint32_t (&wb)[2], uint32_t cb) {
    return pair_general<MCEMU_ARCH_EXACT, ID, RM>(m, wa, wb, cb);
  }
};

// A warp's queue of flagged sets, kept with their data: the four operand words of a set
// in one 16-byte entry and (c, index) in an 8-byte one, so that a set goes in and out
// with one vector access of each.
struct PairQueue {
  uint4 *ab;
  uint2 *ci;
};
constexpr int kPairQueue = 96;      // entries per warp: fewer than 32 left over plus 64 new ones

// Append the flagged sets of this iteration (at most two per lane) to a warp queue and
// resolve it 32 entries at a time; qn is warp-uniform.
template <class Fn>
__device__ __forceinline__ void pair_enqueue(PairQueue q, int &qn, bool s0, bool s1, uint4 xa, uint4 xb, uint2 xc,
                                             uint32_t p, uint32_t below, int lane, uint32_t *d32, Fn resolve) {
  const uint32_t m0 = __ballot_sync(0xFFFFFFFFu, s0), m1 = __ballot_sync(0xFFFFFFFFu, s1);
  if (!(m0 | m1)) return;
  if (s0) {
    const int j = qn + __popc(m0 & below);
    q.ab[j] = make_uint4(xa.x, xa.y, xb.x, xb.y);
    q.ci[j] = make_uint2(xc.x, 2 * p);
  }
  qn += __popc(m0);
  if (s1) {
    const int j = qn + __popc(m1 & below);
    q.ab[j] = make_uint4(xa.z, xa.w, xb.z, xb.w);
    q.ci[j] = make_uint2(xc.y, 2 * p + 1);
  }
  qn += __popc(m1);
  while (qn >= 32) {
    __syncwarp();
    const uint4 e = q.ab[qn - 32 + lane];
    const uint2 ci = q.ci[qn - 32 + lane];
    const uint32_t ua[2] = {e.x, e.y}, ub[2] = {e.z, e.w};
    d32[ci.y] = resolve(ua, ub, ci.x);
    qn -= 32;
    __syncwarp();
  }
}

template <class Fn>
__device__ __forceinline__ void pair_drain(PairQueue q, int qn, int lane, uint32_t *d32, Fn resolve) {
  __syncwarp();
  if (lane < qn) {
    const uint4 e = q.ab[lane];
    const uint2 ci = q.ci[lane];
    const uint32_t ua[2] = {e.x, e.y}, ub[2] = {e.z, e.w};
    d32[ci.y] = resolve(ua, ub, ci.x);
  }
}

// Ev::kTable: the evaluator reads a lookup table of Ev::kTableBytes, which every CTA
// copies from global into dynamic shared memory first.  Ev::kMinBlocks: the CTAs per
// SM the register budget is sized for (0 leaves it to the compiler).
template <class Ev>
__global__ void __launch_bounds__(Ev::kThreads, Ev::kMinBlocks) pair_kernel(const __grid_constant__ DevModel m, uint32_t npairs,
                                                            const uint4 *__restrict__ a, const uint4 *__restrict__ b,
                                                            const uint2 *__restrict__ c, uint2 *__restrict__ d,
                                                            const GaPairK k) {
  extern __shared__ uint4 pair_table[];
  const uint16_t *tab = nullptr;
  if constexpr (Ev::kTable) {
    const uint4 *src = reinterpret_cast<const uint4 *>(Ev::table());
    for (int i = threadIdx.x; i < (int)(Ev::kTableBytes / sizeof(uint4)); i += blockDim.x) pair_table[i] = src[i];
    __syncthreads();
    tab = reinterpret_cast<const uint16_t *>(pair_table);
  }
  constexpr int kSpecWarps = Ev::kSpecialQueue ? Ev::kThreads / 32 : 1;
  constexpr int kSlowWarps = Ev::kSlowQueue ? Ev::kThreads / 32 : 1;
  __shared__ uint4 queue_ab[kSpecWarps][kPairQueue];
  __shared__ uint2 queue_ci[kSpecWarps][kPairQueue];
  __shared__ uint4 slow_ab[kSlowWarps][kPairQueue];
  __shared__ uint2 slow_ci[kSlowWarps][kPairQueue];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t below = (1u << lane) - 1u;
  const PairQueue q{queue_ab[Ev::kSpecialQueue ? warp : 0], queue_ci[Ev::kSpecialQueue ? warp : 0]};
  const PairQueue qs{slow_ab[Ev::kSlowQueue ? warp : 0], slow_ci[Ev::kSlowQueue ? warp : 0]};
  int qn = 0, qsn = 0;                                          // warp-uniform
  const uint32_t stride = gridDim.x * blockDim.x;
  const uint32_t first = blockIdx.x * blockDim.x + threadIdx.x;
  const uint32_t pend = (npairs + 31u) & ~31u;                  // every lane of a warp iterates alike
  uint32_t *d32 = reinterpret_cast<uint32_t *>(d);
  auto special = [&](const uint32_t (&ua)[2], const uint32_t (&ub)[2], uint32_t uc) { return Ev::special(m, ua, ub, uc); };
  auto general = [&](const uint32_t (&ua)[2], const uint32_t (&ub)[2], uint32_t uc) { return Ev::general(m, ua, ub, uc); };
  // software pipeline: the next pair is loaded while this one is evaluated
  uint4 na = {}, nb = {};
  uint2 nc = {};
  if (first < npairs) {
    na = __ldcs(a + first);
    nb = __ldcs(b + first);
    nc = __ldcs(c + first);
  }
  for (uint32_t base = first - lane; base < pend; base += stride) {
    const uint32_t p = base + lane;
    const uint4 xa = na, xb = nb;
    const uint2 xc = nc;
    if (p + stride < npairs) {
      na = __ldcs(a + p + stride);
      nb = __ldcs(b + p + stride);
      nc = __ldcs(c + p + stride);
    }
    const uint32_t wa0[2] = {xa.x, xa.y}, wb0[2] = {xb.x, xb.y}, wa1[2] = {xa.z, xa.w}, wb1[2] = {xb.z, xb.w};
    uint32_t f0 = 0, f1 = 0;
    if (p < npairs) {
      uint2 r;
      r.x = Ev::eval(m, k, tab, wa0, wb0, xc.x, f0);
      r.y = Ev::eval(m, k, tab, wa1, wb1, xc.y, f1);
      if constexpr (!Ev::kSlowQueue) {
        if (f0 == 2u) r.x = Ev::general(m, wa0, wb0, xc.x);
        if (f1 == 2u) r.y = Ev::general(m, wa1, wb1, xc.y);
      }
      __stcs(d + p, r);
    }
    if constexpr (Ev::kSpecialQueue)
      pair_enqueue(q, qn, (f0 & 1u) != 0u, (f1 & 1u) != 0u, xa, xb, xc, p, below, lane, d32, special);
    if constexpr (Ev::kSlowQueue)
      pair_enqueue(qs, qsn, f0 == 2u, f1 == 2u, xa, xb, xc, p, below, lane, d32, general);
  }
  if constexpr (Ev::kSpecialQueue) pair_drain(q, qn, lane, d32, special);
  if constexpr (Ev::kSlowQueue) pair_drain(qs, qsn, lane, d32, general);
}

}  // namespace mcemu

// stream.cu -- the block-FMA stream: one vector set (a[0..k-1], b[0..k-1], c)
// per thread, eq. (1) of "Accurate Models of AMD Matrix Cores" under the model.
//
// The data are read once, so the kernel is a grid-stride stream of 8-, 16- or
// 32-byte vector loads with the evict-first cache hint.  The work per vector is
// integer ALU (decode, significand products, max, shifts, one normalisation) for the
// alignment models; exact-then-round runs on the FP32 pipe (exact products, TwoSum)
// and leaves the sets it does not decide to the integer path, batched per warp.
#include <cuda_runtime.h>

#include <type_traits>

#include "core.cuh"

namespace mcemu {

// container sizes: CT 1/2/4 = bytes per element (4 = XF32-style, <= 11-bit
// significands), CT 5 = full binary32 inputs (48-bit significand products)
template <int CT> struct CtBytes { static constexpr int v = CT == 5 ? 4 : CT; };

template <int NB>
__device__ __forceinline__ void load_words(const uint8_t *p, uint32_t (&w)[(NB + 3) / 4]) {
  if constexpr (NB == 1) {
    w[0] = __ldcs(p);
  } else if constexpr (NB == 2) {
    w[0] = __ldcs(reinterpret_cast<const unsigned short *>(p));
  } else if constexpr (NB == 4) {
    w[0] = __ldcs(reinterpret_cast<const unsigned int *>(p));
  } else if constexpr (NB == 8) {
    uint2 v = __ldcs(reinterpret_cast<const uint2 *>(p));
    w[0] = v.x; w[1] = v.y;
  } else {
#pragma unroll
    for (int i = 0; i < NB / 16; i++) {
      uint4 v = __ldcs(reinterpret_cast<const uint4 *>(p) + i);
      w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
    }
  }
}

template <int ESZ, int K, int NW>
__device__ __forceinline__ void split_elems(const uint32_t (&w)[NW], uint32_t (&e)[K], int nt) {
#pragma unroll
  for (int l = 0; l < K; l++) {
    uint32_t x = 0;
    if (l < nt) {
      if constexpr (ESZ == 1) x = (w[l / 4] >> (8 * (l % 4))) & 0xFFu;
      else if constexpr (ESZ == 2) x = (w[l / 2] >> (16 * (l % 2))) & 0xFFFFu;
      else x = w[l];
    }
    e[l] = x;
  }
}

// Integer formats (INT8/UINT8): exact int32 dot product plus c.
template <int KM>
__global__ void __launch_bounds__(256) block_int_kernel(const __grid_constant__ DevModel m, size_t n,
                                                        const uint8_t *__restrict__ a,
                                                        const uint8_t *__restrict__ b,
                                                        const uint32_t *__restrict__ c,
                                                        uint32_t *__restrict__ d) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const bool ss = m.fa.is_signed && m.fb.is_signed, uu = !m.fa.is_signed && !m.fb.is_signed;
  // software pipeline: the next vector set is loaded while this one is reduced
  uint32_t na[KM / 4], nb[KM / 4], nc = 0;
  size_t v = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (v < n) {
    load_words<KM>(a + v * KM, na);
    load_words<KM>(b + v * KM, nb);
    nc = __ldcs(c + v);
  }
  for (; v < n; v += stride) {
    uint32_t wa[KM / 4], wb[KM / 4];
#pragma unroll
    for (int i = 0; i < KM / 4; i++) { wa[i] = na[i]; wb[i] = nb[i]; }
    const uint32_t cb = nc;
    if (v + stride < n) {
      load_words<KM>(a + (v + stride) * KM, na);
      load_words<KM>(b + (v + stride) * KM, nb);
      nc = __ldcs(c + v + stride);
    }
    int32_t s = 0;       // exact: |sum| <= 32 * 255 * 255
    if (ss) {
#pragma unroll
      for (int i = 0; i < KM / 4; i++) s = __dp4a((int)wa[i], (int)wb[i], s);
    } else if (uu) {
#pragma unroll
      for (int i = 0; i < KM / 4; i++) s = (int32_t)__dp4a(wa[i], wb[i], (unsigned)s);
    } else {
      uint32_t ea[KM], eb[KM];
      split_elems<1, KM>(wa, ea, KM);
      split_elems<1, KM>(wb, eb, KM);
      s = (int32_t)block_int<KM>(m, ea, eb, KM, 0u);
    }
    uint32_t r;
    if (m.int_sat) {
      int64_t t = (int64_t)s + (int64_t)(int32_t)cb;
      t = t > INT32_MAX ? INT32_MAX : (t < INT32_MIN ? INT32_MIN : t);
      r = (uint32_t)(int32_t)t;
    } else {
      r = (uint32_t)s + cb;
    }
    __stcs(d + v, r);
  }
}

// Specialised kernel: architecture, format and block size fixed at compile time.
template <int ARCH, int ID, int KM, bool WIDE>
__device__ __forceinline__ uint32_t fast_one(const DevModel &m, const uint8_t *__restrict__ a,
                                             const uint8_t *__restrict__ b, const uint32_t *__restrict__ c,
                                             size_t v) {
  constexpr int NB = KM * Fmt<ID>::BYTES;
  constexpr int NW = (NB + 3) / 4;
  using UT = typename std::conditional<(WIDE || ID == F_FP32), uint64_t, uint32_t>::type;
  using AT = typename std::conditional<(WIDE || ID == F_FP32), int64_t, int32_t>::type;
  uint32_t wa[NW], wb[NW];
  load_words<NB>(a + v * NB, wa);
  load_words<NB>(b + v * NB, wb);
  const uint32_t cb = __ldcs(c + v);
  uint32_t ea[KM], eb[KM];
#pragma unroll
  for (int l = 0; l < KM; l++) {
    ea[l] = felem<ID>(wa, l);
    eb[l] = felem<ID>(wb, l);
  }
  // a queued set has an Inf/NaN operand or addend, so its result is special (the
  // CDNA 3 product overflow can add an infinity: that case takes the whole path)
  constexpr bool kOvf = ID == F_BF16 || ID == F_XF32T || ID == F_XF32R || ID == F_FP32;
  if (!(kOvf && m.prod_ovf)) {
    const uint32_t spec = fspecial_bits<ID, KM>(m, ea, eb, cb);
    if (spec) return resolve_special(m, spec);
  }
  return block_fma_fast<ARCH, ID, KM, UT, AT>(m, ea, eb, cb, true);
}

// One vector set per thread, output rounding RM (1 RNE, 0 toward zero, -1 from the
// model).  A set with an Inf/NaN operand or addend is not evaluated in place: its
// index joins a per-warp queue in shared memory, and each time 32 have gathered the
// warp evaluates them together, so the special-value path runs with every lane busy
// instead of as a divergent branch in nearly every warp.  An exact sum that the
// 64-bit window does not decide joins a second queue of its own, so that the
// full-width evaluator, too, only runs on 32 sets at a time.
constexpr int kStreamThreads = 256;

template <int ARCH, int ID, int KM, bool WIDE, int RM>
__global__ void __launch_bounds__(kStreamThreads) fast_kernel(const __grid_constant__ DevModel m, size_t n,
                                                              const uint8_t *__restrict__ a,
                                                              const uint8_t *__restrict__ b,
                                                              const uint32_t *__restrict__ c,
                                                              uint32_t *__restrict__ d, const W16Consts kc) {
  constexpr int NB = KM * Fmt<ID>::BYTES;
  constexpr int NW = (NB + 3) / 4;
  constexpr bool kWords = Fmt<ID>::BYTES == 2 && Fmt<ID>::XF == 0;   // packed 16-bit decode
  // exact-then-round of FP16 sets on the FP32 pipe first (exact_fp32_sum)
  constexpr bool kFp32Exact = ARCH == MCEMU_ARCH_EXACT && ID == F_FP16;
  // BF16 and truncated XF32 exact-then-round on the FP32 pipe with every term rescaled
  // (exact_scaled)
  constexpr bool kScaled = ARCH == MCEMU_ARCH_EXACT && (ID == F_BF16 || ID == F_XF32T);
  constexpr bool kDefer = ARCH == MCEMU_ARCH_EXACT && (ID == F_FP16 || ID == F_BF16 || ID == F_XF32T ||
                                                       ID == F_XF32R);
  __shared__ size_t queue[kStreamThreads / 32][64];
  __shared__ size_t slow_queue[kDefer ? kStreamThreads / 32 : 1][64];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t below = (1u << lane) - 1u;
  size_t *q = queue[warp], *qs = slow_queue[kDefer ? warp : 0];
  int qn = 0, qsn = 0;                                 // warp-uniform queue lengths
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  // software pipeline: the next vector set's words are loaded while this one is evaluated
  uint32_t na[NW], nb[NW], nc = 0;
  size_t base = (size_t)blockIdx.x * blockDim.x + (size_t)warp * 32;
  if (base + lane < n) {
    load_words<NB>(a + (base + lane) * NB, na);
    load_words<NB>(b + (base + lane) * NB, nb);
    nc = __ldcs(c + base + lane);
  }
  for (; base < n; base += stride) {
    const size_t v = base + lane;
    uint32_t wa[NW], wb[NW];
#pragma unroll
    for (int i = 0; i < NW; i++) { wa[i] = na[i]; wb[i] = nb[i]; }
    const uint32_t cb = nc;
    const size_t vn = v + stride;
    if (vn < n) {
      load_words<NB>(a + vn * NB, na);
      load_words<NB>(b + vn * NB, nb);
      nc = __ldcs(c + vn);
    }
    bool special = false, slow = false;
    if (kFp32Exact && v < n) {
      float p[KM];
#pragma unroll
      for (int i = 0; i < KM / 2; i++) {
        const float2 fa = __half22float2(*reinterpret_cast<const __half2 *>(&wa[i]));
        const float2 fb = __half22float2(*reinterpret_cast<const __half2 *>(&wb[i]));
        p[2 * i] = __fmul_rn(fa.x, fb.x);
        p[2 * i + 1] = __fmul_rn(fa.y, fb.y);
      }
      uint32_t r = 0u;
      slow = exact_fp32_sum<KM>(p, cb, out_rne<RM>(m), m.nan_bits, r) != 0;
      if (!slow) __stcs(d + v, r);
    } else if (v < n) {
      uint32_t sw = (cb & 0x7F800000u) == 0x7F800000u;
#pragma unroll
      for (int i = 0; i < NW; i++) sw |= fspecial_word<ID>(wa[i]) | fspecial_word<ID>(wb[i]);
      special = sw != 0u;
      bool done = special;
      if constexpr (kScaled) {
        // the rescaled products are exact, so a model that turns products of 2^128 or
        // more into Inf (the CDNA 3 rule) keeps the integer path
        if (!done && !m.prod_ovf) {
          uint32_t r = 0u;
          slow = exact_scaled<ID, KM, NW>(wa, wb, cb, out_rne<RM>(m), r) != 0;
          if (!slow) __stcs(d + v, r);
          done = true;
        }
      }
      if (!done) {
        using UT = typename std::conditional<(WIDE || ID == F_FP32), uint64_t, uint32_t>::type;
        using AT = typename std::conditional<(WIDE || ID == F_FP32), int64_t, int32_t>::type;
        uint32_t r;
        if constexpr (kWords) {
          Term<UT> p[KM];
          fterms_w16<ID, KM, UT>(wa, wb, p, kc);
          r = block_fma_terms<ARCH, ID, KM, UT, AT, RM>(m, p, cb, 0u, kDefer ? &slow : nullptr);
        } else {
          uint32_t ea[KM], eb[KM];
#pragma unroll
          for (int l = 0; l < KM; l++) {
            ea[l] = felem<ID>(wa, l);
            eb[l] = felem<ID>(wb, l);
          }
          r = block_fma_fast<ARCH, ID, KM, UT, AT, RM>(m, ea, eb, cb, false, kDefer ? &slow : nullptr);
        }
        if (!slow) __stcs(d + v, r);
      }
    }
    const uint32_t mask = __ballot_sync(0xFFFFFFFFu, special);
    if (mask) {
      if (special) q[qn + __popc(mask & below)] = v;
      qn += __popc(mask);
      if (qn >= 32) {
        __syncwarp();
        const size_t u = q[qn - 32 + lane];
        __stcs(d + u, fast_one<ARCH, ID, KM, WIDE>(m, a, b, c, u));
        qn -= 32;
        __syncwarp();
      }
    }
    if constexpr (kDefer) {
      const uint32_t smask = __ballot_sync(0xFFFFFFFFu, slow);
      if (smask) {
        if (slow) qs[qsn + __popc(smask & below)] = v;
        qsn += __popc(smask);
        if (qsn >= 32) {
          __syncwarp();
          const size_t u = qs[qsn - 32 + lane];
          __stcs(d + u, fast_one<ARCH, ID, KM, WIDE>(m, a, b, c, u));
          qsn -= 32;
          __syncwarp();
        }
      }
    }
  }
  __syncwarp();
  if (lane < qn) {
    const size_t u = q[lane];
    __stcs(d + u, fast_one<ARCH, ID, KM, WIDE>(m, a, b, c, u));
  }
  if (kDefer && lane < qsn) {
    const size_t u = qs[lane];
    __stcs(d + u, fast_one<ARCH, ID, KM, WIDE>(m, a, b, c, u));
  }
}

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
// path.  kSlowQueue: sets with flag 2 are common enough to be batched per warp (else
// they are evaluated in place).
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
  static constexpr bool kSlowQueue = false;
  static __device__ __forceinline__ uint32_t eval(const DevModel &, const GaPairK &k, const uint32_t (&wa)[2],
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

// Exact-then-round on the FP32 pipe: FP16 with exact fp32 products (special values
// from the IEEE sum, in line), BF16 and truncated XF32 with rescaled terms (special
// values queued and resolved from their classes).  A rounding the error bound leaves
// undecided, a subnormal addend or result goes to the integer path, 32 at a time.
template <int ID, int RM> struct ExactPairEv {
  static constexpr bool kSlowQueue = true;
  static __device__ __forceinline__ uint32_t eval(const DevModel &m, const GaPairK &, const uint32_t (&wa)[2],
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

struct QueuedSet {
  uint32_t wa0, wa1, wb0, wb1, c, idx;
};
constexpr int kPairThreads = 256;
constexpr int kPairQueue = 96;    // entries per warp: fewer than 32 left over plus 64 new ones

// Append the flagged sets of this iteration (at most two per lane) to a warp queue and
// resolve it 32 entries at a time; qn is warp-uniform.
template <class Fn>
__device__ __forceinline__ void pair_enqueue(QueuedSet *q, int &qn, bool s0, bool s1, const uint32_t (&wa0)[2],
                                             const uint32_t (&wb0)[2], const uint32_t (&wa1)[2],
                                             const uint32_t (&wb1)[2], uint2 xc, uint32_t p, uint32_t below,
                                             int lane, uint32_t *d32, Fn resolve) {
  const uint32_t m0 = __ballot_sync(0xFFFFFFFFu, s0), m1 = __ballot_sync(0xFFFFFFFFu, s1);
  if (!(m0 | m1)) return;
  if (s0) q[qn + __popc(m0 & below)] = QueuedSet{wa0[0], wa0[1], wb0[0], wb0[1], xc.x, 2 * p};
  qn += __popc(m0);
  if (s1) q[qn + __popc(m1 & below)] = QueuedSet{wa1[0], wa1[1], wb1[0], wb1[1], xc.y, 2 * p + 1};
  qn += __popc(m1);
  while (qn >= 32) {
    __syncwarp();
    const QueuedSet e = q[qn - 32 + lane];
    const uint32_t ua[2] = {e.wa0, e.wa1}, ub[2] = {e.wb0, e.wb1};
    d32[e.idx] = resolve(ua, ub, e.c);
    qn -= 32;
    __syncwarp();
  }
}

template <class Fn>
__device__ __forceinline__ void pair_drain(const QueuedSet *q, int qn, int lane, uint32_t *d32, Fn resolve) {
  __syncwarp();
  if (lane < qn) {
    const QueuedSet e = q[lane];
    const uint32_t ua[2] = {e.wa0, e.wa1}, ub[2] = {e.wb0, e.wb1};
    d32[e.idx] = resolve(ua, ub, e.c);
  }
}

template <class Ev>
__global__ void __launch_bounds__(kPairThreads) pair_kernel(const __grid_constant__ DevModel m, uint32_t npairs,
                                                            const uint4 *__restrict__ a, const uint4 *__restrict__ b,
                                                            const uint2 *__restrict__ c, uint2 *__restrict__ d,
                                                            const GaPairK k) {
  __shared__ QueuedSet queue[kPairThreads / 32][kPairQueue];
  __shared__ QueuedSet slow_queue[Ev::kSlowQueue ? kPairThreads / 32 : 1][kPairQueue];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t below = (1u << lane) - 1u;
  QueuedSet *q = queue[warp], *qs = slow_queue[Ev::kSlowQueue ? warp : 0];
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
      r.x = Ev::eval(m, k, wa0, wb0, xc.x, f0);
      r.y = Ev::eval(m, k, wa1, wb1, xc.y, f1);
      if constexpr (!Ev::kSlowQueue) {
        if (f0 == 2u) r.x = Ev::general(m, wa0, wb0, xc.x);
        if (f1 == 2u) r.y = Ev::general(m, wa1, wb1, xc.y);
      }
      __stcs(d + p, r);
    }
    pair_enqueue(q, qn, (f0 & 1u) != 0u, (f1 & 1u) != 0u, wa0, wb0, wa1, wb1, xc, p, below, lane, d32, special);
    if constexpr (Ev::kSlowQueue)
      pair_enqueue(qs, qsn, f0 == 2u, f1 == 2u, wa0, wb0, wa1, wb1, xc, p, below, lane, d32, general);
  }
  pair_drain(q, qn, lane, d32, special);
  if constexpr (Ev::kSlowQueue) pair_drain(qs, qsn, lane, d32, general);
}

// The pair kernel serves, on 8-byte sets (FP16/BF16 K=4, truncated XF32 K=2) with kept
// subnormals:
//  - early-c global alignment with truncated alignment, F_p >= 23 (P0, P0c >= 0),
//    32-bit sums, no exponent limit and c = 0 discarded;
//  - exact-then-round without the CDNA 3 product-overflow rule;
// with operand pointers 16-byte aligned and c, d 8-byte aligned.
static bool pair_ok(const DevModel &m, int id, const void *a, const void *b, const uint32_t *c, const uint32_t *d) {
  if (!((id == F_FP16 || id == F_BF16) && m.k == 4) && !(id == F_XF32T && m.k == 2)) return false;
  if (m.acc16 || m.sub_out_flush || m.fa.sub_keep == 0u || m.c_sub_keep == 0u || m.prod_ovf) return false;
  if (m.arch == MCEMU_ARCH_GA_EARLY) {
    if (m.align_rd || m.wide || m.emin_lim != kNegE || m.c_zero_exp != kNegE || m.R0 != 0 || m.R0c != 0) return false;
  } else if (m.arch != MCEMU_ARCH_EXACT) {
    return false;
  }
  return ((uintptr_t)a % 16) == 0 && ((uintptr_t)b % 16) == 0 && ((uintptr_t)c % 8) == 0 && ((uintptr_t)d % 8) == 0;
}

static int grid_for(size_t n, const void *kernel);

static int launch_pair(const DevModel &m, int id, size_t n, const void *a, const void *b, const uint32_t *c,
                       uint32_t *d, cudaStream_t s) {
  const int mb = id == F_BF16 ? 7 : 10;            // kE: the 16-bit formats' exponent extraction
  const GaPairK k{m.p0mul, m.p0cmul, -2 * m.fa.bias - m.F, 1u, 2u, 1u << 16, 1u << (16 - mb), 1u << 9, 1u << 23, -1, -2};
  const size_t np = n / 2;
  auto run = [&](auto kern) {
    const int grid = grid_for(np, (const void *)kern);
    kern<<<grid, kPairThreads, 0, s>>>(m, (uint32_t)np, (const uint4 *)a, (const uint4 *)b, (const uint2 *)c,
                                       (uint2 *)d, k);
    return cudaGetLastError() == cudaSuccess ? MCEMU_OK : MCEMU_ERR_CUDA;
  };
  auto by_rm = [&](auto id_tag, auto exact_tag) {
    constexpr int ID = decltype(id_tag)::value;
    if constexpr (decltype(exact_tag)::value)
      return m.rne ? run(pair_kernel<ExactPairEv<ID, 1>>) : run(pair_kernel<ExactPairEv<ID, 0>>);
    else
      return m.rne ? run(pair_kernel<GaPairEv<ID, 1>>) : run(pair_kernel<GaPairEv<ID, 0>>);
  };
  using T = std::true_type;
  using Fl = std::false_type;
  const bool ex = m.arch == MCEMU_ARCH_EXACT;
  if (id == F_BF16) return ex ? by_rm(std::integral_constant<int, F_BF16>{}, T{}) : by_rm(std::integral_constant<int, F_BF16>{}, Fl{});
  if (id == F_XF32T) return ex ? by_rm(std::integral_constant<int, F_XF32T>{}, T{}) : by_rm(std::integral_constant<int, F_XF32T>{}, Fl{});
  return ex ? by_rm(std::integral_constant<int, F_FP16>{}, T{}) : by_rm(std::integral_constant<int, F_FP16>{}, Fl{});
}

// Any model: element loads, the out-of-line evaluator (the fallback for
// combinations without a specialised kernel).
__global__ void __launch_bounds__(256) block_generic_kernel(const __grid_constant__ DevModel m, size_t n, int eb,
                                                            const uint8_t *__restrict__ a,
                                                            const uint8_t *__restrict__ b,
                                                            const uint32_t *__restrict__ c,
                                                            uint32_t *__restrict__ d) {
  const int k = m.k;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t v = (size_t)blockIdx.x * blockDim.x + threadIdx.x; v < n; v += stride) {
    uint32_t ea[32], ebv[32];
    for (int l = 0; l < k; l++) {
      size_t idx = v * k + l;
      if (eb == 1) { ea[l] = a[idx]; ebv[l] = b[idx]; }
      else if (eb == 2) { ea[l] = reinterpret_cast<const uint16_t *>(a)[idx]; ebv[l] = reinterpret_cast<const uint16_t *>(b)[idx]; }
      else { ea[l] = reinterpret_cast<const uint32_t *>(a)[idx]; ebv[l] = reinterpret_cast<const uint32_t *>(b)[idx]; }
    }
    d[v] = block_eval_generic(m, ea, ebv, k, c[v]);
  }
}

// ---------------------------------------------------------------------------
// dispatch: specialised kernels for the block sizes and formats of the
// workloads and the hardware presets; everything else takes the generic kernel
// ---------------------------------------------------------------------------
static int grid_for(size_t n, const void *kernel) {
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, 0);
  if (per_sm < 1) per_sm = 1;
  size_t want = (n + 255) / 256;
  size_t full = (size_t)sms * per_sm;              // one wave of resident blocks
  if (want > full) want = full;
  return (int)(want < 1 ? 1 : want);
}

typedef void (*FpKernel)(const DevModel, size_t, const uint8_t *, const uint8_t *, const uint32_t *, uint32_t *,
                         const W16Consts);

struct Special {
  int arch, id, km, wide, rm;                          // rm: output rounding, -1 = any
  FpKernel fn;
};

#define SPEC(A, F, K, W) {A, F, K, W, -1, fast_kernel<A, F, K, W, -1>}
#define SPEC_RM(A, F, K) {A, F, K, false, 0, fast_kernel<A, F, K, false, 0>}, \
                         {A, F, K, false, 1, fast_kernel<A, F, K, false, 1>}
static const Special kSpecial[] = {
    // early-c global alignment: the randomized-workload truncate / RNE models
    SPEC_RM(MCEMU_ARCH_GA_EARLY, F_FP16, 4), SPEC_RM(MCEMU_ARCH_GA_EARLY, F_BF16, 4),
    SPEC_RM(MCEMU_ARCH_GA_EARLY, F_XF32T, 2), SPEC(MCEMU_ARCH_GA_EARLY, F_E4M3, 8, false),
    SPEC(MCEMU_ARCH_GA_EARLY, F_E5M2, 8, false),
    // exact-then-round on the same vector sets
    SPEC_RM(MCEMU_ARCH_EXACT, F_FP16, 4), SPEC_RM(MCEMU_ARCH_EXACT, F_BF16, 4),
    SPEC_RM(MCEMU_ARCH_EXACT, F_XF32T, 2), SPEC(MCEMU_ARCH_EXACT, F_E4M3, 8, false),
    SPEC(MCEMU_ARCH_EXACT, F_E5M2, 8, false),
    // CDNA 3: Algorithm 1 (fp16/bf16 N_FMA 8, tf19 4), Algorithm 2 (binary8 FNUZ, 16)
    SPEC(MCEMU_ARCH_GA_LATE, F_FP16, 8, false), SPEC(MCEMU_ARCH_GA_LATE, F_BF16, 8, false),
    SPEC(MCEMU_ARCH_GA_LATE, F_XF32T, 4, false), SPEC(MCEMU_ARCH_ODD_EVEN, F_E4M3Z, 16, false),
    SPEC(MCEMU_ARCH_ODD_EVEN, F_E5M2Z, 16, false),
    // Table 3 NVIDIA-like presets
    SPEC(MCEMU_ARCH_GA_EARLY, F_FP16, 16, true), SPEC(MCEMU_ARCH_GA_EARLY, F_FP16, 8, false),
    SPEC(MCEMU_ARCH_GA_EARLY, F_BF16, 8, false), SPEC(MCEMU_ARCH_GA_EARLY, F_XF32T, 4, false),
};
#undef SPEC
#undef SPEC_RM

// compile-time format of a model whose operands share one format, else -1
static int fmt_id(const DevModel &m) {
  const FmtDev &a = m.fa, &b = m.fb;
  if (a.is_int || a.mbits != b.mbits || a.bias != b.bias || a.xf32 != b.xf32 || a.sw_fnuz != b.sw_fnuz ||
      a.emask != b.emask)
    return -1;
  if (a.xf32) return a.xf32 == 2 ? F_XF32R : F_XF32T;
  if (a.mbits == 23) return F_FP32;
  if (a.mbits == 10) return F_FP16;
  if (a.mbits == 7) return F_BF16;
  if (a.mbits == 3) return a.sw_fnuz ? F_E4M3Z : F_E4M3;
  if (a.mbits == 2) return a.sw_fnuz ? F_E5M2Z : F_E5M2;
  return -1;
}

int launch_block_fma(const DevModel &m, size_t n, const void *a, const void *b, const uint32_t *c,
                     uint32_t *d, void *stream) {
  if (n == 0) return MCEMU_OK;
  cudaStream_t s = (cudaStream_t)stream;
  if (m.fa.is_int && (m.k == 16 || m.k == 8 || m.k == 32 || m.k == 4)) {
    auto run = [&](auto kern) {
      int grid = grid_for(n, (const void *)kern);
      kern<<<grid, 256, 0, s>>>(m, n, (const uint8_t *)a, (const uint8_t *)b, c, d);
      return cudaGetLastError() == cudaSuccess ? MCEMU_OK : MCEMU_ERR_CUDA;
    };
    if (m.k == 4) return run(block_int_kernel<4>);
    if (m.k == 8) return run(block_int_kernel<8>);
    if (m.k == 16) return run(block_int_kernel<16>);
    return run(block_int_kernel<32>);
  }
  const int id = fmt_id(m);
  if (id >= 0 && f8_stream_ok(m, id)) return launch_block_fma_f8(m, id, n, a, b, c, d, stream);
  if (id >= 0 && n >= 2 && n / 2 < (1u << 31) && pair_ok(m, id, a, b, c, d)) {
    int st = launch_pair(m, id, n, a, b, c, d, s);
    if (st != MCEMU_OK || n % 2 == 0) return st;
    const size_t t = n - 1, vb = 8;                    // the odd last set: the one-set kernel
    return launch_block_fma(m, 1, (const uint8_t *)a + t * vb, (const uint8_t *)b + t * vb, c + t, d + t, stream);
  }
  // the specialised kernels assume kept subnormals (the fp32 special-value shortcut)
  if (id >= 0 && !m.acc16 && m.arch != MCEMU_ARCH_PAIRWISE && m.fa.sub_keep != 0u && m.c_sub_keep != 0u) {
    for (const Special &sp : kSpecial) {
      if (sp.arch != m.arch || sp.id != id || sp.km != m.k) continue;
      if (m.arch != MCEMU_ARCH_EXACT && sp.wide != (m.wide != 0)) continue;
      if (sp.rm >= 0 && sp.rm != (m.rne != 0 ? 1 : 0)) continue;
      int grid = grid_for(n, (const void *)sp.fn);
      const uint32_t mb = id == F_FP16 ? 10u : 7u;                  // fterms_w16 (FP16, BF16)
      const W16Consts kc{1u, 2u, 1u << 16, 1u << (32 - mb), (1u << 22) - 1u, 1u << 10};
      sp.fn<<<grid, 256, 0, s>>>(m, n, (const uint8_t *)a, (const uint8_t *)b, c, d, kc);
      return cudaGetLastError() == cudaSuccess ? MCEMU_OK : MCEMU_ERR_CUDA;
    }
  }
  const int eb = m.fa.is_int ? 1 : (int)(m.fa.sshift + 1) / 8;
  int grid = grid_for(n, (const void *)block_generic_kernel);
  block_generic_kernel<<<grid, 256, 0, s>>>(m, n, eb, (const uint8_t *)a, (const uint8_t *)b, c, d);
  return cudaGetLastError() == cudaSuccess ? MCEMU_OK : MCEMU_ERR_CUDA;
}

}  // namespace mcemu

// core.cuh -- device side of the emulator: input decoding, the multi-term
// adder architectures of "Accurate Models of AMD Matrix Cores" and the
// rounding of their integer results to fp32.  Shared by every kernel.
//
// Vocabulary (paper notation):  p_l = a_l * b_l is kept as an integer
// significand product U_l = S_a * S_b with fraction bits m_a + m_b and the
// denormalised exponent e_l = E_a + E_b (Sec. 4.3.1); c has significand S_c
// (23 fraction bits) and exponent e_c; e_max is the maximum exponent that the
// terms are aligned to; F_p the fraction bits kept after alignment.
#pragma once
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "model.h"

namespace mcemu {

// ---------------------------------------------------------------------------
// small integer helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t shr32(uint32_t x, int32_t s) {   // s >= 0, 0 when s >= 32
  return __funnelshift_rc(x, 0u, (uint32_t)s);
}
__device__ __forceinline__ uint64_t shr64(uint64_t x, int32_t s) {   // s >= 0
  return s >= 64 ? 0ull : (x >> s);
}
__device__ __forceinline__ int64_t sar64(int64_t x, int32_t s) {     // floor(x / 2^s), s >= 0
  return x >> (s > 63 ? 63 : s);
}
__device__ __forceinline__ uint32_t shl_clamp(uint32_t x, uint32_t s) {   // 0 once s >= 32
  uint32_t r;
  asm("shl.b32 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(s));
  return r;
}
__device__ __forceinline__ int32_t sar32(int32_t x, int32_t s) {
  return x >> (s > 31 ? 31 : s);
}

// ---------------------------------------------------------------------------
// decoding
// ---------------------------------------------------------------------------
// XF32: an fp32 container whose mantissa is reduced to 10 bits (Sec. 4.3.3).
__device__ __forceinline__ uint32_t xf32_reduce(uint32_t bits, uint32_t mode) {
  if (mode == 1u) return bits & 0xFFFFE000u;
  return (bits + 0xFFFu + ((bits >> 13) & 1u)) & 0xFFFFE000u;   // RNE, may carry into Inf
}

// Finite decode: value = (-1)^neg * S * 2^(E - m_eff).  Zero (and flushed
// subnormals) give S = 0.  Inf/NaN decode to garbage and are caught apart.
__device__ __forceinline__ void decode(const FmtDev &f, uint32_t bits, uint32_t &S, int32_t &E,
                                       uint32_t &neg) {
  if (f.xf32) bits = xf32_reduce(bits, f.xf32);
  uint32_t ef = (bits >> f.mbits) & f.emask;
  uint32_t mf = bits & ((1u << f.mbits) - 1u);
  neg = (bits >> f.sshift) & 1u;
  S = (ef ? (mf | (1u << f.mbits)) : (mf & f.sub_keep)) >> f.sig_rshift;
  E = (int32_t)(ef ? ef : 1u) - f.bias;
}

// Special-value class of one element: 0 finite, 1 Inf, 2 NaN (sign apart).
__device__ __forceinline__ uint32_t classify(const FmtDev &f, uint32_t bits) {
  uint32_t ef = (bits >> f.mbits) & f.emask;
  uint32_t mf = bits & ((1u << f.mbits) - 1u);
  if ((bits & f.nan_mask) == f.nan_pat) return 2u;
  if (ef == f.top_special) {
    if (mf) return 2u;
    return 1u;
  }
  if (f.xf32 == 2u) {               // RNE reduction can round the largest finites to Inf
    uint32_t r = xf32_reduce(bits, 2u);
    if (((r >> 23) & 0xFFu) == 0xFFu) return 1u;
  }
  return 0u;
}

__device__ __forceinline__ bool is_zero_elem(const FmtDev &f, uint32_t bits) {
  uint32_t S; int32_t E; uint32_t neg;
  decode(f, bits, S, E, neg);
  return S == 0u && classify(f, bits) == 0u;
}

// SWAR test of a 32-bit word of packed elements: nonzero when some element is
// Inf/NaN (the exponent field all ones carries into the sign position), or, for
// FNUZ, some byte is 0x80.
__device__ __forceinline__ uint32_t special_word(const FmtDev &f, uint32_t w) {
  uint32_t s = ((w & f.sw_mask) + f.sw_add) & f.sw_hi;
  if (f.sw_fnuz) {
    uint32_t x = w ^ 0x80808080u;
    s |= (x - 0x01010101u) & ~x & 0x80808080u;
  }
  if (f.xf32 == 2u) s |= ((xf32_reduce(w, 2u) & 0x7F800000u) + 0x00800000u) & 0x80000000u;
  return s;
}

// fp32 addend c (always binary32 bits).
__device__ __forceinline__ void decode_c(const DevModel &m, uint32_t bits, uint32_t &S, int32_t &E,
                                         uint32_t &neg) {
  uint32_t ef = (bits >> 23) & 0xFFu;
  uint32_t mf = bits & 0x7FFFFFu;
  neg = bits >> 31;
  S = ef ? (mf | 0x800000u) : (mf & m.c_sub_keep);
  E = (int32_t)(ef ? ef : 1u) - 127;
}

// ---------------------------------------------------------------------------
// special values: every model gives NaN for a NaN input, Inf*0 or Inf-Inf, and
// the signed Inf otherwise (Secs. 4.1-4.3).  Bits: 1 NaN, 2 +Inf, 4 -Inf.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t product_special(const DevModel &m, uint32_t ab, uint32_t bb) {
  uint32_t ca = classify(m.fa, ab), cb = classify(m.fb, bb);
  if (ca == 2u || cb == 2u) return 1u;
  if (ca == 0u && cb == 0u) return 0u;
  bool za = (ca == 0u) && is_zero_elem(m.fa, ab);
  bool zb = (cb == 0u) && is_zero_elem(m.fb, bb);
  if (za || zb) return 1u;                                    // Inf * 0
  uint32_t neg = ((ab >> m.fa.sshift) ^ (bb >> m.fb.sshift)) & 1u;
  return neg ? 4u : 2u;
}

__device__ __forceinline__ uint32_t c_special(uint32_t cb) {
  if ((cb & 0x7F800000u) != 0x7F800000u) return 0u;
  if (cb & 0x7FFFFFu) return 1u;
  return (cb >> 31) ? 4u : 2u;
}

__device__ __forceinline__ uint32_t resolve_special(const DevModel &m, uint32_t s) {
  if ((s & 1u) || (s & 6u) == 6u) return m.nan_bits;
  return (s & 2u) ? 0x7F800000u : 0xFF800000u;
}

// ---------------------------------------------------------------------------
// rounding of an exact (or sticky-carrying) magnitude to fp32
// value = (-1)^neg * (M + f) * 2^lsb with f in (0,1) when sticky, else f = 0.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t overflow_bits(int rne) {
  return rne ? 0x7F800000u : 0x7F7FFFFFu;
}

__device__ __forceinline__ uint32_t round_pack(uint64_t M, int32_t lsb, uint32_t neg, bool sticky,
                                               int rne, int flush) {
  // M > 0, M < 2^62.  Branch-free: shift right by rr = clamp(r, 0, 62) or left by
  // ls = clamp(-r, 0, 23), with r the number of bits of M below the fp32 grid.
  const int32_t p = 63 - __clzll((long long)M);
  const int32_t E = lsb + p;
  const int32_t Ec = max(E, -126);
  const int32_t r = Ec - 23 - lsb;
  const int32_t rr = min(max(r, 0), 62), ls = min(max(-r, 0), 31);
  const uint64_t q = (M >> rr) << ls;
  const uint64_t rem = M & ((1ull << rr) - 1ull);
  const uint64_t half = (1ull << rr) >> 1;
  // r > 62: the value is below half of the grid step (M < 2^62), so it rounds down
  const bool up = rne && rr > 0 && r <= 62 && (rem > half || (rem == half && (sticky || (q & 1ull))));
  uint32_t bits = ((uint32_t)(Ec + 126) << 23) + (uint32_t)q + (up ? 1u : 0u);
  bits = (Ec > 127 || bits >= 0x7F800000u) ? overflow_bits(rne) : bits;
  bits = (flush && bits < 0x00800000u) ? 0u : bits;
  return bits | (neg << 31);
}

// 32-bit fast path: M < 2^31, no sticky.
__device__ __forceinline__ uint32_t round_pack32(uint32_t M, int32_t lsb, uint32_t neg, int rne,
                                                 int flush) {
  const int32_t p = 31 - __clz((int)M);
  const int32_t E = lsb + p;
  const int32_t Ec = max(E, -126);
  const int32_t r = Ec - 23 - lsb;
  const uint32_t rr = (uint32_t)min(max(r, 0), 31), ls = (uint32_t)min(max(-r, 0), 31);
  const uint32_t q = (M >> rr) << ls;
  const uint32_t rem = M & ((1u << rr) - 1u);
  const uint32_t half = (1u << rr) >> 1;
  const bool up = rne && rr > 0 && r <= 31 && (rem > half || (rem == half && (q & 1u)));
  uint32_t bits = ((uint32_t)(Ec + 126) << 23) + q + (up ? 1u : 0u);
  bits = (Ec > 127 || bits >= 0x7F800000u) ? overflow_bits(rne) : bits;
  bits = (flush && bits < 0x00800000u) ? 0u : bits;
  return bits | (neg << 31);
}

// Hardware rounding of an integer significand: value = S * 2^k.  The int->fp32
// conversion rounds S to 24 bits exactly as the model's RNE or RTZ does, and
// scaling by powers of two is exact while the result stays normal; an overflow
// gives Inf under RN and the largest finite under RZ, as the model does.  An
// exact value below 2^-126 would be rounded twice: first to 24 bits, which can
// carry it up to the subnormal tie 2^-126 - 2^-150 or onto 2^-126 itself, then
// onto the subnormal grid.  Rounding is monotonic and 2^-126 is on both grids,
// so such a value always lands at or below 2^-126, and a result above 2^-126
// in magnitude proves the exact value was normal.  A result of magnitude 2^-126
// or less (zero, subnormal, or 2^-126 itself) returns false and the caller takes
// the integer path.
__device__ __forceinline__ bool hw_normal(uint32_t bits) { return (bits & 0x7FFFFFFFu) > 0x00800000u; }

__device__ __forceinline__ bool hw_scale(float x, int32_t k, int rne, uint32_t &bits) {
  const int32_t k1 = min(max(k, -96), 96);           // |x| in [1, 2^63): x*2^k1 stays normal
  const int32_t k2 = min(k - k1, 127);                // beyond 127 the result overflows anyway
  if (k2 < -126) return false;
  const float s1 = __uint_as_float((uint32_t)(k1 + 127) << 23);
  const float s2 = __uint_as_float((uint32_t)(k2 + 127) << 23);
  const float y = rne ? __fmul_rn(__fmul_rn(x, s1), s2) : __fmul_rz(__fmul_rz(x, s1), s2);
  bits = __float_as_uint(y);
  return hw_normal(bits);
}
__device__ __forceinline__ bool hw_round32(int32_t S, int32_t k, int rne, uint32_t &bits) {
  return hw_scale(rne ? __int2float_rn(S) : __int2float_rz(S), k, rne, bits);
}
__device__ __forceinline__ bool hw_round64(int64_t S, int32_t k, int rne, uint32_t &bits) {
  return hw_scale(rne ? __ll2float_rn(S) : __ll2float_rz(S), k, rne, bits);
}
// ---------------------------------------------------------------------------
// terms of eq. (1)
// ---------------------------------------------------------------------------
template <class UT>
struct Term {
  UT U;          // |S_a * S_b|
  int32_t e;     // E_a + E_b, kNegE for a zero product
  uint32_t neg;  // 0 / 1
};

template <class UT>
__device__ __forceinline__ Term<UT> make_term(const DevModel &m, uint32_t ab, uint32_t bb) {
  uint32_t Sa, Sb, na, nb;
  int32_t Ea, Eb;
  decode(m.fa, ab, Sa, Ea, na);
  decode(m.fb, bb, Sb, Eb, nb);
  Term<UT> t;
  t.U = (UT)Sa * (UT)Sb;
  t.e = t.U ? Ea + Eb : kNegE;
  t.neg = na ^ nb;
  return t;
}

// CDNA3: |p| >= 2^128 becomes +-Inf (Sec. 4.3.2).  Returns special bits.
template <class UT>
__device__ __forceinline__ uint32_t product_overflow(const DevModel &m, const Term<UT> &t) {
  // |p| = U * 2^(e - mab) >= 2^128  <=>  msb(U) + e - mab >= 128
  if (!t.U) return 0u;
  int32_t msb = (sizeof(UT) == 8) ? 63 - __clzll((long long)t.U) : 31 - __clz((int)t.U);
  if (msb + t.e - m.mab >= 128) return t.neg ? 4u : 2u;
  return 0u;
}

// zero result: negative only when every product is a negative zero and c is -0
template <int K, class UT>
__device__ __forceinline__ uint32_t zero_result(const Term<UT> (&p)[K], int nt, uint32_t cS,
                                                uint32_t cneg) {
  bool all_neg = (cS == 0u) && cneg;
#pragma unroll
  for (int l = 0; l < K; l++)
    if (l < nt) all_neg = all_neg && (p[l].U == 0) && p[l].neg;
  return all_neg ? 0x80000000u : 0u;
}

// ---------------------------------------------------------------------------
// aligned, truncated term: RZ or RD of +-U * 2^(F_p - shift) on the integer grid
// ---------------------------------------------------------------------------
template <class UT, class AT>
__device__ __forceinline__ AT align_term(UT Ushift, uint32_t neg, int32_t sh, int rd) {
  // Ushift = U << P0 (< 2^(width-1)); sh >= 0 is the right shift to the grid.
  if (sizeof(AT) == 4) {
    if (rd) {
      int32_t v = neg ? -(int32_t)Ushift : (int32_t)Ushift;
      return (AT)sar32(v, sh);
    }
    uint32_t t = shr32((uint32_t)Ushift, sh);
    return (AT)(neg ? -(int32_t)t : (int32_t)t);
  } else {
    if (rd) {
      int64_t v = neg ? -(int64_t)Ushift : (int64_t)Ushift;
      return (AT)sar64(v, sh);
    }
    uint64_t t = shr64((uint64_t)Ushift, sh);
    return (AT)(neg ? -(int64_t)t : (int64_t)t);
  }
}

// RM: the output rounding fixed at compile time (1 = RNE, 0 = toward zero), or -1 to
// read it from the model
template <int RM>
__device__ __forceinline__ int out_rne(const DevModel &m) { return RM >= 0 ? RM : m.rne; }

template <class AT, int RM = -1>
__device__ __forceinline__ uint32_t pack_sum(AT S, int32_t lsb, const DevModel &m) {
  const int rne = out_rne<RM>(m);
  if (!m.sub_out_flush) {
    uint32_t bits;
    const bool ok = (sizeof(AT) == 4) ? hw_round32((int32_t)S, lsb, rne, bits)
                                      : hw_round64((int64_t)S, lsb, rne, bits);
    if (ok) return bits;
  }
  uint32_t neg = S < 0 ? 1u : 0u;
  if (sizeof(AT) == 4) {
    uint32_t M = neg ? (uint32_t)(-(int32_t)S) : (uint32_t)S;
    return round_pack32(M, lsb, neg, rne, m.sub_out_flush);
  }
  uint64_t M = neg ? (uint64_t)(-(int64_t)S) : (uint64_t)S;
  return round_pack(M, lsb, neg, false, rne, m.sub_out_flush);
}

// ---------------------------------------------------------------------------
// GA_EARLY: global alignment with c aligned together with the products
// (Table 3, early c; e_{c=0} and e_min^lim as configured).
// ---------------------------------------------------------------------------
template <int K, class UT, class AT, int RM = -1>
__device__ __forceinline__ uint32_t arch_ga_early(const DevModel &m, const Term<UT> (&p)[K], int nt,
                                                  uint32_t cS, int32_t cE, uint32_t cneg) {
  int32_t emax = m.emin_lim;
#pragma unroll
  for (int l = 0; l < K; l++)
    if (l < nt) emax = max(emax, p[l].e);
  int32_t ec = cS ? cE : m.c_zero_exp;
  emax = max(emax, ec);
  AT S = 0;
  const int32_t base = emax + m.R0;
  if (sizeof(AT) == 4 && !m.align_rd) {
    // truncation with 32-bit sums: the pre-shift and the sign as multiplies (FMA pipe),
    // one funnel shift per term on the ALU pipe
#pragma unroll
    for (int l = 0; l < K; l++)
      if (l < nt) {
        const uint32_t t = shr32((uint32_t)p[l].U * m.p0mul, base - p[l].e);
        S += (AT)((int32_t)t * (1 - 2 * (int32_t)p[l].neg));
      }
    if (cS) S += (AT)((int32_t)shr32(cS * m.p0cmul, emax + m.R0c - cE) * (1 - 2 * (int32_t)cneg));
  } else {
#pragma unroll
    for (int l = 0; l < K; l++)
      if (l < nt) S += align_term<UT, AT>(p[l].U << m.P0, p[l].neg, base - p[l].e, m.align_rd);
    if (cS) S += align_term<UT, AT>((UT)cS << m.P0c, cneg, emax + m.R0c - cE, m.align_rd);
  }
  if (S == 0) return zero_result<K, UT>(p, nt, cS, cneg);
  return pack_sum<AT, RM>(S, emax - m.F, m);
}

// ---------------------------------------------------------------------------
// Late c merge: lines 5-15 of Algorithm 1 (lines 9-20 of Algorithm 2, which
// also drops a c shifted by more than 25 places: zero_cut).  Sp is the aligned
// product sum in units of 2^(emax - F_p).
// ---------------------------------------------------------------------------
template <int K, class UT, class AT>
__device__ __forceinline__ uint32_t late_c_merge(const DevModel &m, AT Sp, bool have_p, int32_t emax,
                                                 const Term<UT> (&p)[K], int nt, uint32_t cS,
                                                 int32_t cE, uint32_t cneg, bool zero_cut) {
  int32_t ec = cS ? cE : m.c_zero_exp;      // line 5: e_c = -126 if c = 0
  bool have_c = ec > kNegE / 2;
  if (!have_p && !have_c) return zero_result<K, UT>(p, nt, cS, cneg);
  if (have_p && (!have_c || emax >= ec)) {
    // line 7: shift s_c right by e_max - e_c, RD to c_frac fraction bits (= F_p)
    int64_t sc = 0;
    if (cS && !(zero_cut && emax - ec > 25)) {
      int64_t v = cneg ? -(int64_t)cS : (int64_t)cS;
      int32_t sh = emax - ec + 23 - m.c_frac;
      sc = sh >= 0 ? sar64(v, sh) : v * ((int64_t)1 << (-sh));
    }
    int64_t Sacc = (int64_t)Sp + sc;        // line 8
    if (Sacc == 0) return zero_result<K, UT>(p, nt, cS, cneg);
    if (!m.sub_out_flush) {
      uint32_t bits;
      if (hw_round64(Sacc, emax - m.F, m.rne, bits)) return bits;       // line 15
    }
    uint32_t neg = Sacc < 0 ? 1u : 0u;
    uint64_t M = neg ? (uint64_t)(-Sacc) : (uint64_t)Sacc;
    return round_pack(M, emax - m.F, neg, false, m.rne, m.sub_out_flush);   // line 15
  }
  // line 10: shift S_p right by e_c - e_max, RD to psum_frac fraction bits
  int64_t Sp2 = 0;
  if (have_p) {
    int32_t sh = ec - emax - (m.psum_frac - m.F);
    Sp2 = sh >= 0 ? sar64((int64_t)Sp, sh) : (int64_t)Sp * ((int64_t)1 << (-sh));
  }
  // line 11: S_acc = S'_p + s_c on the 2^(e_c - psum_frac) grid
  int64_t vc = cneg ? -(int64_t)cS : (int64_t)cS;
  int64_t Sacc = Sp2 + vc * ((int64_t)1 << (m.psum_frac - 23));
  if (Sacc == 0) return zero_result<K, UT>(p, nt, cS, cneg);
  uint32_t neg = Sacc < 0 ? 1u : 0u;
  uint64_t M = neg ? (uint64_t)(-Sacc) : (uint64_t)Sacc;
  int32_t lsb = ec - m.psum_frac;
  // line 12: normalise, exponent floored at -126 (subnormal-aware)
  int32_t E = 63 - __clzll((long long)M) + lsb;
  if (E < -126) E = -126;
  // line 13: RD to post_norm_frac fraction bits of the normalised value
  int32_t r = E - m.post_norm_frac - lsb;
  if (r > 0) {
    M = neg ? ((M + ((1ull << r) - 1ull)) >> r) : (M >> r);   // floor of the signed value
    lsb += r;
  }
  if (!m.sub_out_flush) {
    uint32_t bits;
    if (hw_round64(neg ? -(int64_t)M : (int64_t)M, lsb, m.rne, bits)) return bits;   // line 15
  }
  return round_pack(M, lsb, neg, false, m.rne, m.sub_out_flush);   // line 15
}

// Algorithm 1 (CDNA 3 fp16/bf16/tf19): lines 3-4 then the late-c merge.
template <int K, class UT, class AT>
__device__ __forceinline__ uint32_t arch_ga_late(const DevModel &m, const Term<UT> (&p)[K], int nt,
                                                 uint32_t cS, int32_t cE, uint32_t cneg) {
  int32_t emax = kNegE;                     // line 3
#pragma unroll
  for (int l = 0; l < K; l++)
    if (l < nt) emax = max(emax, p[l].e);
  bool have_p = emax > kNegE / 2;
  AT Sp = 0;                                // line 4
  const int32_t base = emax + m.R0;
#pragma unroll
  for (int l = 0; l < K; l++)
    if (l < nt) Sp += align_term<UT, AT>(p[l].U << m.P0, p[l].neg, base - p[l].e, m.align_rd);
  return late_c_merge<K, UT, AT>(m, Sp, have_p, emax, p, nt, cS, cE, cneg, false);
}

// Algorithm 2 (CDNA 3 binary8): odd (p_1, p_3, ...) and even (p_2, p_4, ...)
// products aligned to their own maxima (lines 3-5), shifted to the common e_max
// with RD (lines 6-8), then the late-c merge with the 25-place cut.
template <int K, class UT, class AT>
__device__ __forceinline__ uint32_t arch_odd_even(const DevModel &m, const Term<UT> (&p)[K], int nt,
                                                  uint32_t cS, int32_t cE, uint32_t cneg) {
  int32_t em0 = kNegE, em1 = kNegE;
#pragma unroll
  for (int l = 0; l < K; l++)
    if (l < nt) {
      if ((l & 1) == 0) em0 = max(em0, p[l].e);
      else em1 = max(em1, p[l].e);
    }
  AT S0 = 0, S1 = 0;
#pragma unroll
  for (int l = 0; l < K; l++)
    if (l < nt) {
      if ((l & 1) == 0) S0 += align_term<UT, AT>(p[l].U << m.P0, p[l].neg, em0 + m.R0 - p[l].e, m.align_rd);
      else S1 += align_term<UT, AT>(p[l].U << m.P0, p[l].neg, em1 + m.R0 - p[l].e, m.align_rd);
    }
  int32_t emax = max(em0, em1);
  bool have_p = emax > kNegE / 2;
  AT Sp = 0;
  if (have_p) {
    if (em0 > kNegE / 2) Sp += (AT)sar64((int64_t)S0, emax - em0);
    if (em1 > kNegE / 2) Sp += (AT)sar64((int64_t)S1, emax - em1);
  }
  return late_c_merge<K, UT, AT>(m, Sp, have_p, emax, p, nt, cS, cE, cneg, true);
}

// ---------------------------------------------------------------------------
// EXACT: correct rounding of the exact sum (CDNA 1).  A 128-bit window anchored
// at the largest term holds every term that fits; terms reaching below it are
// floored into it and counted.  The true value then lies in (W, W + nb) units
// of the window LSB; when both ends round alike that is the answer, otherwise
// a full-width exact accumulation decides (rare).
// ---------------------------------------------------------------------------
typedef __int128 i128;
typedef unsigned __int128 u128;

__device__ __forceinline__ uint32_t round_pack128(i128 W, int32_t L, bool sticky, const DevModel &m) {
  uint32_t neg = W < 0 ? 1u : 0u;
  u128 Mag = neg ? (sticky ? (u128)(~W) : (u128)(-W)) : (u128)W;
  uint64_t hi = (uint64_t)(Mag >> 64), lo = (uint64_t)Mag;
  int32_t p = hi ? 127 - __clzll((long long)hi) : (lo ? 63 - __clzll((long long)lo) : -1);
  if (p < 0) return 0u;                     // not reached: the window sum is never empty
  int32_t s = p > 61 ? p - 61 : 0;
  uint64_t M = (uint64_t)(Mag >> s);
  bool st = sticky || (s > 0 && (Mag & (((u128)1 << s) - 1)) != 0);
  if (!m.sub_out_flush && (p - s) >= 26) {
    // bit 0 of M lies at least two places below the rounding point, so it can carry
    // the sticky bit into the hardware conversion
    const uint64_t Ms = M | (st ? 1ull : 0ull);
    uint32_t bits;
    if (hw_round64(neg ? -(int64_t)Ms : (int64_t)Ms, L + s, m.rne, bits)) return bits;
  }
  return round_pack(M, L + s, neg, st, m.rne, m.sub_out_flush);
}

// full-width exact sum: 32-bit digits in signed 64-bit slots covering 2^-320 .. 2^320
static __device__ __noinline__ uint32_t exact_slow(const DevModel &m, const int64_t *V, const int32_t *lsb, int nterm) {
  constexpr int kBase = -320, kDig = 20;
  int64_t acc[kDig];
#pragma unroll
  for (int i = 0; i < kDig; i++) acc[i] = 0;
  for (int t = 0; t < nterm; t++) {
    if (V[t] == 0) continue;
    // split |V| < 2^49 into 24-bit pieces so that piece << 31 fits a slot
    int64_t v = V[t];
    int64_t vlo = v & 0xFFFFFF;             // two's complement: v = vhi * 2^24 + vlo
    int64_t vhi = v >> 24;
    for (int h = 0; h < 2; h++) {
      int64_t piece = h ? vhi : vlo;
      if (!piece) continue;
      int32_t pos = lsb[t] + 24 * h - kBase;
      acc[pos >> 5] += piece * ((int64_t)1 << (pos & 31));
    }
  }
  int64_t carry = 0;
  uint32_t dig[kDig];
  for (int i = 0; i < kDig; i++) {
    int64_t x = acc[i] + carry;
    dig[i] = (uint32_t)x;
    carry = x >> 32;                        // arithmetic: floor
  }
  bool neg = carry < 0;
  if (neg) {                                // magnitude = two's complement negation
    uint32_t c1 = 1;
    for (int i = 0; i < kDig; i++) {
      uint64_t x = (uint64_t)(~dig[i]) + c1;
      dig[i] = (uint32_t)x;
      c1 = (uint32_t)(x >> 32);
    }
  }
  int top = -1;
  for (int i = kDig - 1; i >= 0; i--)
    if (dig[i]) { top = i; break; }
  if (top < 0) return 0u;                   // exact zero: caller handles the sign
  // gather 64 bits below the top digit boundary, the rest as sticky
  uint64_t M = ((uint64_t)dig[top] << 32) | (top > 0 ? dig[top - 1] : 0u);
  bool sticky = false;
  for (int i = 0; i < top - 1; i++) sticky = sticky || dig[i] != 0;
  int32_t lsb0 = kBase + 32 * (top - 1);
  int32_t p = 63 - __clzll((long long)M);
  if (p > 61) {
    int s = p - 61;
    sticky = sticky || (M & ((1ull << s) - 1ull)) != 0;
    M >>= s;
    lsb0 += s;
  }
  return round_pack(M, lsb0, neg ? 1u : 0u, sticky, m.rne, m.sub_out_flush);
}

template <int K, class UT>
__device__ __forceinline__ uint32_t arch_exact(const DevModel &m, const Term<UT> (&p)[K], int nt,
                                               uint32_t cS, int32_t cE, uint32_t cneg) {
  int32_t T = kNegE;                        // bound on the top bit of every term
#pragma unroll
  for (int l = 0; l < K; l++)
    if (l < nt) T = max(T, p[l].e + 2);
  if (cS) T = max(T, cE + 1);
  if (T <= kNegE / 2) return zero_result<K, UT>(p, nt, cS, cneg);
  const int32_t L = T - 121;
  i128 W = 0;
  int32_t nb = 0;
#pragma unroll
  for (int l = 0; l <= K; l++) {
    int64_t v;
    int32_t lsb;
    if (l < K) {
      if (l >= nt) continue;
      v = p[l].neg ? -(int64_t)p[l].U : (int64_t)p[l].U;
      lsb = p[l].e - m.mab;
    } else {
      v = cneg ? -(int64_t)cS : (int64_t)cS;
      lsb = cE - 23;
    }
    if (v == 0) continue;
    int32_t sh = lsb - L;
    if (sh >= 0) {
      W += (i128)((u128)(i128)v << sh);
    } else {
      int32_t s = -sh;
      if (s >= 63) {
        W += (v < 0) ? -1 : 0;
        nb += 1;
      } else {
        W += (i128)(v >> s);
        nb += (v & ((1ll << s) - 1)) != 0;
      }
    }
  }
  if (nb == 0) {
    if (W == 0) return zero_result<K, UT>(p, nt, cS, cneg);
    return round_pack128(W, L, false, m);
  }
  uint32_t lo = round_pack128(W, L, true, m);
  uint32_t hi = round_pack128(W + (nb - 1), L, true, m);
  if (lo == hi) return lo;
  int64_t V[K + 1];
  int32_t Ls[K + 1];
  int n = 0;
#pragma unroll
  for (int l = 0; l < K; l++)
    if (l < nt) {
      V[n] = p[l].neg ? -(int64_t)p[l].U : (int64_t)p[l].U;
      Ls[n] = p[l].e - m.mab;
      n++;
    }
  V[n] = cneg ? -(int64_t)cS : (int64_t)cS;
  Ls[n] = cE - 23;
  n++;
  uint32_t r = exact_slow(m, V, Ls, n);
  return r;
}

// EXACT with a 64-bit window, for products of at most 22 significant bits (FP16,
// BF16, XF32) and an fp32 c.  T bounds the top bit of every term; the window holds
// units of 2^L with L = T - 61 + ceil(log2(K + 1)), so the K + 1 terms sum below
// 2^61.  A term +-v * 2^lsb (|v| < 2^wid) is placed as (v << Q) >> r with the
// constant Q = 62 - wid and r = Q - lsb + L >= 0: one arithmetic shift floors it
// into the window and the bits it drops set the sticky count nb.  The true sum then
// lies in [W, W + nb) units, excluding W itself when nb > 0.  With |W| >= 2^26 the
// rounding boundaries of that range are multiples of 4 units (for subnormal results
// too: the window then sits at least 152 places below 2^-126), so W + 1/2 and
// W + nb - 1/2 round like every value the sum can take next to them: when both give
// the same fp32 value, that value is the correctly rounded sum.  Otherwise (heavy
// cancellation) the full-width evaluator decides.
template <int K>
struct ExactLog {
  static constexpr int v = K + 1 <= 2 ? 1 : K + 1 <= 4 ? 2 : K + 1 <= 8 ? 3 : K + 1 <= 16 ? 4 : K + 1 <= 32 ? 5 : 6;
};

template <int K>
__device__ __forceinline__ void exact64_add(int64_t &W, int32_t &nb, int32_t sv, int32_t Q, int32_t r) {
  // sv * 2^Q has zero low 32 bits (Q >= 32), so only bits of the high word drop out
  const int64_t V = (int64_t)((uint64_t)((uint32_t)sv << (Q - 32)) << 32);
  const int32_t rr = min(r, 63);
  W += V >> rr;
  const uint32_t hi = (uint32_t)(V >> 32);
  nb += (rr > 32 && (hi << (64 - rr)) != 0u) ? 1 : 0;
}

// Correct rounding of Wt * 2^Gw (plus an unknown amount in (0, 2^Gw) when stW) plus
// c, for Wt != 0 with |Wt| < 2^62: both terms are floored into a 64-bit window under
// the larger one and rounded through the same bracket as arch_exact64.  False when
// the bracket does not decide (the caller then takes an exact path).
__device__ __forceinline__ bool merge_c64(const DevModel &m, int64_t Wt, int32_t Gw, int32_t stW, uint32_t cS,
                                          int32_t cE, uint32_t cneg, uint32_t &out) {
  const uint64_t aw = Wt < 0 ? (uint64_t)(-Wt) : (uint64_t)Wt;
  int32_t T = Gw + 64 - __clzll((long long)aw);      // |W| < 2^T
  if (cS) T = max(T, cE + 1);
  const int32_t L = T - 60;                          // two terms: |sum| < 2^61 units
  const int32_t left = max(Gw - L, 0), right = min(max(L - Gw, 0), 63);
  const int64_t Wl = (int64_t)((uint64_t)Wt << left);
  int64_t S = Wl >> right;
  int32_t nb = stW + ((right > 0 && (Wl & (int64_t)((1ull << right) - 1ull)) != 0) ? 1 : 0);
  if (cS) exact64_add<1>(S, nb, cneg ? -(int32_t)cS : (int32_t)cS, 38, 38 - (cE - 23) + L);
  if (nb == 0) {
    if (S == 0) { out = 0u; return true; }             // exact cancellation: +0
    return hw_round64(S, L, m.rne, out);
  }
  uint32_t hi;
  return (S >= (1ll << 26) || S <= -(1ll << 26)) && hw_round64(4 * S + 1, L - 2, m.rne, out) &&
         hw_round64(4 * (S + nb) - 1, L - 2, m.rne, hi) && out == hi;
}

// False when the window does not decide the rounding (out is then unset).
template <int K, class UT, int RM = -1>
__device__ __forceinline__ bool arch_exact64_try(const DevModel &m, const Term<UT> (&p)[K], uint32_t cS,
                                                 int32_t cE, uint32_t cneg, uint32_t &out) {
  int32_t T = kNegE;
#pragma unroll
  for (int l = 0; l < K; l++) T = max(T, p[l].e + 2);
  if (cS) T = max(T, cE + 1);
  if (T <= kNegE / 2) { out = zero_result<K, UT>(p, K, cS, cneg); return true; }
  const int32_t L = T - 61 + ExactLog<K>::v;
  const int32_t QP = 60 - m.mab;                     // products: |U| < 2^(mab + 2)
  int64_t W = 0;
  int32_t nb = 0;
#pragma unroll
  for (int l = 0; l < K; l++) {
    const int32_t sv = p[l].neg ? -(int32_t)p[l].U : (int32_t)p[l].U;
    exact64_add<K>(W, nb, sv, QP, QP - (p[l].e - m.mab) + L);
  }
  if (cS) exact64_add<K>(W, nb, cneg ? -(int32_t)cS : (int32_t)cS, 38, 38 - (cE - 23) + L);
  // The sum is W units when nb == 0, else it lies in (W, W + nb).  With |W| >= 2^26,
  // W + 1/2 and W + nb - 1/2 (2W + 1 and 2(W + nb) - 1 in units of 2^(L-1)) round like
  // every value next to them; for nb == 0 both ends are 2W.  So one branch-free
  // bracket serves both cases; the rest (zero, subnormal or flushed results, dropped
  // bits under heavy cancellation) is rare.
  const int rne = out_rne<RM>(m);
  const int64_t z = nb ? 1 : 0;
  const int64_t X = 2 * W + z, Y = 2 * (W + nb) - z;
  const bool big = W >= (1ll << 26) || W <= -(1ll << 26);
  uint32_t lo, hi;
  if ((big || (nb == 0 && W != 0)) && !m.sub_out_flush) {
    const bool okx = hw_round64(X, L - 1, rne, lo), oky = hw_round64(Y, L - 1, rne, hi);
    if (okx && oky) {
      if (lo == hi) { out = lo; return true; }
      return false;            // both ends correctly rounded and different: undecided
    }
  }
  if (nb == 0) {
    if (W == 0) { out = zero_result<K, UT>(p, K, cS, cneg); return true; }
    // subnormal or flushed result of an exact window: integer rounding
    out = round_pack(W < 0 ? 0ull - (uint64_t)W : (uint64_t)W, L, W < 0 ? 1u : 0u, false, rne, m.sub_out_flush);
    return true;
  }
  if (big) {
    lo = round_pack(X < 0 ? 0ull - (uint64_t)X : (uint64_t)X, L - 1, X < 0 ? 1u : 0u, false, rne, m.sub_out_flush);
    hi = round_pack(Y < 0 ? 0ull - (uint64_t)Y : (uint64_t)Y, L - 1, Y < 0 ? 1u : 0u, false, rne, m.sub_out_flush);
    if (lo == hi) { out = lo; return true; }
  }
  return false;
}

template <int K, class UT>
__device__ __forceinline__ uint32_t arch_exact64(const DevModel &m, const Term<UT> (&p)[K], uint32_t cS,
                                                 int32_t cE, uint32_t cneg) {
  uint32_t r;
  if (arch_exact64_try<K, UT>(m, p, cS, cE, cneg, r)) return r;
  int64_t V[K + 1];
  int32_t Ls[K + 1];
  int n = 0;
#pragma unroll
  for (int l = 0; l < K; l++) {
    V[n] = p[l].neg ? -(int64_t)p[l].U : (int64_t)p[l].U;
    Ls[n] = p[l].e - m.mab;
    n++;
  }
  V[n] = cneg ? -(int64_t)cS : (int64_t)cS;
  Ls[n] = cE - 23;
  n++;
  return exact_slow(m, V, Ls, n);
}

// ---------------------------------------------------------------------------
// PAIRWISE: fl(c + fl(fl(p1+p2) + fl(p3+p4))), fl = RNE to fp32 with optional
// subnormal flush after every operation (Sec. 4.2).  IEEE fp32 hardware
// arithmetic is exactly fl() here: the inputs are exact in fp32.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float fl_flush(float x, int flush) {
  if (flush && fabsf(x) < 1.17549435e-38f) return copysignf(0.0f, x);
  return x;
}

// fp32 bits of the exact value (-1)^neg * S * 2^lsb (exact for every input format)
__device__ __forceinline__ uint32_t exact_fp32_bits(uint32_t S, int32_t lsb, uint32_t neg) {
  if (!S) return neg << 31;
  int32_t p = 31 - __clz((int)S);
  int32_t E = lsb + p;
  uint32_t bits;
  if (E >= -126) bits = ((uint32_t)(E + 127) << 23) | ((S << (31 - p)) >> 8 & 0x7FFFFFu);
  else bits = S << (lsb + 149);            // subnormal: S * 2^(lsb + 149) on the 2^-149 grid
  return bits | (neg << 31);
}

__device__ __forceinline__ float elem_to_float(const FmtDev &f, uint32_t bits) {
  uint32_t cls = classify(f, bits);
  uint32_t sign = ((bits >> f.sshift) & 1u) << 31;
  if (cls == 2u) return __uint_as_float(0x7FC00000u);
  if (cls == 1u) return __uint_as_float(sign | 0x7F800000u);
  uint32_t S, neg;
  int32_t E;
  decode(f, bits, S, E, neg);
  return __uint_as_float(exact_fp32_bits(S, E - f.m_eff, neg));
}

template <int K>
__device__ __forceinline__ uint32_t arch_pairwise(const DevModel &m, const uint32_t (&ab)[K],
                                                  const uint32_t (&bb)[K], int nt, uint32_t cbits) {
  float v[K];
#pragma unroll
  for (int l = 0; l < K; l++) {
    if (l < nt) {
      float x = elem_to_float(m.fa, ab[l]);
      float y = elem_to_float(m.fb, bb[l]);
      v[l] = fl_flush(__fmul_rn(x, y), m.sub_out_flush);
    } else {
      v[l] = 0.0f;
    }
  }
#pragma unroll
  for (int w = 1; w < K; w *= 2) {
#pragma unroll
    for (int l = 0; l + w < K; l += 2 * w)
      if (l + w < nt) v[l] = fl_flush(__fadd_rn(v[l], v[l + w]), m.sub_out_flush);
  }
  uint32_t cb = cbits;
  if (m.c_sub_keep == 0u && (cb & 0x7F800000u) == 0u) cb &= 0x80000000u;
  float c = __uint_as_float(cb);
  float r = nt > 0 ? fl_flush(__fadd_rn(c, v[0]), m.sub_out_flush) : fl_flush(c, m.sub_out_flush);
  if (r != r) return m.nan_bits;
  return __float_as_uint(r);
}

// ---------------------------------------------------------------------------
// one block FMA of nt <= K products under any floating-point architecture.
// a[l], b[l] are raw element bit patterns.
// ---------------------------------------------------------------------------
template <int K, class UT, class AT>
__device__ __forceinline__ uint32_t block_fma_bits(const DevModel &m, const uint32_t (&ab)[K],
                                                   const uint32_t (&bb)[K], int nt, uint32_t cbits,
                                                   bool any_special) {
  if (m.arch == MCEMU_ARCH_PAIRWISE) return arch_pairwise<K>(m, ab, bb, nt, cbits);
  Term<UT> p[K];
#pragma unroll
  for (int l = 0; l < K; l++) p[l] = make_term<UT>(m, ab[l], bb[l]);
  uint32_t cS, cneg;
  int32_t cE;
  decode_c(m, cbits, cS, cE, cneg);
  uint32_t spec = 0;
  if (any_special) {
#pragma unroll
    for (int l = 0; l < K; l++)
      if (l < nt) spec |= product_special(m, ab[l], bb[l]);
    spec |= c_special(cbits);
  }
  if (m.prod_ovf) {
#pragma unroll
    for (int l = 0; l < K; l++)
      if (l < nt) spec |= product_overflow<UT>(m, p[l]);
  }
  if (spec) return resolve_special(m, spec);
  switch (m.arch) {
    case MCEMU_ARCH_GA_EARLY: return arch_ga_early<K, UT, AT>(m, p, nt, cS, cE, cneg);
    case MCEMU_ARCH_GA_LATE: return arch_ga_late<K, UT, AT>(m, p, nt, cS, cE, cneg);
    case MCEMU_ARCH_ODD_EVEN: return arch_odd_even<K, UT, AT>(m, p, nt, cS, cE, cneg);
    default: return arch_exact<K, UT>(m, p, nt, cS, cE, cneg);
  }
}

// integer formats: sum of K byte products plus the int32 c, wrapped or clamped
template <int K>
__device__ __forceinline__ uint32_t block_int(const DevModel &m, const uint32_t (&ab)[K],
                                              const uint32_t (&bb)[K], int nt, uint32_t cbits) {
  int32_t s = 0;
#pragma unroll
  for (int l = 0; l < K; l++)
    if (l < nt) {
      int32_t x = m.fa.is_signed ? (int32_t)(int8_t)(uint8_t)ab[l] : (int32_t)(uint8_t)ab[l];
      int32_t y = m.fb.is_signed ? (int32_t)(int8_t)(uint8_t)bb[l] : (int32_t)(uint8_t)bb[l];
      s += x * y;
    }
  if (m.int_sat) {
    int64_t t = (int64_t)s + (int64_t)(int32_t)cbits;
    t = t > INT32_MAX ? INT32_MAX : (t < INT32_MIN ? INT32_MIN : t);
    return (uint32_t)(int32_t)t;
  }
  return (uint32_t)s + cbits;
}

}  // namespace mcemu

namespace mcemu {
// A block FMA whose addend and result are binary16 (the fp16 output of Table 3's
// note, "Accurate Models of AMD Matrix Cores"): the early-c global alignment or the
// exact model, FP16/FP8 operands.  Every product of those formats and the binary16 c
// are multiples of 2^-48 below 2^37 in magnitude, so each term is an exact 128-bit
// integer in units of 2^-48; global alignment cuts the terms to the grid
// 2^(e_max - F_p) (toward zero, or down), and the sum is rounded once to 11 bits
// (exponents -14 .. 15, subnormal grid 2^-24).  c is the low half of cbits.
static __device__ __noinline__ uint32_t block_eval_acc16(const DevModel &m, const uint32_t *ea, const uint32_t *eb,
                                                         int nt, uint32_t cbits) {
  constexpr int32_t kG = -48;                    // unit of the exact terms
  const uint32_t ch = cbits & 0xFFFFu;
  uint32_t spec = 0;
  for (int l = 0; l < nt; l++) spec |= product_special(m, ea[l], eb[l]);
  if ((ch & 0x7C00u) == 0x7C00u) spec |= (ch & 0x3FFu) ? 1u : ((ch >> 15) ? 4u : 2u);
  if (spec) return ((spec & 1u) || (spec & 6u) == 6u) ? m.nan_bits : ((spec & 2u) ? 0x7C00u : 0xFC00u);
  const uint32_t cef = (ch >> 10) & 0x1Fu, cneg = ch >> 15;
  const uint32_t cS = cef ? ((ch & 0x3FFu) | 0x400u) : (ch & m.c_sub_keep);
  const int32_t cE = (int32_t)(cef ? cef : 1u) - 15;
  Term<uint64_t> p[32];
  int32_t emax = m.emin_lim;
  bool all_neg_zero = cS == 0u && cneg;
  for (int l = 0; l < nt; l++) {
    p[l] = make_term<uint64_t>(m, ea[l], eb[l]);
    if (p[l].U) emax = max(emax, p[l].e);
    all_neg_zero = all_neg_zero && p[l].U == 0 && p[l].neg;
  }
  emax = max(emax, cS ? cE : m.c_zero_exp);
  // the alignment grid in units of 2^-48 (no cut when it is not above the unit)
  const int32_t cut = (m.arch == MCEMU_ARCH_GA_EARLY) ? emax - m.F - kG : 0;
  i128 S = 0;
  for (int l = 0; l <= nt; l++) {
    u128 v;
    uint32_t neg;
    if (l < nt) {
      if (!p[l].U) continue;
      v = (u128)p[l].U << (p[l].e - m.mab - kG);  // U * 2^(e - mab), e - mab >= -48
      neg = p[l].neg;
    } else {
      if (!cS) continue;
      v = (u128)cS << (cE - 10 - kG);
      neg = cneg;
    }
    if (cut > 0) {                               // cut <= 88: the model's exponents are checked
      const u128 low = v & (((u128)1 << cut) - 1);
      v -= low;                                  // toward zero on the magnitude
      if (m.align_rd && neg && low) v += (u128)1 << cut;   // floor of a negative term
    }
    S += neg ? -(i128)v : (i128)v;
  }
  if (S == 0) return all_neg_zero ? 0x8000u : 0u;
  const uint32_t neg = S < 0 ? 1u : 0u;
  const u128 M = neg ? (u128)(-S) : (u128)S;
  const uint64_t hi = (uint64_t)(M >> 64), lo = (uint64_t)M;
  const int32_t msb = hi ? 127 - __clzll((long long)hi) : 63 - __clzll((long long)lo);
  const int32_t Ec = max(msb + kG, -14);         // exponent of the result, floored at e_min
  const int32_t r = Ec - 10 - kG;                // bits below the binary16 grid: >= 24
  const uint32_t q = (uint32_t)(M >> r);         // < 2^11
  const u128 rem = M & (((u128)1 << r) - 1), half = (u128)1 << (r - 1);
  const bool up = m.rne && (rem > half || (rem == half && (q & 1u)));
  uint32_t bits = ((uint32_t)(Ec + 14) << 10) + q + (up ? 1u : 0u);
  if (Ec > 15 || bits >= 0x7C00u) bits = m.rne ? 0x7C00u : 0x7BFFu;
  if (m.sub_out_flush && bits < 0x0400u) bits = 0u;
  return bits | (neg << 15);
}

// Any model, any block size up to 32: one out-of-line copy per translation unit
// for the general (non-specialised) kernels.  64-bit significand arithmetic.
static __device__ __noinline__ uint32_t block_eval_generic(const DevModel &m, const uint32_t *ea,
                                                           const uint32_t *eb, int nt, uint32_t cbits) {
  if (m.acc16) return block_eval_acc16(m, ea, eb, nt, cbits);
  uint32_t a[32], b[32];
  bool anys = (cbits & 0x7F800000u) == 0x7F800000u;
#pragma unroll
  for (int l = 0; l < 32; l++) {
    a[l] = l < nt ? ea[l] : 0u;
    b[l] = l < nt ? eb[l] : 0u;
    if (l < nt) anys = anys || special_word(m.fa, a[l]) || special_word(m.fb, b[l]);
  }
  if (m.fa.is_int) return block_int<32>(m, a, b, nt, cbits);
  return block_fma_bits<32, uint64_t, int64_t>(m, a, b, nt, cbits, anys);
}
}  // namespace mcemu

// ===========================================================================
// Compile-time formats for the specialised kernels: every mask and shift is an
// immediate, and special values are classified straight from the bits.
// ===========================================================================
namespace mcemu {

enum FmtId { F_FP16 = 0, F_BF16, F_XF32T, F_XF32R, F_E4M3, F_E4M3Z, F_E5M2, F_E5M2Z, F_FP32 };

template <int ID> struct Fmt;
// EB/MB: exponent/mantissa field bits; BIAS; MEFF: significand fraction bits used;
// IEEE: top exponent encodes Inf/NaN; FNUZ: 0x80 is NaN; E4OCP: S.1111.111 is NaN
#define MCEMU_FMT(ID, BYTES_, EB_, MB_, BIAS_, MEFF_, IEEE_, FNUZ_, E4OCP_, XF_)                     \
  template <> struct Fmt<ID> {                                                                      \
    static constexpr int BYTES = BYTES_, EB = EB_, MB = MB_, BIAS = BIAS_, MEFF = MEFF_;           \
    static constexpr bool IEEE = IEEE_, FNUZ = FNUZ_, E4OCP = E4OCP_;                               \
    static constexpr int XF = XF_; /* 0 none, 1 truncate to 10 bits, 2 RNE to 10 bits */          \
    static constexpr uint32_t EMASK = (1u << EB_) - 1u, MMASK = (1u << MB_) - 1u;                   \
    static constexpr int SSHIFT = EB_ + MB_;                                                        \
  };
MCEMU_FMT(F_FP16, 2, 5, 10, 15, 10, true, false, false, 0)
MCEMU_FMT(F_BF16, 2, 8, 7, 127, 7, true, false, false, 0)
MCEMU_FMT(F_XF32T, 4, 8, 23, 127, 10, true, false, false, 1)
MCEMU_FMT(F_XF32R, 4, 8, 23, 127, 10, true, false, false, 2)
MCEMU_FMT(F_E4M3, 1, 4, 3, 7, 3, false, false, true, 0)
MCEMU_FMT(F_E4M3Z, 1, 4, 3, 8, 3, false, true, false, 0)
MCEMU_FMT(F_E5M2, 1, 5, 2, 15, 2, true, false, false, 0)
MCEMU_FMT(F_E5M2Z, 1, 5, 2, 16, 2, false, true, false, 0)
MCEMU_FMT(F_FP32, 4, 8, 23, 127, 23, true, false, false, 0)
#undef MCEMU_FMT

template <int ID>
__device__ __forceinline__ void fdecode(uint32_t x, uint32_t sub_keep, uint32_t &S, int32_t &E, uint32_t &neg) {
  using F = Fmt<ID>;
  if constexpr (F::XF == 2) x = xf32_reduce(x, 2u);
  const uint32_t ef = (x >> F::MB) & F::EMASK;
  const uint32_t mf = x & F::MMASK;
  neg = (x >> F::SSHIFT) & 1u;
  uint32_t s = ef ? (mf | (1u << F::MB)) : (mf & sub_keep);
  if constexpr (F::XF != 0) s >>= 13;
  S = s;
  E = (int32_t)max(ef, 1u) - F::BIAS;
}

// Is the element an Inf or NaN (or a value that the XF32 RNE reduction turns into Inf)?
template <int ID>
__device__ __forceinline__ bool fspecial(uint32_t x) {
  using F = Fmt<ID>;
  if constexpr (F::FNUZ) return (x & 0xFFu) == 0x80u;
  else if constexpr (F::E4OCP) return (x & 0x7Fu) == 0x7Fu;
  else if constexpr (F::XF == 2) return ((x >> 23) & 0xFFu) == 0xFFu || ((xf32_reduce(x, 2u) >> 23) & 0xFFu) == 0xFFu;
  else return ((x >> F::MB) & F::EMASK) == F::EMASK;
}
template <int ID>
__device__ __forceinline__ bool fnan(uint32_t x) {
  using F = Fmt<ID>;
  if constexpr (F::FNUZ || F::E4OCP) return fspecial<ID>(x);
  else return ((x >> F::MB) & F::EMASK) == F::EMASK && (x & F::MMASK) != 0u;
}
template <int ID>
__device__ __forceinline__ bool fzero(uint32_t x, uint32_t sub_keep) {
  using F = Fmt<ID>;
  uint32_t ef = (x >> F::MB) & F::EMASK;
  if constexpr (F::FNUZ) { if (x == 0x80u) return false; }
  if constexpr (F::XF != 0) return ef == 0u && ((x & F::MMASK) >> 13 & (sub_keep >> 13)) == 0u;
  else return ef == 0u && (x & F::MMASK & sub_keep) == 0u;
}

// SWAR "some element is special" over a 32-bit word of packed elements
template <int ID>
__device__ __forceinline__ uint32_t fspecial_word(uint32_t w) {
  using F = Fmt<ID>;
  if constexpr (F::FNUZ) {
    uint32_t x = w ^ 0x80808080u;
    return (x - 0x01010101u) & ~x & 0x80808080u;
  } else if constexpr (F::E4OCP) {
    return ((w & 0x7F7F7F7Fu) + 0x01010101u) & 0x80808080u;
  } else if constexpr (F::BYTES == 1) {
    return ((w & 0x7C7C7C7Cu) + 0x04040404u) & 0x80808080u;       // E5M2 OCP
  } else if constexpr (F::BYTES == 2) {
    constexpr uint32_t em = F::EMASK << F::MB, lsb = 1u << F::MB;
    return ((w & (em | em << 16)) + (lsb | lsb << 16)) & 0x80008000u;
  } else {
    uint32_t s = ((w & 0x7F800000u) + 0x00800000u) & 0x80000000u;
    if constexpr (F::XF == 2) s |= ((xf32_reduce(w, 2u) & 0x7F800000u) + 0x00800000u) & 0x80000000u;
    return s;
  }
}

template <int ID>
__device__ __forceinline__ uint32_t felem(const uint32_t *w, int l) {
  using F = Fmt<ID>;
  if constexpr (F::BYTES == 1) return (w[l / 4] >> (8 * (l % 4))) & 0xFFu;
  else if constexpr (F::BYTES == 2) return (w[l / 2] >> (16 * (l % 2))) & 0xFFFFu;
  else return w[l];
}

// special result bits (1 NaN, 2 +Inf, 4 -Inf) of one product a*b
template <int ID>
__device__ __forceinline__ uint32_t fprod_special(uint32_t a, uint32_t b, uint32_t sub_keep) {
  using F = Fmt<ID>;
  const bool sa = fspecial<ID>(a), sb = fspecial<ID>(b);
  if (!(sa || sb)) return 0u;
  bool nan = fnan<ID>(a) || fnan<ID>(b) || (sa && fzero<ID>(b, sub_keep)) || (sb && fzero<ID>(a, sub_keep));
  if constexpr (F::XF == 2) nan = nan || (((a >> 23) & 0xFFu) == 0xFFu && (a & 0x7FFFFFu)) ||
                                   (((b >> 23) & 0xFFu) == 0xFFu && (b & 0x7FFFFFu));
  if (nan) return 1u;
  return (((a ^ b) >> F::SSHIFT) & 1u) ? 4u : 2u;
}

// exact fp32 value of an fp16 / OCP fp8 element (hardware conversions)
template <int ID>
__device__ __forceinline__ float felem_float(uint32_t x) {
  if constexpr (ID == F_FP16) {
    return __half2float(__ushort_as_half((unsigned short)x));
  } else {
    __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)x, ID == F_E4M3 ? __NV_E4M3 : __NV_E5M2);
    return __half2float(__half(h));
  }
}

template <int ID, class UT>
__device__ __forceinline__ Term<UT> fterm(uint32_t a, uint32_t b, uint32_t sub_keep) {
  uint32_t Sa, Sb, na, nb;
  int32_t Ea, Eb;
  fdecode<ID>(a, sub_keep, Sa, Ea, na);
  fdecode<ID>(b, sub_keep, Sb, Eb, nb);
  Term<UT> t;
  t.U = (UT)Sa * (UT)Sb;
  t.e = t.U ? Ea + Eb : kNegE;
  t.neg = na ^ nb;
  return t;
}

template <int ID>
__device__ __forceinline__ uint32_t exact_fixed_merge(const DevModel &m, i128 W, uint32_t cS, int32_t cE,
                                                      uint32_t cneg, uint32_t cbits);

// Exact-then-round for formats whose products lie on one fixed grid (fp16, fp8):
// every product is a multiple of 2^Lp, Lp = 2 (e_min - m), and below 2^(Tp + log2 K),
// so the exact product sum P fits a 128-bit window with LSB L = Lp - 40.  The addend
// is then added exactly, or floored into the window when it reaches below L (the
// result is at least 2^(Lp-1), so its rounding boundaries are multiples of 2^L), or,
// when it reaches above the window, the window moves up to c and P is floored into
// it.  One rounding of a floored value plus a sticky bit is exact in every case.
template <int ID, int K>
__device__ __forceinline__ uint32_t arch_exact_fixed(const DevModel &m, const Term<uint32_t> (&p)[K],
                                                     uint32_t cS, int32_t cE, uint32_t cneg, uint32_t cbits) {
  using F = Fmt<ID>;
  constexpr int32_t Lp = 2 * (1 - F::BIAS - F::MEFF);
  constexpr int32_t L = Lp - 40;
  constexpr int32_t MAB = 2 * F::MEFF;
  i128 W = 0;
#pragma unroll
  for (int l = 0; l < K; l++) {
    const int32_t sh = p[l].e - MAB - L;           // >= 40 for nonzero products
    const i128 v = (i128)((u128)p[l].U << (p[l].U ? sh : 0));
    W += p[l].neg ? -v : v;
  }
  if (cS == 0 && W == 0) return zero_result<K, uint32_t>(p, K, cS, cneg);
  return exact_fixed_merge<ID>(m, W, cS, cE, cneg, cbits);
}

// The addend step of arch_exact_fixed: W (units of 2^L, L = Lp - 40) is the exact
// product sum, not zero unless c is.
template <int ID>
__device__ __forceinline__ uint32_t exact_fixed_merge(const DevModel &m, i128 W, uint32_t cS, int32_t cE,
                                                      uint32_t cneg, uint32_t cbits) {
  using F = Fmt<ID>;
  constexpr int32_t L = 2 * (1 - F::BIAS - F::MEFF) - 40;
  if (cS == 0) return round_pack128(W, L, false, m);
  if (W == 0) return cbits;                          // c alone: already an fp32 value
  const int32_t lc = cE - 23;                        // c = +-S_c * 2^lc, S_c < 2^24
  const int64_t vc = cneg ? -(int64_t)cS : (int64_t)cS;
  if (lc + 24 <= L + 125) {
    if (lc >= L) {
      W += (i128)((u128)(i128)vc << (lc - L));
      return round_pack128(W, L, false, m);
    }
    const int32_t s = min(L - lc, 62);
    const bool st = (vc & ((1ll << s) - 1)) != 0;
    W += (i128)(vc >> s);
    return round_pack128(W, L, st, m);
  }
  const int32_t L2 = lc + 24 - 125;                  // window anchored at c
  const int32_t s2 = L2 - L;                         // > 0
  i128 Pq;
  bool st;
  if (s2 >= 127) {
    Pq = W < 0 ? -1 : 0;
    st = true;
  } else {
    Pq = W >> s2;
    st = (W & (((i128)1 << s2) - 1)) != 0;
  }
  const i128 W2 = (i128)((u128)(i128)vc << (lc - L2)) + Pq;
  return round_pack128(W2, L2, st, m);
}

// Special-value bits (1 NaN, 2 +Inf, 4 -Inf) of a block with an Inf/NaN operand or
// addend, format fixed at compile time.
template <int ID, int K>
__device__ __forceinline__ uint32_t fspecial_bits(const DevModel &m, const uint32_t (&ea)[K],
                                                  const uint32_t (&eb)[K], uint32_t cbits) {
  uint32_t spec = 0;
  if constexpr (ID == F_FP16 || ID == F_E4M3 || ID == F_E5M2) {
    // the inputs are exact in fp32 and their products cannot overflow it, so the
    // IEEE sum c + sum a*b is NaN / +-Inf exactly when the model's result is
    // (subnormal flushing changes Inf*0 and is not taken on this path)
    float t = __uint_as_float(cbits);
#pragma unroll
    for (int l = 0; l < K; l++) t = __fadd_rn(t, __fmul_rn(felem_float<ID>(ea[l]), felem_float<ID>(eb[l])));
    if (!(fabsf(t) <= 3.4028235e38f)) spec = (t != t) ? 1u : (t > 0.0f ? 2u : 4u);
  } else {
    spec = c_special(cbits);
#pragma unroll
    for (int l = 0; l < K; l++) spec |= fprod_special<ID>(ea[l], eb[l], m.fa.sub_keep);
  }
  return spec;
}

// One block FMA from its K product terms, architecture and format fixed at compile
// time; spec holds the special-value bits found so far.  With `slow` given, a set
// whose exact sum needs the full-width evaluator is not evaluated: *slow is set and
// the result is left to the caller.
template <int ARCH, int ID, int K, class UT, class AT, int RM = -1>
__device__ __forceinline__ uint32_t block_fma_terms(const DevModel &m, const Term<UT> (&p)[K], uint32_t cbits,
                                                    uint32_t spec, bool *slow = nullptr) {
  if constexpr (ID == F_BF16 || ID == F_XF32T || ID == F_XF32R || ID == F_FP32) {
    if (m.prod_ovf) {
#pragma unroll
      for (int l = 0; l < K; l++) spec |= product_overflow<UT>(m, p[l]);
      if (spec) spec |= c_special(cbits);
    }
  }
  if (spec) return resolve_special(m, spec);
  uint32_t cS, cneg;
  int32_t cE;
  decode_c(m, cbits, cS, cE, cneg);
  if constexpr (ARCH == MCEMU_ARCH_GA_EARLY) return arch_ga_early<K, UT, AT, RM>(m, p, K, cS, cE, cneg);
  else if constexpr (ARCH == MCEMU_ARCH_GA_LATE) return arch_ga_late<K, UT, AT>(m, p, K, cS, cE, cneg);
  else if constexpr (ARCH == MCEMU_ARCH_ODD_EVEN) return arch_odd_even<K, UT, AT>(m, p, K, cS, cE, cneg);
  else if constexpr (ID == F_E4M3 || ID == F_E4M3Z || ID == F_E5M2 || ID == F_E5M2Z)
    return arch_exact_fixed<ID, K>(m, p, cS, cE, cneg, cbits);
  else if constexpr (ID == F_FP16 || ID == F_BF16 || ID == F_XF32T || ID == F_XF32R) {
    if (slow) {
      uint32_t r = 0u;
      if (!arch_exact64_try<K, UT, RM>(m, p, cS, cE, cneg, r)) *slow = true;
      return r;
    }
    return arch_exact64<K, UT>(m, p, cS, cE, cneg);
  }
  else return arch_exact<K, UT>(m, p, K, cS, cE, cneg);
}

// One block FMA of K products from the elements' bit patterns.
template <int ARCH, int ID, int K, class UT, class AT, int RM = -1>
__device__ __forceinline__ uint32_t block_fma_fast(const DevModel &m, const uint32_t (&ea)[K],
                                                   const uint32_t (&eb)[K], uint32_t cbits, bool any_special,
                                                   bool *slow = nullptr) {
  const uint32_t sk = m.fa.sub_keep;
  Term<UT> p[K];
#pragma unroll
  for (int l = 0; l < K; l++) p[l] = fterm<ID, UT>(ea[l], eb[l], sk);
  const uint32_t spec = any_special ? fspecial_bits<ID, K>(m, ea, eb, cbits) : 0u;
  return block_fma_terms<ARCH, ID, K, UT, AT, RM>(m, p, cbits, spec, slow);
}

// ---------------------------------------------------------------------------
// EXACT on the FP32 pipe, for operands whose products fp32 holds exactly and
// whose sum with an fp32 c cannot overflow (FP16: |p| < 2^32 and >= 2^-48 when
// nonzero; FP8 likewise).  Error-free transformations (Knuth's TwoSum) carry the
// exact sum S = c + p_1 + ... + p_K as s + e_1 + ... + e_K; E' = fl(sum e_l) is off
// from the exact error sum by at most gamma_(K-1) * sum |e_l| (Higham, Accuracy and
// Stability of Numerical Algorithms, Sec. 4.2), bounded above by b with upward
// rounding; then TwoSum(s, E') = t + r exactly, so S = t + r + d with |d| <= b.
// t = RN(s + E') is RN(S) when |r| + b < ulp(t)/2 (or b = 0: S = t + r exactly, and
// the hardware's RNE of that sum is t); RZ(S) is t when sign(t) r >= b and the
// neighbour of t toward zero when sign(t) r < -b, given b < ulp(t)/4.  Everything
// else (a result below 2^-124, an undecided rounding) is left to the integer path.
// The IEEE sum s of the cascade is not finite exactly when an operand or c is Inf or
// NaN (the products cannot overflow), and its class is then the model's special
// result: NaN for a NaN operand, Inf * 0 or Inf - Inf, else the signed Inf; that
// result (nan_bits for NaN) is returned with the other decided ones.
// Returns 0 with out set, 2 when the rounding is not decided here.
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
  s = __fadd_rn(a, b);
  const float bb = __fadd_rn(s, -a);
  e = __fadd_rn(__fadd_rn(a, -__fadd_rn(s, -bb)), __fadd_rn(b, -bb));
}

__device__ __forceinline__ int exact_fp32_round(float s, float E, float b, int rne, uint32_t &out);

template <int K>
__device__ __forceinline__ int exact_fp32_sum(const float (&p)[K], uint32_t cbits, int rne, uint32_t nan_bits,
                                              uint32_t &out) {
  float s = __uint_as_float(cbits), e[K];
#pragma unroll
  for (int l = 0; l < K; l++) two_sum(s, p[l], s, e[l]);
  if (!(fabsf(s) <= 3.4028235e38f)) {
    out = s != s ? nan_bits : (__float_as_uint(s) & 0x80000000u) | 0x7F800000u;
    return 0;
  }
  float E = e[0], a = fabsf(e[0]);
#pragma unroll
  for (int l = 1; l < K; l++) {
    E = __fadd_rn(E, e[l]);
    a = __fadd_ru(a, fabsf(e[l]));
  }
  // gamma_(K-1) = (K-1) u / (1 - (K-1) u) < (K-1) 2^-23.9 <= 2^(ceil(log2(K-1)) - 23)
  constexpr float kGamma = K <= 2 ? 0x1p-23f : K <= 3 ? 0x1p-22f : K <= 5 ? 0x1p-21f : K <= 9 ? 0x1p-20f
                                                     : K <= 17 ? 0x1p-19f : 0x1p-18f;
  return exact_fp32_round(s, E, __fmul_ru(a, kGamma), rne, out);
}

// The rounding step of exact_fp32_sum: S = s + E + d exactly with |d| <= b.
__device__ __forceinline__ int exact_fp32_round(float s, float E, float b, int rne, uint32_t &out) {
  float t, r;
  two_sum(s, E, t, r);
  const uint32_t tb = __float_as_uint(t), ef = tb & 0x7F800000u;
  if (ef < (3u << 23) || ef == 0x7F800000u) return 2;  // |t| < 2^-124 (zero, subnormal) or beyond
  const float pt = __uint_as_float(ef);                // 2^e_t
  if (rne) {
    if (b == 0.0f || ((tb & 0x7FFFFFu) != 0u && __fadd_ru(fabsf(r), b) < __fmul_rn(pt, 0x1p-24f))) {
      out = tb;
      return 0;
    }
    return 2;
  }
  if (b >= __fmul_rn(pt, 0x1p-25f)) return 2;
  const float sr = (tb >> 31) ? -r : r;                // r measured away from zero
  if (sr >= b) { out = tb; return 0; }
  if (-sr > b) { out = tb - 1u; return 0; }            // the neighbour of t toward zero
  return 2;
}

// The sign of r + (the terms exact_scaled drops): -1, +1, or 0 when it is not decided.
// The dropped terms are products with E_a + E_b - 2 - e_ref < DMIN, and c (exponent
// e_c) when cdrop.  They are summed by the same rescaling one level down: e2 = the
// largest dropped exponent, every dropped term scaled by 2^-e2 (exact while within DMIN
// of it, else bounded), summed in fp32 with the upward-rounded bound gamma_K sum |x|
// plus the bounded ones, so their sum D lies in [lo, hi] * 2^(e2 - e_ref) in magnitude.
// r (on the 2^e_ref scale) decides when it has D's sign, or when its binade is clear of
// [lo, hi]'s scaled binades; D decides alone when r = 0 and lo > 0.
template <int ID, int K>
__device__ __forceinline__ int dropped_sum_sign(const float (&pp)[K], const int32_t (&el)[K], int32_t eref,
                                                uint32_t cb, int32_t ce, bool cdrop, float r) {
  constexpr int32_t DMIN = ID == F_BF16 ? -110 : -104;
  constexpr float kDrop = ID == F_BF16 ? 0x1p-106f : 0x1p-100f;
  int32_t e2 = cdrop ? ce + 2 : -100000;                    // c's value is below 2^(e_c + 1)
#pragma unroll
  for (int l = 0; l < K; l++)
    if (el[l] - 2 - eref < DMIN && pp[l] != 0.0f) e2 = max(e2, el[l]);
  float sum = 0.0f, mag = 0.0f, bnd = 0.0f;
#pragma unroll
  for (int l = 0; l < K; l++) {
    if (!(el[l] - 2 - eref < DMIN) || pp[l] == 0.0f) continue;
    const int32_t d = el[l] - 2 - e2;                         // <= -2
    if (d < DMIN) {
      bnd = __fadd_ru(bnd, kDrop);
      continue;
    }
    const float x = __fmul_rn(pp[l], __uint_as_float((uint32_t)(d + 127) << 23));
    sum = __fadd_rn(sum, x);
    mag = __fadd_ru(mag, fabsf(x));
  }
  if (cdrop) {
    if (ce - e2 >= -126) {                                    // c * 2^-e2 is normal: exact
      // a normal c by its exponent field; a subnormal one (e_c = -126, so e2 <= 0) by a
      // multiply with 2^-e2 <= 2^124
      const float x = (cb & 0x7F800000u) ? __uint_as_float(cb - ((uint32_t)e2 << 23))
                                         : __fmul_rn(__uint_as_float(cb), __uint_as_float((uint32_t)(127 - e2) << 23));
      sum = __fadd_rn(sum, x);
      mag = __fadd_ru(mag, fabsf(x));
    } else {
      bnd = __fadd_ru(bnd, 0x1p-125f);
    }
  }
  // K + 1 terms at most: K additions, gamma_K < (K + 1) 2^-24
  bnd = __fadd_ru(bnd, __fmul_ru(mag, (float)(K + 1) * 0x1p-24f));
  const float hi = __fadd_ru(fabsf(sum), bnd), lo = __fadd_rd(fabsf(sum), -bnd);
  const int sd = lo > 0.0f ? (sum < 0.0f ? -1 : 1) : 0;
  if (r == 0.0f) return sd;
  const int sr = r < 0.0f ? -1 : 1;
  if (sd == sr) return sr;
  const uint32_t rf = (__float_as_uint(r) >> 23) & 0xFFu;
  if (rf == 0u) return 0;                                     // a subnormal r: leave it
  const int32_t er = (int32_t)rf - 127, s = e2 - eref;        // |r| in [2^er, 2^(er + 1))
  const int32_t eh = (int32_t)((__float_as_uint(hi) >> 23) & 0xFFu) - 127 + s;   // hi 2^s < 2^(eh + 1)
  if (er > eh + 1) return sr;
  if (sd != 0) {
    const int32_t elo = (int32_t)((__float_as_uint(lo) >> 23) & 0xFFu) - 127 + s;  // lo 2^s >= 2^elo
    if ((__float_as_uint(lo) & 0x7F800000u) != 0u && er + 1 < elo) return sd;
  }
  return 0;
}

// EXACT for BF16 and XF32 products (which fp32 cannot hold: they span 2^+-266 and
// 2^+-254) on the FP32 pipe, with every term scaled by 2^-e_ref, e_ref = max(E_a + E_b,
// e_c):
//  - a' = a * 2^(1 - E_a) lies in [2, 4) (normal a) or, for a subnormal a (E_a = -126),
//    in [2^-6, 2) (BF16) or [2^-9, 2) (XF32, 10 stored mantissa bits); b' likewise, so
//    p' = a' b' is exact and p * 2^-e_ref = p' * 2^d with d = E_a + E_b - 2 - e_ref <= -2;
//  - p' * 2^d is exact while it stays normal: d >= -110 (BF16) or -104 (XF32); a
//    product further down is dropped, and 2^(DMIN + 4) > |p' 2^d| joins the bound;
//  - c * 2^-e_ref (|.| < 2) is c with its exponent field lowered by e_ref while that
//    stays normal, else dropped with 2^-125 in the bound;
// then the TwoSum cascade of exact_fp32_sum adds the K + 1 terms.  With RNE its error
// bound and decision follow exact_fp32_sum.  With RZ the errors are summed by TwoSum too
// (the bound is 0 when that sum is exact), and a kept sum that is exact takes its
// direction from the dropped terms when they all have one sign (RZ needs the sign of
// the remainder, which no fixed bound gives).
// The scaled result t' goes back by adding e_ref to its exponent field.  When that
// reaches 2^128 the correctly rounded sum overflows: +-Inf under RNE, +-max-finite
// under RTZ.  A subnormal c scales up exactly when e_ref <= 0 and is dropped otherwise.
// A subnormal result and an undecided rounding return 2 (the integer path).  Inf/NaN operands and the CDNA 3 product-overflow rule are the
// caller's.  e_ref may exceed the largest nonzero product's exponent (a zero operand
// counts with E = -126): that only moves terms toward the dropped range, and the bound
// covers them.
template <int ID, int K, int NW>
__device__ __forceinline__ int exact_scaled(const uint32_t (&wa)[NW], const uint32_t (&wb)[NW], uint32_t cb,
                                            int rne, uint32_t &out) {
  static_assert(ID == F_BF16 || ID == F_XF32T, "BF16 or truncated XF32 elements");
  constexpr int32_t DMIN = ID == F_BF16 ? -110 : -104;
  constexpr float kDrop = ID == F_BF16 ? 0x1p-106f : 0x1p-100f;
  const uint32_t cf = (cb >> 23) & 0xFFu;
  const bool csub = cf == 0u && (cb & 0x7FFFFFu) != 0u;    // a subnormal c, exponent -126
  const int32_t ce = cf ? (int32_t)cf - 127 : -126;
  float pp[K];
  int32_t el[K];
  int32_t eref = (cf || csub) ? ce : -1000;                 // c = 0 takes no part
#pragma unroll
  for (int l = 0; l < K; l++) {
    uint32_t xa, xb;                                        // the fp32 bits of a and b
    if constexpr (ID == F_BF16) {
      xa = (l & 1) ? (wa[l / 2] & 0xFFFF0000u) : (wa[l / 2] << 16);
      xb = (l & 1) ? (wb[l / 2] & 0xFFFF0000u) : (wb[l / 2] << 16);
    } else {
      xa = wa[l] & 0xFFFFE000u;                             // 10 mantissa bits, truncated
      xb = wb[l] & 0xFFFFE000u;
    }
    const uint32_t fa = max((xa >> 23) & 0xFFu, 1u), fb = max((xb >> 23) & 0xFFu, 1u);
    const float a1 = __fmul_rn(__uint_as_float(xa), __uint_as_float((255u - fa) << 23));
    const float b1 = __fmul_rn(__uint_as_float(xb), __uint_as_float((255u - fb) << 23));
    pp[l] = __fmul_rn(a1, b1);
    el[l] = (int32_t)(fa + fb) - 254;
    eref = max(eref, el[l]);
  }
  float bx = 0.0f;                                          // bound of the dropped terms
  uint32_t dsg = 0u;                                        // their signs: bit 0 +, bit 1 -
  float sv = 0.0f;
  bool cdrop = false;
  if (cf) {
    if ((int32_t)cf - eref >= 1) sv = __uint_as_float(cb - ((uint32_t)eref << 23));
    else cdrop = true;
  } else if (csub) {
    // a subnormal c scales up exactly (e_ref <= 0, so 2^-e_ref <= 2^126); with e_ref > 0
    // it falls below 2^-126 and is dropped
    if (eref <= 0) sv = __fmul_rn(__uint_as_float(cb), __uint_as_float((uint32_t)(127 - eref) << 23));
    else cdrop = true;
  }
  if (cdrop) {
    bx = 0x1p-125f;
    dsg = (cb >> 31) + 1u;
  }
  float e[K];
#pragma unroll
  for (int l = 0; l < K; l++) {
    const int32_t d = el[l] - 2 - eref;
    const bool keep = d >= DMIN;
    const float sc = __uint_as_float(keep ? (uint32_t)(d + 127) << 23 : 0u);
    if (!keep) {
      bx = __fadd_ru(bx, kDrop);
      if (pp[l] != 0.0f) dsg |= (__float_as_uint(pp[l]) >> 31) + 1u;
    }
    two_sum(sv, __fmul_rn(pp[l], sc), sv, e[l]);
  }
  uint32_t tb;
  if (rne) {
    float E = e[0], a = fabsf(e[0]);
#pragma unroll
    for (int l = 1; l < K; l++) {
      E = __fadd_rn(E, e[l]);
      a = __fadd_ru(a, fabsf(e[l]));
    }
    constexpr float kGamma = K <= 2 ? 0x1p-23f : K <= 3 ? 0x1p-22f : K <= 5 ? 0x1p-21f : K <= 9 ? 0x1p-20f
                                                       : K <= 17 ? 0x1p-19f : 0x1p-18f;
    if (exact_fp32_round(sv, E, __fadd_ru(__fmul_ru(a, kGamma), bx), 1, tb)) return 2;
  } else {
    // RZ needs the sign of S - t, which can lie far below any error bound: the errors
    // are summed by TwoSum as well (E + sum f = sum e exactly, fb >= sum |f|, 0 when
    // that sum is exact), so S = t + r + (sum f) + (dropped terms), and the sign of the
    // remainder is known when |r| clears the rest, or when the rest is one-signed
    // dropped terms (fb = 0) agreeing with r or standing alone (r = 0)
    float E = e[0], fb = 0.0f;
#pragma unroll
    for (int l = 1; l < K; l++) {
      float f;
      two_sum(E, e[l], E, f);
      fb = __fadd_ru(fb, fabsf(f));
    }
    float t, r;
    two_sum(sv, E, t, r);
    tb = __float_as_uint(t);
    const uint32_t ef = tb & 0x7F800000u;
    if (ef < (3u << 23) || ef == 0x7F800000u) return 2;    // |t| < 2^-124, or beyond
    const float b = __fadd_ru(fb, bx);
    if (b >= __fmul_rn(__uint_as_float(ef), 0x1p-25f)) return 2;
    const float sr = (tb >> 31) ? -r : r;                   // r measured away from zero
    int dir;                                                // sign of S - t, away from zero
    if (sr >= b) dir = 1;                                   // S = t or beyond it: RZ gives t
    else if (-sr > b) dir = -1;
    else if (fb == 0.0f && (dsg == 1u || dsg == 2u) && ef >= (56u << 23) &&
             (r == 0.0f || (__float_as_uint(r) >> 31) + 1u == dsg)) {
      // the dropped terms, below 2^-98 in all and under ulp(t) / 2 for |t| >= 2^-71,
      // decide alone (r = 0) or agree with r
      dir = ((tb >> 31) + 1u == dsg) ? 1 : -1;
    } else if (fb == 0.0f && dsg != 0u && ef >= (56u << 23)) {
      // S - t = r + (dropped terms) exactly: its sign from a second rescaled sum over the
      // dropped terms, set against r
      const int sd = dropped_sum_sign<ID, K>(pp, el, eref, cb, ce, cdrop, r);
      if (sd == 0) return 2;
      dir = (sd < 0) == ((tb >> 31) != 0u) ? 1 : -1;
    } else {
      return 2;
    }
    if (dir < 0) tb -= 1u;                                   // the neighbour of t toward zero
  }
  const int32_t fr = (int32_t)((tb >> 23) & 0xFFu) + eref;
  if (fr > 254) {                                           // the rounded sum reaches 2^128
    out = (tb & 0x80000000u) | (rne ? 0x7F800000u : 0x7F7FFFFFu);
    return 0;
  }
  if (fr < 1) return 2;                                     // a subnormal result
  out = tb + ((uint32_t)eref << 23);
  return 0;
}

// Powers of two (and 2^22 - 1) for fterms_w16, passed in at run time so that the
// compiler keeps them as multiplies (FMA pipe) instead of shifts and masks (ALU).
struct W16Consts {
  uint32_t one, two, k16, kmb, nzadd, nzmul;   // 1, 2, 2^16, 2^(32 - MB), 2^22 - 1, 2^10
};

// Product terms of K 16-bit elements (FP16 or BF16 with subnormals kept, no Inf or
// NaN), two elements per 32-bit word.  Both halves of a word are decoded at once:
// the exponent fields (mask), the hidden bits (the field plus the field mask carries
// into bit 15 / 31 exactly when it is nonzero), the significands with their hidden
// bits, and max(field, 1) for the subnormal exponent e_min.  The two products' field
// sums come from one add.  Splitting the halves, the shifts by MB and the
// zero-product case (e = kNegE) are multiplies by the constants in kc.
template <int ID, int K, class UT>
__device__ __forceinline__ void fterms_w16(const uint32_t *wa, const uint32_t *wb, Term<UT> (&p)[K],
                                           const W16Consts &kc) {
  using F = Fmt<ID>;
  static_assert(F::BYTES == 2 && F::XF == 0 && K % 2 == 0, "16-bit formats, an even block size");
  constexpr uint32_t EM2 = (F::EMASK << F::MB) * 0x10001u, MM2 = F::MMASK * 0x10001u;
  constexpr uint32_t LSB2 = (1u << F::MB) * 0x10001u;
  constexpr int SH = 15 - F::MB;
  constexpr uint32_t C0 = (uint32_t)(-2 * F::BIAS - kNegE);   // e - kNegE = field sum + C0
#pragma unroll
  for (int i = 0; i < K / 2; i++) {
    uint32_t Sw[2], Ep[2];
#pragma unroll
    for (int o = 0; o < 2; o++) {
      const uint32_t w = o ? wb[i] : wa[i];
      const uint32_t ef = w & EM2;
      const uint32_t hs = ((ef + EM2) & 0x80008000u) >> SH;    // hidden bits at MB and MB + 16
      Sw[o] = (w & MM2) | hs;
      Ep[o] = ef | (~hs & LSB2);                               // max(field, 1) << MB per half
    }
    const uint32_t Es = Ep[0] + Ep[1];                          // (Ea' + Eb') << MB per half
    const uint32_t Eh = __umulhi(Es, kc.k16), El = Es - Eh * kc.k16;
    const uint32_t Sah = __umulhi(Sw[0], kc.k16), Sal = Sw[0] - Sah * kc.k16;
    const uint32_t Sbh = __umulhi(Sw[1], kc.k16), Sbl = Sw[1] - Sbh * kc.k16;
    const uint32_t X = wa[i] ^ wb[i];                           // product signs at bits 15, 31
    const uint32_t Ul = Sal * Sbl, Uh = Sah * Sbh;               // < 2^22
    const uint32_t nzl = __umulhi(Ul * kc.one + kc.nzadd, kc.nzmul);   // U != 0
    const uint32_t nzh = __umulhi(Uh * kc.one + kc.nzadd, kc.nzmul);
    p[2 * i].U = (UT)Ul;
    p[2 * i].e = (int32_t)(nzl * (__umulhi(El, kc.kmb) + C0)) + kNegE;
    p[2 * i].neg = __umulhi(X * kc.k16, kc.two);
    p[2 * i + 1].U = (UT)Uh;
    p[2 * i + 1].e = (int32_t)(nzh * (__umulhi(Eh, kc.kmb) + C0)) + kNegE;
    p[2 * i + 1].neg = __umulhi(X, kc.two);
  }
}

}  // namespace mcemu

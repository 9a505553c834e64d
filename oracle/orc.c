/*
 * orc.c -- CPU oracle for bit-exact matrix-multiplier emulation.
 *
 * TEST INFRASTRUCTURE ONLY (see orc.h).  Plain and slow on purpose: every
 * quantity is an exact signed big integer scaled by 2^-ORC_FIX, and each step
 * of a model is written in the order and notation of
 * "Accurate Models of AMD Matrix Cores" (arXiv 2609.14845):
 *   - eq. (1), Sec. 2: d = sum p_l + c, p_l = a_l * b_l;
 *   - Sec. 4.1 (CDNA 1): exact products, exact sum, one RNE at the end;
 *   - Sec. 4.2 (CDNA 2): pair-wise sums of fp32-rounded products;
 *   - Sec. 4.3, Algorithm 1 (CDNA 3 fp16/bf16/tf19) and Algorithm 2 (binary8);
 *   - Table 3: the early-c global-alignment variant (NVIDIA-like features).
 * The GEMM, 2:4 sparse and multi-word drivers follow the MFMA/SWMMAC tile
 * semantics of the CDNA3 dense MFMA and RDNA4 sparse WMMA builtin pages.
 */
#include "orc.h"
#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------------------
 * Exact big integers: sign-magnitude, ORC_NL limbs of 32 bits.  A "big" x
 * stands for the real number (-1)^neg * mag * 2^-ORC_FIX.
 * ------------------------------------------------------------------------- */
#define ORC_NL 26
#define ORC_FIX 400

typedef struct { int neg; uint32_t mag[ORC_NL]; } big;

static void big_zero(big *x) { memset(x, 0, sizeof *x); }

static int big_is_zero(const big *x) {
  for (int i = 0; i < ORC_NL; i++)
    if (x->mag[i]) return 0;
  return 1;
}

static int big_bit(const big *x, int pos) {
  if (pos < 0 || pos >= 32 * ORC_NL) return 0;
  return (x->mag[pos / 32] >> (pos % 32)) & 1u;
}

static void big_set_bit(big *x, int pos) { x->mag[pos / 32] |= 1u << (pos % 32); }

/* Index of the highest set bit of the magnitude, -1 for zero. */
static int big_top(const big *x) {
  for (int i = ORC_NL - 1; i >= 0; i--)
    if (x->mag[i])
      for (int b = 31; b >= 0; b--)
        if ((x->mag[i] >> b) & 1u) return 32 * i + b;
  return -1;
}

/* Are any of the bits 0 .. pos-1 of the magnitude set? */
static int big_any_below(const big *x, int pos) {
  for (int p = 0; p < pos && p < 32 * ORC_NL; p++)
    if (big_bit(x, p)) return 1;
  return 0;
}

/* x = (-1)^neg * S * 2^e, exactly. */
static void big_from(big *x, int neg, uint64_t S, int e) {
  big_zero(x);
  for (int b = 0; b < 64; b++)
    if ((S >> b) & 1u) big_set_bit(x, b + e + ORC_FIX);
  x->neg = (S != 0) ? neg : 0;
}

static int mag_cmp(const big *a, const big *b) {
  for (int i = ORC_NL - 1; i >= 0; i--)
    if (a->mag[i] != b->mag[i]) return a->mag[i] > b->mag[i] ? 1 : -1;
  return 0;
}

/* r = a + b (r may alias a or b). */
static void big_add(big *r, const big *a, const big *b) {
  big t;
  big_zero(&t);
  if (a->neg == b->neg) {
    uint64_t carry = 0;
    for (int i = 0; i < ORC_NL; i++) {
      uint64_t s = (uint64_t)a->mag[i] + b->mag[i] + carry;
      t.mag[i] = (uint32_t)s;
      carry = s >> 32;
    }
    t.neg = a->neg;
  } else {
    const big *hi = a, *lo = b;
    if (mag_cmp(a, b) < 0) { hi = b; lo = a; }
    int64_t borrow = 0;
    for (int i = 0; i < ORC_NL; i++) {
      int64_t s = (int64_t)hi->mag[i] - lo->mag[i] - borrow;
      borrow = s < 0;
      t.mag[i] = (uint32_t)(s + (borrow ? ((int64_t)1 << 32) : 0));
    }
    t.neg = hi->neg;
  }
  if (big_is_zero(&t)) t.neg = 0;
  *r = t;
}

/* floor(log2 |x|) of a nonzero x. */
static int big_log2(const big *x) { return big_top(x) - ORC_FIX; }

/* Integer made of the magnitude bits lo .. lo+n-1 (n <= 64). */
static uint64_t big_bits(const big *x, int lo, int n) {
  uint64_t v = 0;
  for (int k = n - 1; k >= 0; k--) v = (v << 1) | (uint64_t)big_bit(x, lo + k);
  return v;
}

/* Rounding of an exact value to a multiple of 2^g. */
enum { GRID_RZ, GRID_RD, GRID_RNE };

static void big_round_grid(big *r, const big *v, int g, int mode) {
  int k = g + ORC_FIX;              /* number of magnitude bits below the grid */
  big t = *v;
  if (k <= 0) { *r = t; return; }   /* v is already a multiple of 2^g */
  int dropped = big_any_below(&t, k);
  int half = big_bit(&t, k - 1);
  int below_half = big_any_below(&t, k - 1);
  int q_odd = big_bit(&t, k);
  for (int p = 0; p < k && p < 32 * ORC_NL; p++) t.mag[p / 32] &= ~(1u << (p % 32));
  int bump = 0;                     /* add one grid step to the magnitude? */
  if (mode == GRID_RD) bump = t.neg && dropped;
  if (mode == GRID_RNE) bump = half && (below_half || q_odd);
  if (bump) {
    big step;
    big_from(&step, t.neg, 1, g);
    big_add(&t, &t, &step);
  }
  if (big_is_zero(&t)) t.neg = 0;
  *r = t;
}

/* ---------------------------------------------------------------------------
 * Input formats (Table 1) and their decoding into exact values.
 * ------------------------------------------------------------------------- */
enum { CL_ZERO, CL_FIN, CL_INF, CL_NAN };

typedef struct {
  int cls, neg;
  int E;        /* exponent: value = S * 2^(E - m); subnormals use the minimum normal E */
  uint64_t S;   /* integer significand, hidden bit included for normals */
  int m;        /* mantissa bits of the format */
} num;

int orc_elem_bytes(int32_t fmt) {
  switch (fmt) {
    case ORC_FP16: case ORC_BF16: return 2;
    case ORC_XF32: case ORC_FP32: return 4;
    case ORC_E4M3: case ORC_E5M2: case ORC_INT8: case ORC_UINT8: return 1;
    default: return 0;
  }
}

/* An IEEE-style binary format with e exponent bits, m mantissa bits and the
 * given bias.  ieee_top: the all-ones exponent encodes Inf (m = 0) and NaN. */
static num decode_binary(uint32_t bits, int e, int m, int bias, int ieee_top) {
  num x;
  x.neg = (bits >> (e + m)) & 1u;
  x.m = m;
  uint32_t ef = (bits >> m) & ((1u << e) - 1u);
  uint32_t mf = bits & ((1u << m) - 1u);
  if (ieee_top && ef == (1u << e) - 1u) {
    x.cls = mf ? CL_NAN : CL_INF; x.E = 0; x.S = 0;
  } else if (ef == 0) {
    x.cls = mf ? CL_FIN : CL_ZERO; x.E = 1 - bias; x.S = mf;
  } else {
    x.cls = CL_FIN; x.E = (int)ef - bias; x.S = mf | (1u << m);
  }
  return x;
}

static num decode(int fmt, int enc, int xr, uint32_t bits) {
  num x;
  switch (fmt) {
    case ORC_FP16: return decode_binary(bits & 0xFFFFu, 5, 10, 15, 1);
    case ORC_BF16: return decode_binary(bits & 0xFFFFu, 8, 7, 127, 1);
    case ORC_FP32: return decode_binary(bits, 8, 23, 127, 1);
    case ORC_XF32: {
      /* fp32 input whose mantissa is reduced to 10 bits (Sec. 4.3.3). */
      x = decode_binary(bits, 8, 23, 127, 1);
      if (x.cls == CL_NAN || x.cls == CL_INF) { x.m = 10; return x; }
      uint32_t ef = (bits >> 23) & 0xFFu, mf = bits & 0x7FFFFFu;
      uint32_t q = mf >> 13, r = mf & 0x1FFFu;
      if (xr == ORC_XF32_RNE && (r > 0x1000u || (r == 0x1000u && (q & 1u)))) q += 1;
      if (q == 1024u) { q = 0; ef += 1; }
      if (ef == 255u) { x.cls = CL_INF; x.m = 10; x.S = 0; x.E = 0; return x; }
      uint32_t nb = (bits & 0x80000000u) | (ef << 23) | (q << 13);
      x = decode_binary(nb, 8, 23, 127, 1);
      x.S >>= 13; x.m = 10;   /* the 13 low mantissa bits are now zero */
      return x;
    }
    case ORC_E4M3:
      if (enc == ORC_FNUZ) {
        if ((bits & 0xFFu) == 0x80u) { x.cls = CL_NAN; x.neg = 1; x.E = 0; x.S = 0; x.m = 3; return x; }
        return decode_binary(bits & 0xFFu, 4, 3, 8, 0);
      }
      if ((bits & 0x7Fu) == 0x7Fu) { x.cls = CL_NAN; x.neg = (bits >> 7) & 1u; x.E = 0; x.S = 0; x.m = 3; return x; }
      return decode_binary(bits & 0xFFu, 4, 3, 7, 0);
    case ORC_E5M2:
      if (enc == ORC_FNUZ) {
        if ((bits & 0xFFu) == 0x80u) { x.cls = CL_NAN; x.neg = 1; x.E = 0; x.S = 0; x.m = 2; return x; }
        return decode_binary(bits & 0xFFu, 5, 2, 16, 0);
      }
      return decode_binary(bits & 0xFFu, 5, 2, 15, 1);
    default:
      x.cls = CL_NAN; x.neg = 0; x.E = 0; x.S = 0; x.m = 0;
      return x;
  }
}

/* Decoding of one input under the model's subnormal-input rule. */
static num decode_in(const orc_model *md, int fmt, uint32_t bits) {
  num x = decode(fmt, md->fp8_enc, md->xf32_round, bits);
  if (md->sub_in && x.cls == CL_FIN && x.S < ((uint64_t)1 << x.m)) { x.cls = CL_ZERO; x.S = 0; }
  return x;
}

/* ---------------------------------------------------------------------------
 * Terms of eq. (1): the products p_l and the addend c, with their exponents.
 * ------------------------------------------------------------------------- */
typedef struct {
  int cls, neg;
  int e;        /* exponent used for alignment (denormalised product: E_a + E_b) */
  big v;        /* exact value */
} term;

static term make_product(const orc_model *md, num a, num b) {
  term p;
  p.neg = a.neg ^ b.neg;
  p.e = 0;
  big_zero(&p.v);
  if (a.cls == CL_NAN || b.cls == CL_NAN ||
      (a.cls == CL_INF && b.cls == CL_ZERO) || (a.cls == CL_ZERO && b.cls == CL_INF)) {
    p.cls = CL_NAN; return p;
  }
  if (a.cls == CL_INF || b.cls == CL_INF) { p.cls = CL_INF; return p; }
  if (a.cls == CL_ZERO || b.cls == CL_ZERO) { p.cls = CL_ZERO; return p; }
  /* "products are computed as the product of significands multiplied by
   * 2^(sum of exponents) and are kept denormalised" (Sec. 4.3.1). */
  p.cls = CL_FIN;
  p.e = a.E + b.E;
  big_from(&p.v, p.neg, a.S * b.S, a.E + b.E - a.m - b.m);
  /* CDNA3: overflow is detected on the magnitude |p| >= 2^128 (Sec. 4.3.2). */
  if (md->prod_ovf && big_log2(&p.v) >= 128) { p.cls = CL_INF; big_zero(&p.v); }
  return p;
}

/* The addend in the accumulator format: binary32, or binary16 from the low half. */
static term make_c(const orc_model *md, uint32_t cbits) {
  num c = md->acc_fmt == ORC_ACC_FP16 ? decode(ORC_FP16, 0, 0, cbits & 0xFFFFu) : decode(ORC_FP32, 0, 0, cbits);
  if (md->sub_in && c.cls == CL_FIN && c.S < ((uint64_t)1 << c.m)) { c.cls = CL_ZERO; c.S = 0; }
  term t;
  t.cls = c.cls; t.neg = c.neg; t.e = c.E;
  big_zero(&t.v);
  if (c.cls == CL_FIN) big_from(&t.v, c.neg, c.S, c.E - c.m);
  return t;
}

/* ---------------------------------------------------------------------------
 * Encoding of an exact value as an fp32 bit pattern.
 * ------------------------------------------------------------------------- */
static uint32_t fp32_signed_zero(int neg) { return neg ? 0x80000000u : 0u; }

/* Round v to fp32 with RNE or RTZ.  zero_neg gives the sign of an exact zero. */
static uint32_t to_fp32(const big *v, int out_round, int flush_sub, int zero_neg) {
  if (big_is_zero(v)) return fp32_signed_zero(zero_neg);
  int neg = v->neg;
  int E = big_log2(v);
  if (E < -126) E = -126;                      /* subnormal grid 2^-149 */
  big r;
  big_round_grid(&r, v, E - 23, out_round == ORC_RNE ? GRID_RNE : GRID_RZ);
  if (big_is_zero(&r)) return fp32_signed_zero(neg);
  int E2 = big_log2(&r);
  if (E2 > 127)                                /* overflow */
    return out_round == ORC_RNE ? (neg ? 0xFF800000u : 0x7F800000u)
                                : (neg ? 0xFF7FFFFFu : 0x7F7FFFFFu);
  uint32_t bits;
  if (E2 < -126) {                             /* subnormal result */
    if (flush_sub) return fp32_signed_zero(neg);
    bits = (uint32_t)big_bits(&r, -149 + ORC_FIX, 23);
  } else {
    uint32_t q = (uint32_t)big_bits(&r, E2 - 23 + ORC_FIX, 24);
    bits = ((uint32_t)(E2 + 127) << 23) | (q & 0x7FFFFFu);
  }
  return bits | (neg ? 0x80000000u : 0u);
}

/* Round v to binary16 (11-bit significand, exponents -14 .. 15, subnormal grid
 * 2^-24) with RNE or RTZ; overflow gives Inf under RNE and +-65504 under RTZ. */
static uint32_t to_fp16(const big *v, int out_round, int flush_sub, int zero_neg) {
  if (big_is_zero(v)) return zero_neg ? 0x8000u : 0u;
  int neg = v->neg;
  int E = big_log2(v);
  if (E < -14) E = -14;                        /* subnormal grid 2^-24 */
  big r;
  big_round_grid(&r, v, E - 10, out_round == ORC_RNE ? GRID_RNE : GRID_RZ);
  if (big_is_zero(&r)) return neg ? 0x8000u : 0u;
  int E2 = big_log2(&r);
  if (E2 > 15)
    return (neg ? 0x8000u : 0u) | (out_round == ORC_RNE ? 0x7C00u : 0x7BFFu);
  uint32_t bits;
  if (E2 < -14) {
    if (flush_sub) return neg ? 0x8000u : 0u;
    bits = (uint32_t)big_bits(&r, -24 + ORC_FIX, 10);
  } else {
    uint32_t q = (uint32_t)big_bits(&r, E2 - 10 + ORC_FIX, 11);
    bits = ((uint32_t)(E2 + 15) << 10) | (q & 0x3FFu);
  }
  return bits | (neg ? 0x8000u : 0u);
}

/* The result in the accumulator format. */
static uint32_t to_acc(const orc_model *md, const big *v, int zero_neg) {
  if (md->acc_fmt == ORC_ACC_FP16) return to_fp16(v, md->out_round, md->sub_out, zero_neg);
  return to_fp32(v, md->out_round, md->sub_out, zero_neg);
}

/* Sign of an exactly-zero result: negative only when every product is a
 * negative zero and c is -0 (IEEE 754 rule for sums of zeros under RNE/RTZ). */
static int zero_sign(const term *p, int n, const term *c) {
  for (int l = 0; l < n; l++)
    if (p[l].cls != CL_ZERO || !p[l].neg) return 0;
  return c->cls == CL_ZERO && c->neg;
}

/* Special values, checked before any arithmetic (Secs. 4.1-4.3): a NaN input,
 * Inf*0, or Inf + (-Inf) give NaN; otherwise an infinite term gives that Inf.
 * Returns 1 and sets *d when the result is special. */
static int special_result(const orc_model *md, const term *p, int n, const term *c, uint32_t *d) {
  int pinf = 0, ninf = 0;
  for (int l = 0; l < n + 1; l++) {
    const term *t = (l < n) ? &p[l] : c;
    if (t->cls == CL_NAN) { *d = md->nan_bits; return 1; }
    if (t->cls == CL_INF) { if (t->neg) ninf = 1; else pinf = 1; }
  }
  if (pinf && ninf) { *d = md->nan_bits; return 1; }
  const int h = md->acc_fmt == ORC_ACC_FP16;
  if (pinf) { *d = h ? 0x7C00u : 0x7F800000u; return 1; }
  if (ninf) { *d = h ? 0xFC00u : 0xFF800000u; return 1; }
  return 0;
}

/* ---------------------------------------------------------------------------
 * The multi-term adder architectures.
 * ------------------------------------------------------------------------- */

/* correct_rounding (CDNA 1, Sec. 4.1.2-4.1.4): full-precision products, an
 * exact sum, one rounding of the result to fp32. */
static uint32_t arch_exact(const orc_model *md, const term *p, int n, const term *c) {
  big V = c->v;
  for (int l = 0; l < n; l++) big_add(&V, &V, &p[l].v);
  return to_acc(md, &V, zero_sign(p, n, c));
}

/* Global alignment with early c (Table 3, NVIDIA columns): c joins the
 * products in the maximum exponent and in the alignment; every term is shifted
 * to e_max and cut to F_p fraction bits; the integer sum is rounded once. */
static uint32_t arch_ga_early(const orc_model *md, const term *p, int n, const term *c) {
  int have = 0, e_max = 0;
#define TAKE_MAX(x) do { int _x = (x); if (!have || _x > e_max) e_max = _x; have = 1; } while (0)
  for (int l = 0; l < n; l++)
    if (p[l].cls == CL_FIN) TAKE_MAX(p[l].e);
  if (c->cls == CL_FIN) TAKE_MAX(c->e);
  else if (md->c_zero_exp != ORC_NO_EXP) TAKE_MAX(md->c_zero_exp);
  if (md->emin_lim != ORC_NO_EXP) TAKE_MAX(md->emin_lim);
#undef TAKE_MAX
  big S;
  big_zero(&S);
  if (have) {
    int g = e_max - md->align_frac;
    int mode = md->align_round == ORC_RD ? GRID_RD : GRID_RZ;
    big t;
    for (int l = 0; l < n; l++) {
      big_round_grid(&t, &p[l].v, g, mode);
      big_add(&S, &S, &t);
    }
    big_round_grid(&t, &c->v, g, mode);
    big_add(&S, &S, &t);
  }
  return to_acc(md, &S, zero_sign(p, n, c));
}

/* Algorithm 1 (CDNA 3 fp16/bf16/tf32 inputs), lines 3-15, with the late-c
 * branch taken when the addend's exponent exceeds every product exponent.
 * `sum`/`e_max`/`have_p` carry the aligned product sum S_{p_i,sum} (line 4). */
static uint32_t late_c_merge(const orc_model *md, const big *S_p, int have_p, int e_max,
                             const term *p, int n, const term *c, int zero_cut) {
  /* line 5: e_c = -126 if c = 0 (the c_zero_exp of the model) */
  int have_c_exp = 1, e_c = c->e;
  if (c->cls == CL_ZERO) {
    if (md->c_zero_exp == ORC_NO_EXP) have_c_exp = 0;
    else e_c = md->c_zero_exp;
  }
  big S_acc;
  if (have_p && (!have_c_exp || e_max >= e_c)) {
    /* line 7: shift s_c right by e_max - e_c and RD it to c_frac fraction bits.
     * Algorithm 2 (line 11-14) zeroes it when e_max - e_c exceeds zero_cut. */
    big s_c;
    if (zero_cut >= 0 && have_c_exp && e_max - e_c > zero_cut) big_zero(&s_c);
    else big_round_grid(&s_c, &c->v, e_max - md->c_frac, GRID_RD);
    big_add(&S_acc, S_p, &s_c);                                  /* line 8 */
  } else {
    /* line 10: shift S_p right by e_c - e_max and RD it to psum_frac bits */
    big S_p2;
    big_round_grid(&S_p2, S_p, e_c - md->psum_frac, GRID_RD);
    big_add(&S_acc, &S_p2, &c->v);                               /* line 11 */
    if (!big_is_zero(&S_acc)) {
      /* line 12: subnormal-aware normalisation (exponent floored at -126) */
      int E = big_log2(&S_acc);
      if (E < -126) E = -126;
      /* line 13: RD to post_norm_frac fraction bits of the normalised value */
      big_round_grid(&S_acc, &S_acc, E - md->post_norm_frac, GRID_RD);
    }
  }
  /* line 15: convert to fp32 */
  return to_fp32(&S_acc, md->out_round, md->sub_out, zero_sign(p, n, c));
}

static uint32_t arch_ga_late(const orc_model *md, const term *p, int n, const term *c) {
  /* line 3: e_max over the products (zero products take no part) */
  int have_p = 0, e_max = 0;
  for (int l = 0; l < n; l++)
    if (p[l].cls == CL_FIN && (!have_p || p[l].e > e_max)) { e_max = p[l].e; have_p = 1; }
  /* line 4: align to e_max, truncate to F_p fraction bits, accumulate */
  big S_p, t;
  big_zero(&S_p);
  if (have_p)
    for (int l = 0; l < n; l++) {
      big_round_grid(&t, &p[l].v, e_max - md->align_frac,
                     md->align_round == ORC_RD ? GRID_RD : GRID_RZ);
      big_add(&S_p, &S_p, &t);
    }
  return late_c_merge(md, &S_p, have_p, e_max, p, n, c, -1);
}

/* Algorithm 2 (CDNA 3 binary8 inputs): odd- and even-indexed products are
 * aligned and truncated separately, the two partial sums are shifted to the
 * common e_max with RD, then c is merged as in Algorithm 1 except that a c
 * shifted by more than 25 places is dropped (lines 11-15). */
static uint32_t arch_odd_even(const orc_model *md, const term *p, int n, const term *c) {
  int have[2] = {0, 0}, em[2] = {0, 0};
  /* line 3: p_1, p_3, ... are "odd" (index 0 here); p_2, p_4, ... "even" */
  for (int l = 0; l < n; l++) {
    int g = l & 1;
    if (p[l].cls == CL_FIN && (!have[g] || p[l].e > em[g])) { em[g] = p[l].e; have[g] = 1; }
  }
  big S[2], t;
  big_zero(&S[0]); big_zero(&S[1]);
  for (int l = 0; l < n; l++) {   /* lines 4-5 */
    int g = l & 1;
    if (!have[g]) continue;
    big_round_grid(&t, &p[l].v, em[g] - md->align_frac,
                   md->align_round == ORC_RD ? GRID_RD : GRID_RZ);
    big_add(&S[g], &S[g], &t);
  }
  int have_p = have[0] || have[1];
  int e_max = 0;                  /* line 6 */
  if (have[0]) e_max = em[0];
  if (have[1] && (!have[0] || em[1] > e_max)) e_max = em[1];
  big S_p;
  big_zero(&S_p);
  for (int g = 0; g < 2; g++) {   /* lines 7-8 */
    if (!have[g]) continue;
    big_round_grid(&t, &S[g], e_max - md->align_frac, GRID_RD);
    big_add(&S_p, &S_p, &t);
  }
  return late_c_merge(md, &S_p, have_p, e_max, p, n, c, 25);
}

/* ---- pair-wise sum (CDNA 2, Sec. 4.2): fl() is an RNE rounding to fp32 with
 * subnormals flushed when the model flushes them; infinities may appear in any
 * fl() and propagate with the usual IEEE rules, Inf - Inf giving NaN. */
typedef struct { int cls, neg; big v; } fl32;

static fl32 fl_round(const orc_model *md, const big *v) {
  fl32 r;
  r.cls = CL_FIN; r.neg = v->neg;
  uint32_t bits = to_fp32(v, ORC_RNE, md->sub_out, v->neg);
  uint32_t ef = (bits >> 23) & 0xFFu, mf = bits & 0x7FFFFFu;
  r.neg = bits >> 31;
  big_zero(&r.v);
  if (ef == 255u) { r.cls = CL_INF; return r; }
  if (ef == 0 && mf == 0) { r.cls = CL_ZERO; return r; }
  if (ef == 0) big_from(&r.v, r.neg, mf, -149);
  else big_from(&r.v, r.neg, mf | 0x800000u, (int)ef - 127 - 23);
  return r;
}

static fl32 fl_add(const orc_model *md, fl32 x, fl32 y) {
  fl32 r;
  big_zero(&r.v);
  r.neg = 0;
  if (x.cls == CL_NAN || y.cls == CL_NAN || (x.cls == CL_INF && y.cls == CL_INF && x.neg != y.neg)) {
    r.cls = CL_NAN; return r;
  }
  if (x.cls == CL_INF) return x;
  if (y.cls == CL_INF) return y;
  if (x.cls == CL_ZERO && y.cls == CL_ZERO) { r.cls = CL_ZERO; r.neg = x.neg && y.neg; return r; }
  big s;
  big_add(&s, &x.v, &y.v);
  if (big_is_zero(&s)) { r.cls = CL_ZERO; return r; }
  return fl_round(md, &s);
}

static fl32 fl_from_term(const orc_model *md, const term *t) {
  fl32 r;
  big_zero(&r.v);
  r.neg = t->neg;
  if (t->cls != CL_FIN) { r.cls = t->cls; return r; }
  return fl_round(md, &t->v);
}

static uint32_t arch_pairwise(const orc_model *md, const term *p, int n, const term *c) {
  /* products are converted to fp32 first ("products are converted to fp32
   * before accumulation", Sec. 4.2.2), then summed pair-wise in groups. */
  fl32 level[64];
  int cnt = n;
  for (int l = 0; l < n; l++) level[l] = fl_from_term(md, &p[l]);
  while (cnt > 1) {
    int k = 0;
    for (int l = 0; l + 1 < cnt; l += 2) level[k++] = fl_add(md, level[l], level[l + 1]);
    if (cnt & 1) level[k++] = level[cnt - 1];
    cnt = k;
  }
  fl32 cc = fl_from_term(md, c);
  fl32 r = (n > 0) ? fl_add(md, cc, level[0]) : cc;
  if (r.cls == CL_NAN) return md->nan_bits;
  if (r.cls == CL_INF) return r.neg ? 0xFF800000u : 0x7F800000u;
  if (r.cls == CL_ZERO) return fp32_signed_zero(r.neg);
  return to_fp32(&r.v, ORC_RNE, md->sub_out, 0);
}

/* ---------------------------------------------------------------------------
 * One block FMA on widened bit patterns.
 * ------------------------------------------------------------------------- */
static int is_int_fmt(int f) { return f == ORC_INT8 || f == ORC_UINT8; }

static uint32_t block_int(const orc_model *md, int n, const uint32_t *a, const uint32_t *b, uint32_t c) {
  int64_t s = (int32_t)c;
  for (int l = 0; l < n; l++) {
    int64_t x = md->fmt_a == ORC_INT8 ? (int8_t)(uint8_t)a[l] : (int64_t)(uint8_t)a[l];
    int64_t y = md->fmt_b == ORC_INT8 ? (int8_t)(uint8_t)b[l] : (int64_t)(uint8_t)b[l];
    s += x * y;
  }
  if (md->int_sat) {
    if (s > INT32_MAX) s = INT32_MAX;
    if (s < INT32_MIN) s = INT32_MIN;
  }
  return (uint32_t)(uint64_t)s;   /* wrap modulo 2^32 */
}

static uint32_t block_eval(const orc_model *md, int n, const uint32_t *a, const uint32_t *b, uint32_t c) {
  if (is_int_fmt(md->fmt_a)) return block_int(md, n, a, b, c);
  term p[64], cc;
  for (int l = 0; l < n; l++)
    p[l] = make_product(md, decode_in(md, md->fmt_a, a[l]), decode_in(md, md->fmt_b, b[l]));
  cc = make_c(md, c);
  uint32_t d;
  /* The pair-wise model is a sequence of fp32 operations (Sec. 4.2): an fl() that
   * overflows creates an infinity that then meets the inputs' infinities under
   * the IEEE rules, so its special values are resolved inside arch_pairwise. */
  if (md->arch != ORC_PAIRWISE && special_result(md, p, n, &cc, &d)) return d;
  switch (md->arch) {
    case ORC_EXACT: return arch_exact(md, p, n, &cc);
    case ORC_GA_EARLY: return arch_ga_early(md, p, n, &cc);
    case ORC_GA_LATE: return arch_ga_late(md, p, n, &cc);
    case ORC_ODD_EVEN: return arch_odd_even(md, p, n, &cc);
    case ORC_PAIRWISE: return arch_pairwise(md, p, n, &cc);
    default: return md->nan_bits;
  }
}

static uint32_t load_elem(const void *base, int fmt, int64_t idx) {
  switch (orc_elem_bytes(fmt)) {
    case 1: return ((const uint8_t *)base)[idx];
    case 2: return ((const uint16_t *)base)[idx];
    default: return ((const uint32_t *)base)[idx];
  }
}

static int model_ok(const orc_model *md) {
  if (md->n_fma < 1 || md->n_fma > 64) return 0;
  if (!orc_elem_bytes(md->fmt_a) || !orc_elem_bytes(md->fmt_b)) return 0;
  if (is_int_fmt(md->fmt_a) != is_int_fmt(md->fmt_b)) return 0;
  if (md->acc_fmt != ORC_ACC_FP32 && md->acc_fmt != ORC_ACC_FP16) return 0;
  if (md->acc_fmt == ORC_ACC_FP16) {
    /* fp16 output: fp16 and fp8 inputs, the exact and early-c architectures */
    if (md->arch != ORC_EXACT && md->arch != ORC_GA_EARLY) return 0;
    for (int i = 0; i < 2; i++) {
      int f = i ? md->fmt_b : md->fmt_a;
      if (f != ORC_FP16 && f != ORC_E4M3 && f != ORC_E5M2) return 0;
    }
  }
  return 1;
}

int orc_block_fma_n(const orc_model *md, int64_t n, int32_t nt, const void *a, const void *b,
                    const uint32_t *c, uint32_t *d) {
  if (!model_ok(md) || nt < 0 || nt > md->n_fma) return -1;
  uint32_t av[64], bv[64];
  for (int64_t v = 0; v < n; v++) {
    for (int l = 0; l < nt; l++) {
      av[l] = load_elem(a, md->fmt_a, v * nt + l);
      bv[l] = load_elem(b, md->fmt_b, v * nt + l);
    }
    d[v] = block_eval(md, nt, av, bv, c[v]);
  }
  return 0;
}

int orc_block_fma(const orc_model *md, int64_t n, const void *a, const void *b,
                  const uint32_t *c, uint32_t *d) {
  return orc_block_fma_n(md, n, md->n_fma, a, b, c, d);
}

/* ---------------------------------------------------------------------------
 * GEMM drivers.  An MFMA instruction with inner size kt computes each output
 * as ceil(kt / N_FMA) chained block FMAs over consecutive k, with the fp32
 * accumulator as the next c; a GEMM chains the instructions over K.
 * ------------------------------------------------------------------------- */
static uint32_t chain(const orc_model *md, int K, int kt, const uint32_t *av, const uint32_t *bv,
                      uint32_t acc) {
  if (kt <= 0) kt = K;
  for (int k0 = 0; k0 < K; k0 += kt) {
    int kend = k0 + kt < K ? k0 + kt : K;
    for (int kb = k0; kb < kend; kb += md->n_fma) {
      int ke = kb + md->n_fma < kend ? kb + md->n_fma : kend;
      acc = block_eval(md, ke - kb, av + kb, bv + kb, acc);
    }
  }
  return acc;
}

int orc_gemm_entries(const orc_model *md, int32_t K, int32_t kt, const void *A, int64_t lda,
                     const void *Bt, int64_t ldb, const uint32_t *C, int64_t ldc,
                     int64_t n_entries, const int32_t *ii, const int32_t *jj, uint32_t *out) {
  if (!model_ok(md) || K < 0) return -1;
  uint32_t *av = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)(K + 1));
  uint32_t *bv = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)(K + 1));
  if (!av || !bv) { free(av); free(bv); return -2; }
  for (int64_t e = 0; e < n_entries; e++) {
    int64_t i = ii[e], j = jj[e];
    for (int k = 0; k < K; k++) {
      av[k] = load_elem(A, md->fmt_a, i * lda + k);
      bv[k] = load_elem(Bt, md->fmt_b, j * ldb + k);
    }
    out[e] = chain(md, K, kt, av, bv, C[i * ldc + j]);
  }
  free(av); free(bv);
  return 0;
}

/* ---------------------------------------------------------------------------
 * 2:4 structured sparsity (RDNA4 sparse WMMA page, "Structured sparsity"):
 * in every group of four along K at most two entries are nonzero; the two
 * kept positions are stored with their values, here as one metadata byte
 * idx0 | idx1 << 2 per group with idx0 < idx1.  A group with fewer than two
 * nonzeros is padded with its lowest-index zero positions.
 * ------------------------------------------------------------------------- */
static int is_zero_elem(int fmt, int enc, uint32_t bits) {
  if (is_int_fmt(fmt)) return (bits & 0xFFu) == 0;
  num x = decode(fmt, enc, ORC_XF32_TRUNC, bits);
  return x.cls == CL_ZERO;
}

static void store_elem(void *base, int fmt, int64_t idx, uint32_t v) {
  switch (orc_elem_bytes(fmt)) {
    case 1: ((uint8_t *)base)[idx] = (uint8_t)v; break;
    case 2: ((uint16_t *)base)[idx] = (uint16_t)v; break;
    default: ((uint32_t *)base)[idx] = v; break;
  }
}

int64_t orc_sparse24_compress(int32_t fmt, int32_t enc, int32_t M, int32_t K, const void *A,
                              int64_t lda, void *Ac, int64_t ldac, uint8_t *meta, int64_t ldm) {
  if (K % 4 != 0 || !orc_elem_bytes(fmt)) return -1;
  int64_t violations = 0;
  for (int64_t i = 0; i < M; i++)
    for (int g = 0; g < K / 4; g++) {
      uint32_t v[4];
      int nz[4], nnz = 0;
      for (int q = 0; q < 4; q++) {
        v[q] = load_elem(A, fmt, i * lda + 4 * g + q);
        if (!is_zero_elem(fmt, enc, v[q])) nz[nnz++] = q;
      }
      int keep[2], nk = 0;
      if (nnz > 2) violations++;
      for (int q = 0; q < nnz && nk < 2; q++) keep[nk++] = nz[q];
      for (int q = 0; q < 4 && nk < 2; q++) {
        int used = 0;
        for (int r = 0; r < nk; r++) used |= keep[r] == q;
        int is_nz = 0;
        for (int r = 0; r < nnz; r++) is_nz |= nz[r] == q;
        if (!used && !is_nz) keep[nk++] = q;
      }
      if (keep[0] > keep[1]) { int s = keep[0]; keep[0] = keep[1]; keep[1] = s; }
      store_elem(Ac, fmt, i * ldac + 2 * g, v[keep[0]]);
      store_elem(Ac, fmt, i * ldac + 2 * g + 1, v[keep[1]]);
      meta[i * ldm + g] = (uint8_t)(keep[0] | (keep[1] << 2));
    }
  return violations;
}

/* The sparse instruction multiplies compressed A against the B rows that the
 * index selects; the chain runs over the compressed terms in order, kt/2 of
 * them per instruction, in blocks of N_FMA. */
int orc_sparse24_entries(const orc_model *md, int32_t K, int32_t kt, const void *Ac, int64_t ldac,
                         const uint8_t *meta, int64_t ldm, const void *Bt, int64_t ldb,
                         const uint32_t *C, int64_t ldc, int64_t n_entries, const int32_t *ii,
                         const int32_t *jj, uint32_t *out) {
  if (!model_ok(md) || K % 4 != 0) return -1;
  int Kc = K / 2;
  uint32_t *av = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)(Kc + 1));
  uint32_t *bv = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)(Kc + 1));
  if (!av || !bv) { free(av); free(bv); return -2; }
  for (int64_t e = 0; e < n_entries; e++) {
    int64_t i = ii[e], j = jj[e];
    for (int kc = 0; kc < Kc; kc++) {
      uint8_t mb = meta[i * ldm + kc / 2];
      int idx = (kc % 2 == 0) ? (mb & 3) : ((mb >> 2) & 3);
      av[kc] = load_elem(Ac, md->fmt_a, i * ldac + kc);
      bv[kc] = load_elem(Bt, md->fmt_b, j * ldb + 4 * (kc / 2) + idx);
    }
    out[e] = chain(md, Kc, kt > 0 ? kt / 2 : 0, av, bv, C[i * ldc + j]);
  }
  free(av); free(bv);
  return 0;
}

/* ---------------------------------------------------------------------------
 * Multi-word arithmetic (Sec. 8.1): x = x_1 + x_2 + ... with x_1 = RNE_bf16(x)
 * and each next word the RNE_bf16 of the exact binary64 residual.
 * ------------------------------------------------------------------------- */
static uint16_t rne_bf16(double x) {
  int neg = signbit(x) ? 1 : 0;
  double ax = fabs(x);
  if (isnan(x)) return 0x7FC0u;
  if (ax == 0.0) return (uint16_t)(neg << 15);
  if (isinf(ax)) return (uint16_t)((neg << 15) | 0x7F80u);
  int e2;
  (void)frexp(ax, &e2);           /* ax = f * 2^e2, f in [0.5, 1) */
  int E = e2 - 1;                 /* ax in [2^E, 2^(E+1)) */
  if (E < -126) E = -126;         /* bf16 subnormal grid 2^-133 */
  double q = ldexp(ax, 7 - E);    /* exact: scaling by a power of two */
  double fq = floor(q), rem = q - fq;
  if (rem > 0.5 || (rem == 0.5 && fmod(fq, 2.0) == 1.0)) fq += 1.0;
  if (fq >= 256.0) { fq /= 2.0; E += 1; }
  if (E > 127) return (uint16_t)((neg << 15) | 0x7F80u);
  uint32_t qi = (uint32_t)fq;
  uint32_t bits = (qi < 128u) ? qi : (((uint32_t)(E + 127) << 7) | (qi - 128u));
  return (uint16_t)((neg << 15) | bits);
}

static double bf16_value(uint16_t w) {
  num x = decode(ORC_BF16, 0, 0, w);
  if (x.cls == CL_ZERO) return x.neg ? -0.0 : 0.0;
  if (x.cls == CL_INF) return x.neg ? -INFINITY : INFINITY;
  if (x.cls == CL_NAN) return NAN;
  double v = ldexp((double)x.S, x.E - x.m);
  return x.neg ? -v : v;
}

int orc_split_bf16(int64_t n, int32_t nw, const double *x, uint16_t *words) {
  if (nw < 1 || nw > 8) return -1;
  for (int64_t t = 0; t < n; t++) {
    double r = x[t];
    for (int w = 0; w < nw; w++) {
      uint16_t b = rne_bf16(r);
      words[(int64_t)w * n + t] = b;
      r = r - bf16_value(b);      /* exact residual */
    }
  }
  return 0;
}

static double fp32_value(uint32_t bits) {
  num x = decode(ORC_FP32, 0, 0, bits);
  if (x.cls == CL_ZERO) return x.neg ? -0.0 : 0.0;
  if (x.cls == CL_INF) return x.neg ? -INFINITY : INFINITY;
  if (x.cls == CL_NAN) return NAN;
  double v = ldexp((double)x.S, x.E - 23);
  return x.neg ? -v : v;
}

int orc_multiword_entries(const orc_model *wm, int32_t kt, int32_t nw, int32_t truncated, int32_t K,
                          const double *A, int64_t lda, const double *Bt, int64_t ldb,
                          int64_t n_entries, const int32_t *ii, const int32_t *jj, double *out) {
  if (!model_ok(wm) || wm->fmt_a != ORC_BF16 || wm->fmt_b != ORC_BF16 || nw < 1 || nw > 8) return -1;
  uint16_t *aw = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)nw * (size_t)(K + 1));
  uint16_t *bw = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)nw * (size_t)(K + 1));
  uint32_t *av = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)(K + 1));
  uint32_t *bv = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)(K + 1));
  if (!aw || !bw || !av || !bv) { free(aw); free(bw); free(av); free(bv); return -2; }
  for (int64_t e = 0; e < n_entries; e++) {
    int64_t i = ii[e], j = jj[e];
    orc_split_bf16(K, nw, A + i * lda, aw);
    orc_split_bf16(K, nw, Bt + j * ldb, bw);
    /* word products in the fixed order: i+j descending, then i ascending */
    double D = 0.0;
    for (int s = 2 * nw; s >= 2; s--)
      for (int wi = 1; wi <= nw; wi++) {
        int wj = s - wi;
        if (wj < 1 || wj > nw) continue;
        if (truncated && wi + wj > nw + 1) continue;
        for (int k = 0; k < K; k++) {
          av[k] = aw[(int64_t)(wi - 1) * K + k];
          bv[k] = bw[(int64_t)(wj - 1) * K + k];
        }
        uint32_t d = chain(wm, K, kt, av, bv, 0u);
        D = D + fp32_value(d);
      }
    out[e] = D;
  }
  free(aw); free(bw); free(av); free(bv);
  return 0;
}

/* ---------------------------------------------------------------------------
 * Tile facts of the CDNA3 dense MFMA page ("Accumulator layout") and of the
 * RDNA4 sparse WMMA page ("Fragment layouts").
 * ------------------------------------------------------------------------- */
int orc_tile_blocks(int32_t family, int32_t M, int32_t N, int32_t K, int32_t epl,
                    int32_t *blocks, int32_t *acc_regs) {
  if (M <= 0 || N <= 0 || K <= 0 || epl <= 0) return -1;
  if (family == 0) {
    /* A wave64 instruction holds 64 * epl elements of A; one block needs M*K
     * of them, which agrees with the Ops column: Ops = 2*M*N*K*blocks. */
    if ((64 * epl) % (M * K) != 0) return -1;
    *blocks = 64 * epl / (M * K);
    if ((*blocks * M * N) % 64 != 0) return -1;
    *acc_regs = *blocks * M * N / 64;     /* accVGPRs = blocks * M*N / wavefront */
    return 0;
  }
  if (family == 1) {
    *blocks = 1;
    *acc_regs = M * N / 32;
    return 0;
  }
  return -1;
}

int orc_tile_acc_pos(int32_t family, int32_t M, int32_t N, int32_t blocks, int32_t f64,
                     int32_t i, int32_t j, int32_t b, int32_t *lane, int32_t *reg) {
  if (i < 0 || i >= M || j < 0 || j >= N || b < 0 || b >= blocks) return -1;
  if (family == 1 && M == 16 && N == 16) {
    *lane = (i / 8) * 16 + j;
    *reg = i % 8;
    return 0;
  }
  if (family != 0 || M != N) return -1;
  if (!f64) {
    if (M == 32) { *lane = (32 * (i / 4)) % 64 + j; *reg = 16 * b + 4 * (i / 8) + i % 4; return 0; }
    if (M == 16) { *lane = 16 * (i / 4) + j; *reg = 4 * b + i % 4; return 0; }
    if (M == 4) { *lane = 4 * b + j; *reg = i; return 0; }
    return -1;
  }
  if (M == 16) { *lane = 16 * (i % 4) + j; *reg = i / 4; return 0; }
  if (M == 4) { *lane = 16 * i + 4 * b + j; *reg = 0; return 0; }
  return -1;
}

/* SWMMAC 16x16x32 source fragments (RDNA4 sparse WMMA page, "srcA" and "srcB"):
 * operand 0 = compressed A, position k in 0..15 of row `idx`; operand 1 = dense B,
 * K row k in 0..31 of column `idx`.  Two 16-bit values share a VGPR (half 0, 1). */
int orc_swmmac_src_pos(int32_t operand, int32_t idx, int32_t k, int32_t *lane, int32_t *vgpr,
                       int32_t *half) {
  if (idx < 0 || idx >= 16) return -1;
  if (operand == 0) {
    if (k < 0 || k >= 16) return -1;
    int group = (k / 4) % 2;             /* {0-3, 8-11} -> lanes 0-15, {4-7, 12-15} -> 16-31 */
    *lane = 16 * group + idx;
    *vgpr = 2 * (k / 8) + (k % 4) / 2;
    *half = k % 2;
    return 0;
  }
  if (operand == 1) {
    if (k < 0 || k >= 32) return -1;
    int group = (k / 8) % 2;             /* {0-7, 16-23} -> lanes 0-15, {8-15, 24-31} -> 16-31 */
    *lane = 16 * group + idx;
    *vgpr = 4 * (k / 16) + (k % 8) / 2;
    *half = k % 2;
    return 0;
  }
  return -1;
}
